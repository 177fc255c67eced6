// Large-M ("prefill") kernel of the group-quantized weight-only GEMM (gq_prefill.cuh): the
// instances for 256-row tiles, a four-deep ring and no K split, with those fixed at compile
// time, and this unit's wait limit and error word.
#include "gq_prefill.cuh"

namespace gq {

cudaError_t launch_prefill_fixed(const Plan &p, int M, int K, int N, int G, int prec,
                                 const CUtensorMap &mw, const CUtensorMap &ma, const void *scales,
                                 const void *zeros, void *out, unsigned token, cudaStream_t s) {
  return launch_pf_g<1>(p, M, K, N, G, prec, mw, ma, scales, zeros, out, nullptr, nullptr, token,
                        s);
}

int prefill_fixed_set_wait_limit(long long cycles) { return pf_tu_set_wait_limit(cycles); }

int prefill_fixed_read_error(int clear) { return pf_tu_read_error(clear); }

}  // namespace gq

// Small-batch kernel (gq_batch.cuh) with float zero points (GQ_ZP_FLOAT): its instantiations
// and error word, in a translation unit of their own so that they compile in parallel with
// the other forms.
#include "gq_batch.cuh"

namespace gq {

template <int G, int SC>
static cudaError_t launch_zf_m(const Plan &pl, const BtParams &bp, cudaStream_t s) {
  return launch_bt_m<G, SC, kZmFloat>(pl, bp, s);
}

template <int G>
static cudaError_t launch_zf_g(const Plan &pl, int prec, const BtParams &bp, cudaStream_t s) {
  if (prec & GQ_SC_F32) return launch_zf_m<G, kScF32>(pl, bp, s);
  if (prec & GQ_SC_BF16) return launch_zf_m<G, kScBF16>(pl, bp, s);
  return launch_zf_m<G, kScF16>(pl, bp, s);
}

cudaError_t launch_batch_zf(const Plan &pl, int prec, int G, const BtParams &bp, cudaStream_t s) {
  switch (G) {
    case 32: return launch_zf_g<32>(pl, prec, bp, s);
    case 64: return launch_zf_g<64>(pl, prec, bp, s);
    case 128: return launch_zf_g<128>(pl, prec, bp, s);
    case 256: return launch_zf_g<256>(pl, prec, bp, s);
    default: return cudaErrorInvalidValue;
  }
}

int batch_zf_set_wait_limit(long long cycles) {
  return cudaMemcpyToSymbol(g_batch_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? 0 : -1;
}

int batch_zf_read_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_batch_error, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(g_batch_error, &z, sizeof(int));
  }
  return v;
}

}  // namespace gq

// Large-M ("prefill") kernel of the group-quantized weight-only GEMM (gq_prefill.cuh): the
// host side (tensor maps, ring depth, the launch) and the instances whose tile height, ring
// depth and K split are read at run time.
#include <atomic>

#include "gq_prefill.cuh"
#include "gq_tma_host.h"

namespace gq {

// ------------------------------------------------------------------ host side

static int encode_maps(int M, int K, int N, int BM, const void *A, const void *Wq,
                       CUtensorMap *mw, CUtensorMap *ma) {
  // packed codes as uint32 [tiles][K/64 chunks][128 words]
  const cuuint64_t wdims[3] = {128, (cuuint64_t)(K / 64), (cuuint64_t)((N + 15) / 16)};
  const cuuint64_t wstr[2] = {512, (cuuint64_t)(K / 64) * 512};
  const cuuint32_t wbox[3] = {128, 1, 8};
  const cuuint32_t ones[3] = {1, 1, 1};
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) {
    note_cuda_error_code("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", -1);
    return GQ_ERR_CUDA;
  }
  CUresult r = enc(mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(Wq),
                                      wdims, wstr, wbox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                      CU_TENSOR_MAP_SWIZZLE_NONE,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    note_cuda_error_code("cuTensorMapEncodeTiled(packed codes)", (int)r);
    return GQ_ERR_CUDA;
  }
  // activations bf16 [M][K], BM rows x 64 k per box, 128-byte swizzle
  const cuuint64_t adims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t astr[1] = {(cuuint64_t)K * 2};
  const cuuint32_t abox[2] = {64, (cuuint32_t)BM};
  r = enc(ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(A), adims,
                             astr, abox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    note_cuda_error_code("cuTensorMapEncodeTiled(activations)", (int)r);
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

// per-launch token: a launch that gives up marks only itself
static unsigned next_token() {
  static std::atomic<unsigned> t{0};
  return t.fetch_add(1u) + 1u;
}

size_t prefill_smem_bytes(int BM, int stages) {
  return (size_t)stages * pf_stage_bytes(BM) + (size_t)kPfDqBufs * kPfDqBytes + 1024;
}

// The deepest ring (at most kPfMaxStages) of BM-row stages that fits smem_cap bytes.
int prefill_stages(int BM, size_t smem_cap) {
  for (int s = kPfMaxStages; s >= kPfMinStages; --s)
    if (prefill_smem_bytes(BM, s) <= smem_cap) return s;
  return 0;
}

bool prefill_supported(int M, int K, int N, int G, int prec) {
  if (!(prec & GQ_W4) || (prec & GQ_ACT_F32)) return false;
  if (!(G == 64 || G == 128 || G == 256)) return false;
  return M >= 1 && N >= 8 && K % G == 0 && K % 64 == 0;
}

cudaError_t launch_prefill(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                           const void *Wq, const void *scales, const void *zeros, void *out,
                           float *part, unsigned *counters, cudaStream_t s) {
  CUtensorMap mw, ma;
  if (encode_maps(M, K, N, p.m_tile, A, Wq, &mw, &ma) != GQ_OK) return cudaErrorInvalidValue;
  const unsigned token = next_token();
  if (p.m_tile == kPfFixedTileM && p.slots == kPfFixedStages && p.nsplit == 1)
    return launch_prefill_fixed(p, M, K, N, G, prec, mw, ma, scales, zeros, out, token, s);
  return launch_pf_g<0>(p, M, K, N, G, prec, mw, ma, scales, zeros, out, part, counters, token, s);
}

int prefill_set_wait_limit(long long cycles) {
  const int a = pf_tu_set_wait_limit(cycles);
  const int b = prefill_fixed_set_wait_limit(cycles);
  return a != 0 ? a : b;
}

int prefill_read_error(int clear) {
  const int a = pf_tu_read_error(clear);
  const int b = prefill_fixed_read_error(clear);
  return a != 0 ? a : b;
}

}  // namespace gq

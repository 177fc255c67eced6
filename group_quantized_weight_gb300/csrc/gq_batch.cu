// Small-batch kernel (gq_batch.cuh): launches for the symmetric and INT4 zero-point forms,
// plan helpers and the host side of its error word.
#include "gq_batch.cuh"

namespace gq {

template <int G, int SC>
static cudaError_t launch_bt_z(const Plan &pl, int prec, const BtParams &bp, cudaStream_t s) {
  if (prec & GQ_ZP) return launch_bt_m<G, SC, kZmInt4>(pl, bp, s);
  return launch_bt_m<G, SC, kZmSym>(pl, bp, s);
}

template <int G>
static cudaError_t launch_bt_g(const Plan &pl, int prec, const BtParams &bp, cudaStream_t s) {
  if (prec & GQ_SC_F32) return launch_bt_z<G, kScF32>(pl, prec, bp, s);
  if (prec & GQ_SC_BF16) return launch_bt_z<G, kScBF16>(pl, prec, bp, s);
  return launch_bt_z<G, kScF16>(pl, prec, bp, s);
}

int batch_set_wait_limit(long long cycles) {
  const int a = cudaMemcpyToSymbol(g_batch_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? 0 : -1;
  const int b = batch_zf_set_wait_limit(cycles);
  return a != 0 ? a : b;
}

int batch_read_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_batch_error, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(g_batch_error, &z, sizeof(int));
  }
  const int vz = batch_zf_read_error(clear);
  return v ? v : vz;
}

bool batch_supported(int M, int K, int G, int prec) {
  return (prec & GQ_W4) && !(prec & GQ_ACT_F32) && M >= 1 && K % kBtSlotK == 0 &&
         G <= kBtSlotK;
}

// K slice: the largest multiple of 256 that divides K with a 32-row (or M-row, when fewer)
// bf16 activation slice of at most 64 KiB.
int batch_slice_k(int M, int K) {
  const int rows = M < kBtRows ? M : kBtRows;
  int best = kBtSlotK;
  for (int ksl = kBtSlotK; ksl <= K; ksl += kBtSlotK)
    if (K % ksl == 0 && (size_t)rows * ksl * 2 <= (64u << 10)) best = ksl;
  return best;
}

size_t batch_smem_bytes(int M, int K_slice, int G, int prec, int slots) {
  const int es = (prec & GQ_SC_F32) ? 4 : 2;
  const int rows = M < kBtRows ? M : kBtRows;
  const size_t act = ((size_t)rows * act_row_words(K_slice / kChunkK) * 4 + 127) & ~(size_t)127;
  const size_t asum = (prec & GQ_ZP_FLOAT) ? batch_asum_bytes(K_slice, G, batch_mt(M)) : 0;
  return act + asum + (size_t)batch_warps(batch_mt(M)) * slots * batch_slot_bytes(G, es);
}

int batch_threads(int M) { return batch_warps(batch_mt(M)) * 32; }

int batch_slots_for(int M, int K_slice, int G, int prec, size_t smem_cap) {
  for (int s = kBtMaxSlots; s >= 2; --s)
    if (batch_smem_bytes(M, K_slice, G, prec, s) <= smem_cap) return s;
  return 0;
}

cudaError_t launch_batch(const Plan &pl, int M, int K, int N, int G, int prec, const void *A,
                         const void *Wq, const void *scales, const void *zeros, void *out,
                         float *part, unsigned *counters, cudaStream_t s) {
  BtParams bp;
  bp.Wp = reinterpret_cast<const uint8_t *>(Wq);
  bp.A32 = reinterpret_cast<const uint32_t *>(A);
  bp.scales = scales;
  bp.zeros = (prec & GQ_ZP) ? reinterpret_cast<const uint32_t *>(zeros) : nullptr;
  bp.zf = (prec & GQ_ZP_FLOAT) ? zeros : nullptr;
  bp.out = out;
  bp.part = part;
  bp.counters = counters;
  bp.M = M;
  bp.K = K;
  bp.N = N;
  bp.T = (N + kTileN - 1) / kTileN;
  bp.KS = pl.nsplit;
  bp.KSL = pl.unit_k;
  bp.cps = pl.split_count;
  bp.S = pl.slots;
  bp.out_f32 = (prec & GQ_OUT_F32) ? 1 : 0;
  bp.static_w = (prec & GQ_STATIC_W) ? 1 : 0;
  bp.gate_up = (prec & GQ_GATE_UP) ? 1 : 0;
  if (prec & GQ_ZP_FLOAT) return launch_batch_zf(pl, prec, G, bp, s);
  switch (G) {
    case 32: return launch_bt_g<32>(pl, prec, bp, s);
    case 64: return launch_bt_g<64>(pl, prec, bp, s);
    case 128: return launch_bt_g<128>(pl, prec, bp, s);
    case 256: return launch_bt_g<256>(pl, prec, bp, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gq

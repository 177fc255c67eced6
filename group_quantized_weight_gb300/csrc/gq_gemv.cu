// Warp-specialized small-M decode kernel (M <= 4) of the group-quantized weight-only GEMM.
//
// At decode the path is bound by the bytes of the packed weights ("GPU Kernel 工程（09）：量化
// 与融合 kernel", section 3.2), so what matters is keeping HBM busy while spending as few
// instructions per byte as possible.  One CTA per SM, two roles:
//   producer warp   streams this CTA's slots (256 k of one 16-column tile: 2 KB of codes, a
//                   contiguous piece of the packed layout) into a ring of S stages.  A stage
//                   holds one slot per consumer warp: lane w issues consumer w's cp.async.bulk
//                   of codes and one TMA tensor copy of the slot's group scales (a 16-column x
//                   G-row box of the canonical [K/G][N] scale matrix); everything completes on
//                   the stage's "full" mbarrier.
//   consumer warps  wait for a stage, decode their slot's codes in registers (the FP16
//                   magic-number trick of section 2.4 of the same page), multiply on tensor
//                   cores (mma.sync m16n8k16, the 16 MMA rows on the tile's columns) and
//                   release the stage on its "empty" mbarrier.
// A consumer's only per-slot bookkeeping is one wait and one arrive; address arithmetic for
// the copies lives in the producer.  The shared memory (activations in exponent bands, the
// ring, and the consumers' partial sums) is sized so that two CTAs fit on an SM where the
// shape allows: the next call's CTA then starts streaming its weights (GQ_STATIC_W) while
// this one finishes, so consecutive calls overlap on every SM.
//
// Work partition (the striped partitioning of section 3.3 item 4 of the same page): the
// packed codes are a sequence of 16-column tiles with K contiguous, so the (tile, slot) pairs
// form one byte stream.  CTA c owns a contiguous range of slots — whole tiles when there are
// enough of them, otherwise an equal share — and its consumer warps split that range into
// contiguous sub-ranges.  Every partial sum is a sum of whole scaled groups: a tile split
// between warps is summed in warp order, one split between CTAs in CTA order by whichever
// CTA finishes its part last, so the result is bitwise reproducible.
//
// Activations: bf16 rows are carried into fp16 exactly as two exponent bands per row (MMA
// columns 2m and 2m + 1), as in the striped kernel; each group starts a fresh FP32
// accumulator and is multiplied by its scale after its last MMA step (the group-wise GEMM of
// "04 · 分组量化 GEMM 内核", section 2).
#include <type_traits>

#include "gq_device.cuh"
#include "gq_tma_host.h"

namespace gq {

namespace gv {
constexpr int kSlotChunks = 4;                          // 64-k chunks per slot
constexpr int kSlotK = kSlotChunks * kChunkK;           // 256 k
constexpr int kSlotCodes = kSlotChunks * 512;           // 2 KB of codes per slot
constexpr int kMaxStages = 8;
constexpr int kMaxConsumers = 16;
constexpr long long kWaitCycles = 4000000000ll;         // bounded waits: about two seconds
constexpr uint32_t kMagic = 0x64006400u;                // fp16 1024 in both halves
constexpr uint32_t kSixteenth = 0x2C002C00u;            // fp16 1/16
constexpr uint32_t kLoSym = 0x64086408u;                // fp16 1024 + 8
constexpr uint32_t kHiSym = 0xD480D480u;                // fp16 -(64 + 8)
}  // namespace gv

// Sticky device-side status (GQ_ERR_TIMEOUT after a bounded wait gave up).
static __device__ int g_gemv_error;

namespace gv {

__device__ __forceinline__ uint32_t saddr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ bool try_phase(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait until the phase of parity `parity` of the mbarrier completes; bounded (about two
// seconds of SM clock), then GQ_ERR_TIMEOUT is recorded and false returned.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity) {
  if (try_phase(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (try_phase(bar, parity)) return true;
    if ((it & 63u) == 0u && clock64() - t0 > kWaitCycles) {
      atomicExch(&g_gemv_error, GQ_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tensor_copy_2d(uint32_t dst, const CUtensorMap *map,
                                               uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

}  // namespace gv

struct GemvParams {
  const uint8_t *Wp;          // packed codes
  const uint16_t *A;          // activations, bf16 [M][K]
  const uint32_t *zeros;      // [K/G][N/8] or NULL
  void *out;                  // [M][N] (gate+up: [M][N/2])
  float *part;                // [gridDim.x][2][4][16] per-CTA partial sums (shared tiles only)
  unsigned *counters;         // per-tile arrival counters (shared tiles only)
  int M, K, N;
  int split_count, split_mult;   // CTA c owns slots zsplit(split_count, grid, c) * split_mult
  int S;                         // ring stages
  int slot_bytes;                // codes + scale regions of one slot in the ring
  int scale_b_off;               // byte offset of the scales of the tile's columns 8..15
  int out_f32;
  int static_w;                  // weights may be read before the preceding kernel ends
  int gate_up;                   // fused gate+up: out[m][j] = silu(col j) * (col N/2 + j)
};

// Shared memory (dynamic): [bands][ring][pieces]
//   bands   (1 + 2M) rows of act_row_words(K / 64) words: a zero row, then the two exponent
//           bands of each activation row, permuted for the B operands
//   ring    S stages x NC slots x slot_bytes: 2 KB of codes, then the slot's group scales
//   pieces  NC x 2 x M x 16 floats: a warp's partial sums of its first and last tile
template <int G, int SC, bool ZP, int NC>
__global__ void __launch_bounds__((NC + 1) * 32, NC <= 8 ? 2 : 1)
    w4_gemv_kernel(const __grid_constant__ CUtensorMap smap, const GemvParams p) {
  using namespace gv;
  constexpr int ES = SC == kScF32 ? 4 : 2;          // bytes per scale
  constexpr int GPS = kSlotK / G;                   // groups per slot
  constexpr int SPG = G / 16;                       // 16-k MMA steps per group
  typedef typename std::conditional<SC == kScF32, uint32_t, unsigned short>::type sc_t;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the tensor copies of the scales land at 128-byte aligned addresses
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  // full_bar[stage][w]: consumer w's slot of the stage landed; empty_bar[stage]: every consumer
  // released the stage
  __shared__ __align__(8) uint64_t full_bar[kMaxStages][kMaxConsumers], empty_bar[kMaxStages];
  __shared__ int s_emax[4], s_emin[4];
  __shared__ int s_last[kMaxConsumers];
  asm volatile("griddepcontrol.launch_dependents;");

  const int M = p.M, K = p.K, N = p.N, S = p.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = K / kChunkK;                        // chunks per tile
  const int SPT = K / kSlotK;                       // slots per tile
  int cb, ce;                                       // this CTA's slots
  zsplit_dev(p.split_count, gridDim.x, blockIdx.x, cb, ce);
  cb *= p.split_mult;
  ce *= p.split_mult;
  const int RS = act_row_words(C);
  uint32_t *bands = reinterpret_cast<uint32_t *>(smem);
  uint8_t *ring = smem + (((size_t)(1 + 2 * M) * RS * 4 + 127) & ~(size_t)127);
  float *pieces = reinterpret_cast<float *>(ring + (size_t)S * NC * p.slot_bytes);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      for (int w = 0; w < NC; ++w)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&full_bar[s][w])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&empty_bar[s])), "r"(NC)
                   : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x < 4) {
    s_emax[threadIdx.x] = 0;
    s_emin[threadIdx.x] = 255;
  }
  __syncthreads();

  // ================================================================ producer warp
  if (warp == NC) {
    if (!p.static_w) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&smap) : "memory");
    // lane w < NC feeds consumer w: slots [wb, we) of the CTA's range
    int wb = 0, we = 0;
    if (lane < NC) {
      zsplit_dev(ce - cb, NC, lane, wb, we);
      wb += cb;
      we += cb;
    }
    int n0, e0;                                     // consumer 0 has the most slots
    zsplit_dev(ce - cb, NC, 0, n0, e0);
    const int nmax = e0 - n0;
    const int full_bytes_slot = kSlotCodes + 16 * GPS * ES;
    int st = 0;
    for (int j = 0; j < nmax; ++j) {
      if (j >= S) {
        // fill j of stage st reuses it after fill j - S: wait until every consumer released
        // that one (empty phase j / S - 1)
        bool ok = true;
        if (lane == 0) ok = wait_phase(saddr(&empty_bar[st]), (uint32_t)((j / S + 1) & 1));
        if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;
      }
      // lane w fills consumer w's slot of the stage, if it still has one
      if (lane < NC && wb + j < we) {
        const uint32_t fb = saddr(&full_bar[st][lane]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                     "r"(full_bytes_slot)
                     : "memory");
        const int slot = wb + j, t = slot / SPT, js = slot - t * SPT;
        const uint32_t dst = saddr(ring + ((size_t)st * NC + lane) * p.slot_bytes);
        bulk_copy(dst, p.Wp + (size_t)slot * kSlotCodes, kSlotCodes, fb);
        if (p.gate_up) {                            // gate columns 8t.., up columns N/2 + 8t..
          tensor_copy_2d(dst + kSlotCodes, &smap, fb, 8 * t, js * GPS);
          tensor_copy_2d(dst + p.scale_b_off, &smap, fb, N / 2 + 8 * t, js * GPS);
        } else {
          tensor_copy_2d(dst + kSlotCodes, &smap, fb, 16 * t, js * GPS);
        }
      }
      if (++st == S) st = 0;
    }
    return;
  }

  // ================================================================ consumer warps
  const int r0 = lane >> 2, q = lane & 3;
  int wb, we;                                       // this warp's slots
  zsplit_dev(ce - cb, NC, warp, wb, we);
  wb += cb;
  we += cb;
  const int n = we - wb;
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- exponent bands (the consumer warps only; the producer is already streaming)
  const int nth = NC * 32, tid = threadIdx.x;
  for (int idx = tid; idx < RS; idx += nth) bands[idx] = 0u;   // zero row 0
  const int ppr = K >> 3;                          // 16-byte pieces per row
  const uint4 *A4 = reinterpret_cast<const uint4 *>(p.A);
  for (int m = 0; m < M; ++m) {
    unsigned mx = 0u, mn = 0xFFFFu;
    for (int pc = tid; pc < ppr; pc += nth) {
      const uint4 v = A4[(size_t)m * ppr + pc];
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t mag = wv[e] & 0x7FFF7FFFu;
        const uint32_t lo = mag & 0xFFFFu, hi = mag >> 16;
        mx = max(mx, max(lo, hi));
        mn = min(mn, min(lo ? lo : 0xFFFFu, hi ? hi : 0xFFFFu));   // smallest non-zero
      }
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    mn = __reduce_min_sync(0xffffffffu, mn);
    if (lane == 0) {
      atomicMax(&s_emax[m], (int)(mx >> 7));
      atomicMin(&s_emin[m], (int)(mn >> 7));
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(nth) : "memory");
  for (int v = 0; v < 2 * M; ++v) {
    const int m = v >> 1, b = v & 1;
    const int emax = s_emax[m], emin = s_emin[m];
    const int nbu = emin > emax ? 0 : min(2, ((emax - emin) >> 5) + 1);
    if (b >= nbu) continue;
    const int sb_ = 142 - emax + 32 * b;           // scale exponent of band b
    uint32_t *brw = bands + (1 + v) * RS;
    const bool fast = nbu == 1 && emax < 255;
    const int s1 = sb_ / 2, s2 = sb_ - s1;
    const float c1 = __int_as_float((127 + s1) << 23), c2 = __int_as_float((127 + s2) << 23);
    for (int pc = tid; pc < ppr; pc += nth) {
      const uint4 vv = A4[(size_t)m * ppr + pc];
      const uint32_t wv[4] = {vv.x, vv.y, vv.z, vv.w};
      uint32_t *dst = brw + (pc >> 3) * 32 + ((pc & 7) >> 2) * 16 + ((pc >> 1) & 1) * 2 + (pc & 1);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t raw = wv[e];
        uint32_t pair = 0u;
        if (fast) {
          const __half2 h = __floats2half2_rn(__uint_as_float(raw << 16) * c1 * c2,
                                              __uint_as_float(raw & 0xFFFF0000u) * c1 * c2);
          pair = *reinterpret_cast<const uint32_t *>(&h);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t bits = (raw >> (16 * h)) & 0xFFFFu;
            const int ex = (bits >> 7) & 0xFF;
            if ((bits & 0x7FFFu) && ((emax - ex) >> 5) == b) {
              float f;
              if (ex == 255)
                f = __uint_as_float(bits << 16);                        // inf / nan stay so
              else if (ex == 0)
                f = ldexpf(__uint_as_float(bits << 16), sb_);           // bf16 subnormal
              else
                f = __uint_as_float((bits << 16) + ((uint32_t)sb_ << 23));  // exponent + sb
              pair |= (uint32_t)__half_as_ushort(__float2half_rn(f)) << (16 * h);
            }
          }
        }
        dst[4 * e] = pair;
      }
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(nth) : "memory");

  // B-operand row of this lane: MMA column r0 = band r0 % 2 of activation row r0 / 2, or the
  // zero row
  const uint32_t *brow;
  {
    const int m = r0 >> 1, b = r0 & 1;
    int row = 0;
    if (m < M) {
      const int emax = s_emax[m], emin = s_emin[m];
      const int nbu = emin > emax ? 0 : min(2, ((emax - emin) >> 5) + 1);
      if (b < nbu) row = 1 + 2 * m + b;
    }
    brow = bands + row * RS + q * 4;
  }
  auto zlo_of = [&](uint32_t zw) -> uint32_t {     // fp16(1024 + z) in both halves
    return (0x6400u | ((zw >> (4 * r0)) & 0xFu)) * 0x00010001u;
  };
  auto zhi_of = [&](uint32_t zw) -> uint32_t {     // fp16(-(64 + z)) in both halves
    return (0xD400u | (((zw >> (4 * r0)) & 0xFu) << 4)) * 0x00010001u;
  };
  auto scale_f = [&](uint32_t bits) -> float {
    if (SC == kScF32) return __uint_as_float(bits);
    if (SC == kScBF16) return __uint_as_float(bits << 16);
    return __half2float(__ushort_as_half((unsigned short)bits));
  };
  const int NW = N >> 3;
  auto load_zeros = [&](int tz, int jz, uint32_t (&z)[GPS][2]) {
#pragma unroll
    for (int gi = 0; gi < GPS; ++gi) {
      const uint32_t *zr = p.zeros + (size_t)(jz * GPS + gi) * NW;
      z[gi][0] = __ldg(zr + min(p.gate_up ? tz : 2 * tz, NW - 1));
      z[gi][1] = __ldg(zr + min(p.gate_up ? NW / 2 + tz : 2 * tz + 1, NW - 1));
    }
  };
  const int t_first = wb / SPT;
  int t = t_first, j = wb - t_first * SPT;
  int j0 = j;                                      // first slot of this warp's share of t
  uint32_t zcur[GPS][2], znext[GPS][2];
  if (ZP && n > 0) load_zeros(t, j, znext);
  const int scale_row = p.gate_up ? 8 : 16;        // scale elements per group row in a slot

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  // end of the warp's share of tile t (slots j0 .. j1 - 1): combine the bands, then store a
  // whole tile or keep the share for the reduction
  auto flush = [&](int j1) {
    const int mrow = q;
    const int emax = mrow < M ? s_emax[mrow] : 127;
    const float v0 = scale_pow2(acc[0], emax - 142) + scale_pow2(acc[1], emax - 174);
    const float v1 = scale_pow2(acc[2], emax - 142) + scale_pow2(acc[3], emax - 174);
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    if (mrow >= M) return;
    if (j0 == 0 && j1 == SPT) {
      if (p.gate_up) {
        store_out_rt(p.out, (size_t)mrow * (N / 2) + t * 8 + r0, silu_mul(v0, v1), p.out_f32 != 0);
      } else {
        const int n0 = t * kTileN + r0;
        if (n0 < N) store_out_rt(p.out, (size_t)mrow * N + n0, v0, p.out_f32 != 0);
        if (n0 + 8 < N) store_out_rt(p.out, (size_t)mrow * N + n0 + 8, v1, p.out_f32 != 0);
      }
    } else {
      float *pc = pieces + ((warp * 2 + (t == t_first ? 0 : 1)) * M + mrow) * kTileN;
      pc[r0] = v0;
      pc[r0 + 8] = v1;
    }
  };

  int st = 0;
  uint32_t ph = 0;
  for (int i = 0; i < n; ++i) {
    if (!wait_phase(saddr(&full_bar[st][warp]), ph)) break;
    if (ZP) {
#pragma unroll
      for (int gi = 0; gi < GPS; ++gi) {
        zcur[gi][0] = znext[gi][0];
        zcur[gi][1] = znext[gi][1];
      }
      if (i + 1 < n) {
        if (j + 1 < SPT) load_zeros(t, j + 1, znext);
        else load_zeros(t + 1, 0, znext);
      }
    }
    const uint8_t *slot = ring + ((size_t)st * NC + warp) * p.slot_bytes;
    const sc_t *sca = reinterpret_cast<const sc_t *>(slot + kSlotCodes);
    const sc_t *scb = reinterpret_cast<const sc_t *>(slot + p.scale_b_off);
    const uint32_t *bslot = brow + j * (kSlotChunks * 32);
#pragma unroll
    for (int ch = 0; ch < kSlotChunks; ++ch) {
      const uint4 wv = *reinterpret_cast<const uint4 *>(slot + ch * 512 + lane * 16);
      const uint4 blo = *reinterpret_cast<const uint4 *>(bslot + ch * 32);
      const uint4 bhi = *reinterpret_cast<const uint4 *>(bslot + ch * 32 + 16);
      const uint32_t bq[8] = {blo.x, blo.y, blo.z, blo.w, bhi.x, bhi.y, bhi.z, bhi.w};
      const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
      float d[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int stp = ch * 4 + jj;                 // compile-time 16-k step of the slot
        const int gi = stp / SPG;
        const uint32_t zl = ZP ? zlo_of(zcur[gi][0]) : kLoSym;
        const uint32_t zh = ZP ? zhi_of(zcur[gi][1]) : kHiSym;
        const uint32_t w = words[jj], w8 = w >> 8;
        const uint32_t a0 = hsub2_u(lop3_and_or<0x000F000Fu>(w, kMagic), zl);
        const uint32_t a1 = hfma2_u(lop3_and_or<0x00F000F0u>(w, kMagic), kSixteenth, zh);
        const uint32_t a2 = hsub2_u(lop3_and_or<0x000F000Fu>(w8, kMagic), zl);
        const uint32_t a3 = hfma2_u(lop3_and_or<0x00F000F0u>(w8, kMagic), kSixteenth, zh);
        if (stp % SPG == 0)
          mma_16816_f16_zc(d, a0, a1, a2, a3, bq[2 * jj], bq[2 * jj + 1]);
        else
          mma_16816_f16(d, a0, a1, a2, a3, bq[2 * jj], bq[2 * jj + 1]);
        if ((stp + 1) % SPG == 0) {                 // a whole group: scale it in
          const float fa = scale_f((uint32_t)sca[gi * scale_row + r0]);
          const float fb = scale_f((uint32_t)scb[gi * scale_row + r0]);
          acc[0] = fmaf(fa, d[0], acc[0]);
          acc[1] = fmaf(fa, d[1], acc[1]);
          acc[2] = fmaf(fb, d[2], acc[2]);
          acc[3] = fmaf(fb, d[3], acc[3]);
        }
      }
    }
    // every lane has read the slot (its values fed the instructions above): one arrival per
    // warp releases it
    __syncwarp();
    if (lane == 0)
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(&empty_bar[st])) : "memory");
    if (++st == S) {
      st = 0;
      ph ^= 1u;
    }
    if (++j == SPT) {
      flush(SPT);
      ++t;
      j = 0;
      j0 = 0;
    }
  }
  if (n > 0 && j != 0) flush(j);

  // Final value `sum` of tile tt, row m, tile column nl, held by lane idx % 32 of a 32-value
  // pass (idx = m * 16 + nl; every lane of the warp calls this).  With gate+up the lane of
  // gate column nl < 8 takes its up value from lane + 8 and stores silu(gate) * up.
  auto store_tile_value = [&](int tt, int idx, int m, int nl, float sum) {
    const bool valid = idx < M * kTileN;
    if (p.gate_up) {
      const float up = __shfl_down_sync(0xffffffffu, sum, 8);
      if (valid && nl < 8)
        store_out_rt(p.out, (size_t)m * (N / 2) + tt * 8 + nl, silu_mul(sum, up), p.out_f32 != 0);
    } else {
      const int nn = tt * kTileN + nl;
      if (valid && nn < N) store_out_rt(p.out, (size_t)m * N + nn, sum, p.out_f32 != 0);
    }
  };

  // ---- reduction of the tiles shared between warps (shared memory) and CTAs (global)
  asm volatile("bar.sync 1, %0;" ::"r"(nth) : "memory");
  for (int pass = 0; pass < 2 && n > 0; ++pass) {
    const int tt = pass == 0 ? t_first : (we - 1) / SPT;
    if (pass == 1 && tt == t_first) break;
    const int tb = tt * SPT, te = tb + SPT;         // the tile's slots
    if (max(tb, wb) == tb && min(te, we) == te) continue;          // stored directly
    if (pass == 0 && wb > cb && wb % SPT != 0) continue;          // a lower warp reduces it
    const bool cta_whole = tb >= cb && te <= ce;
    const int region = tb < cb ? 0 : 1;
    for (int base = 0; base < M * kTileN; base += 32) {
      const int idx = base + lane;
      const int m = idx / kTileN, nl = idx - m * kTileN;
      float sum = 0.f;
      if (idx < M * kTileN) {
        for (int w2 = warp; w2 < NC; ++w2) {
          int b2, e2;
          zsplit_dev(ce - cb, NC, w2, b2, e2);
          b2 += cb;
          e2 += cb;
          if (e2 <= b2 || b2 >= te) break;
          sum += pieces[((w2 * 2 + (b2 / SPT == tt ? 0 : 1)) * M + m) * kTileN + nl];
        }
      }
      if (cta_whole) {
        store_tile_value(tt, idx, m, nl, sum);
      } else if (idx < M * kTileN) {
        __stcg(p.part + ((size_t)blockIdx.x * 2 + region) * (4 * kTileN) + m * kTileN + nl, sum);
      }
    }
    if (cta_whole) continue;
    // last arriver over the CTAs holding slots of the tile (no CTA waits for another)
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      const unsigned mine = (unsigned)(min(te, ce) - max(tb, cb));
      const unsigned prev = atomicAdd(p.counters + tt, mine);
      const bool last = prev + mine == (unsigned)SPT;
      if (last) p.counters[tt] = 0u;
      s_last[warp] = last ? 1 : 0;
    }
    __syncwarp();
    if (!s_last[warp]) continue;
    __threadfence();
    int c_lo = blockIdx.x;
    for (;;) {
      if (c_lo == 0) break;
      int b2, e2;
      zsplit_dev(p.split_count, gridDim.x, c_lo - 1, b2, e2);
      if (e2 * p.split_mult <= tb) break;
      --c_lo;
    }
    for (int base = 0; base < M * kTileN; base += 32) {
      const int idx = base + lane;
      const int m = idx / kTileN, nl = idx - m * kTileN;
      float sum = 0.f;
      if (idx < M * kTileN) {
        for (int c2 = c_lo; c2 < (int)gridDim.x; ++c2) {
          int b2, e2;
          zsplit_dev(p.split_count, gridDim.x, c2, b2, e2);
          b2 *= p.split_mult;
          e2 *= p.split_mult;
          if (b2 >= te) break;
          if (e2 <= b2) continue;
          const int r2 = tb < b2 ? 0 : 1;           // the region that CTA wrote
          sum += __ldcg(p.part + ((size_t)c2 * 2 + r2) * (4 * kTileN) + m * kTileN + nl);
        }
      }
      store_tile_value(tt, idx, m, nl, sum);
    }
  }
}

// ------------------------------------------------------------------ host side

namespace {

size_t round128(size_t x) { return (x + 127) & ~(size_t)127; }

int scale_region_bytes(int G, int prec) {
  const int es = (prec & GQ_SC_F32) ? 4 : 2, gps = gv::kSlotK / G;
  if (prec & GQ_GATE_UP) return 2 * (int)round128((size_t)gps * 8 * es);
  return (int)round128((size_t)gps * 16 * es);
}

}  // namespace

bool gemv_supported(int M, int K, int G, int prec) {
  return (prec & GQ_W4) && !(prec & (GQ_ACT_F32 | GQ_ZP_FLOAT)) && M >= 1 && M <= 4 &&
         K % gv::kSlotK == 0 && G <= gv::kSlotK;
}

int gemv_slot_bytes(int G, int prec) { return gv::kSlotCodes + scale_region_bytes(G, prec); }

size_t gemv_smem_bytes(int M, int K, int G, int prec, int consumers, int stages) {
  const size_t bands = round128((size_t)(1 + 2 * M) * act_row_words(K / kChunkK) * 4);
  const size_t ring = (size_t)stages * consumers * gemv_slot_bytes(G, prec);
  const size_t pieces = (size_t)consumers * 2 * M * kTileN * 4;
  return 128 + bands + ring + pieces;                // 128: alignment of the dynamic base
}

// Consumer warps and ring depth.  Eight consumers and the deepest ring of four to six
// stages that keeps two CTAs on an SM (so that consecutive calls overlap); where that does
// not fit, sixteen consumers and the deepest ring that fits one CTA.
int gemv_config(int M, int K, int G, int prec, size_t smem_cap, int *consumers, int *stages,
                int *ctas_per_sm) {
  const size_t half = 113u * 1024u;                // two CTAs per SM (228 KB less 1 KB each)
  for (int s = 6; s >= 4; --s)
    if (gemv_smem_bytes(M, K, G, prec, 8, s) <= half) {
      *consumers = 8;
      *stages = s;
      *ctas_per_sm = 2;
      return GQ_OK;
    }
  for (int s = gv::kMaxStages; s >= 3; --s)
    if (gemv_smem_bytes(M, K, G, prec, 16, s) <= smem_cap) {
      *consumers = 16;
      *stages = s;
      *ctas_per_sm = 1;
      return GQ_OK;
    }
  return GQ_ERR_UNSUPPORTED;
}

template <int G, int SC, bool ZP, int NC>
static cudaError_t launch_gemv_t(const Plan &pl, const CUtensorMap &map, const GemvParams &gp,
                                 cudaStream_t s) {
  auto kern = w4_gemv_kernel<G, SC, ZP, NC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid_x);
  cfg.blockDim = dim3(pl.block_threads);
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, map, gp);
}

template <int G, int SC>
static cudaError_t launch_gemv_z(const Plan &pl, int prec, const CUtensorMap &map,
                                 const GemvParams &gp, cudaStream_t s) {
  if (pl.consumers == 16) {
    if (prec & GQ_ZP) return launch_gemv_t<G, SC, true, 16>(pl, map, gp, s);
    return launch_gemv_t<G, SC, false, 16>(pl, map, gp, s);
  }
  if (prec & GQ_ZP) return launch_gemv_t<G, SC, true, 8>(pl, map, gp, s);
  return launch_gemv_t<G, SC, false, 8>(pl, map, gp, s);
}

template <int G>
static cudaError_t launch_gemv_g(const Plan &pl, int prec, const CUtensorMap &map,
                                 const GemvParams &gp, cudaStream_t s) {
  if (prec & GQ_SC_F32) return launch_gemv_z<G, kScF32>(pl, prec, map, gp, s);
  if (prec & GQ_SC_BF16) return launch_gemv_z<G, kScBF16>(pl, prec, map, gp, s);
  return launch_gemv_z<G, kScF16>(pl, prec, map, gp, s);
}

cudaError_t launch_gemv(const Plan &pl, int M, int K, int N, int G, int prec, const void *A,
                        const void *Wq, const void *scales, const void *zeros, void *out,
                        float *part, unsigned *counters, cudaStream_t s) {
  // the canonical scale matrix [K/G][N] as a 2-D tensor: 16 columns (8 for gate+up halves) x
  // the slot's groups per box
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) {
    note_cuda_error_code("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", -1);
    return cudaErrorInvalidValue;
  }
  const bool f32 = (prec & GQ_SC_F32) != 0;
  const int es = f32 ? 4 : 2;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)(K / G)};
  const cuuint64_t strides[1] = {(cuuint64_t)N * es};
  const cuuint32_t box[2] = {(cuuint32_t)((prec & GQ_GATE_UP) ? 8 : 16),
                             (cuuint32_t)(gv::kSlotK / G)};
  const cuuint32_t ones[2] = {1, 1};
  const CUresult r = enc(&map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                         2, const_cast<void *>(scales), dims, strides, box, ones,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    note_cuda_error_code("cuTensorMapEncodeTiled(scales)", (int)r);
    return cudaErrorInvalidValue;
  }
  GemvParams gp;
  gp.Wp = reinterpret_cast<const uint8_t *>(Wq);
  gp.A = reinterpret_cast<const uint16_t *>(A);
  gp.zeros = reinterpret_cast<const uint32_t *>(zeros);
  gp.out = out;
  gp.part = part;
  gp.counters = counters;
  gp.M = M;
  gp.K = K;
  gp.N = N;
  gp.split_count = pl.split_count;
  gp.split_mult = pl.split_mult;
  gp.S = pl.slots;
  gp.slot_bytes = gemv_slot_bytes(G, prec);
  gp.scale_b_off = (prec & GQ_GATE_UP) ? gv::kSlotCodes + scale_region_bytes(G, prec) / 2
                                       : gv::kSlotCodes + 8 * es;
  gp.out_f32 = (prec & GQ_OUT_F32) ? 1 : 0;
  gp.static_w = (prec & GQ_STATIC_W) ? 1 : 0;
  gp.gate_up = (prec & GQ_GATE_UP) ? 1 : 0;
  switch (G) {
    case 32: return launch_gemv_g<32>(pl, prec, map, gp, s);
    case 64: return launch_gemv_g<64>(pl, prec, map, gp, s);
    case 128: return launch_gemv_g<128>(pl, prec, map, gp, s);
    case 256: return launch_gemv_g<256>(pl, prec, map, gp, s);
    default: return cudaErrorInvalidValue;
  }
}

int gemv_read_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(g_gemv_error, &z, sizeof(int));
  }
  return v;
}

}  // namespace gq

// Warp-specialized small-M decode kernel (M <= 4) of the group-quantized weight-only GEMM.
//
// At decode the path is bound by the bytes of the packed weights ("GPU Kernel 工程（09）：量化
// 与融合 kernel", section 3.2), so what matters is keeping HBM busy while spending as few
// instructions per byte as possible.  One CTA per SM, two roles:
//   producer warp   streams this CTA's slots (256 k of one 16-column tile: 2 KB of codes, a
//                   contiguous piece of the packed layout) into a ring of S stages.  A stage
//                   holds one slot per consumer warp: lane w issues consumer w's
//                   cp.async.bulk of codes, completing on that consumer's own "full" mbarrier.
//   consumer warps  first copy the group scales (and zero points) of every slot they own into
//                   a table of their own in shared memory (cp.async, once per call), then wait
//                   for a slot, decode its codes in registers (the FP16 magic-number trick of
//                   section 2.4 of the same page), multiply on tensor cores (mma.sync
//                   m16n8k16, the 16 MMA rows on the tile's columns) and release the slot on
//                   their "empty" mbarrier.
// A consumer's only per-slot bookkeeping is one wait and one arrive; address arithmetic for
// the copies lives in the producer.  One CTA per SM.  With GQ_STATIC_W the weight stream and the
// scale tables start before the wait on the previous kernel in the stream (programmatic
// dependent launch), so they overlap the previous call's tail.
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
#include <atomic>
#include <type_traits>

#include "gq_device.cuh"

namespace gq {

namespace gv {
constexpr int kSlotChunks = 4;                          // 64-k chunks per slot
constexpr int kSlotK = kSlotChunks * kChunkK;           // 256 k
constexpr int kSlotCodes = kSlotChunks * 512;           // 2 KB of codes per slot
constexpr uint32_t kMagic = 0x64006400u;                // fp16 1024 in both halves
constexpr uint32_t kSixteenth = 0x2C002C00u;            // fp16 1/16
constexpr uint32_t kLoSym = 0x64086408u;                // fp16 1024 + 8
constexpr uint32_t kHiSym = 0xD480D480u;                // fp16 -(64 + 8)
}  // namespace gv

// Sticky device-side status (GQ_ERR_TIMEOUT after a bounded wait gave up).
static __device__ int g_gemv_error;
// bounded waits: SM clock cycles before a wait gives up (about two seconds by default;
// gq_set_wait_limit changes it)
static __device__ long long g_gemv_wait_limit = 4000000000ll;
// Failure-path test (gq_set_fault_injection(GQ_FAULT_DEVICE_WAIT)): launches made while it is
// set tell every producer (GemvParams::withhold) to withhold consumer 0's first slot, so that
// consumer's bounded wait runs out.  A kernel parameter, not a device variable: the
// producer's first copies must not wait for a global load.
static std::atomic<int> g_gemv_withhold{0};

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
    if ((it & 63u) == 0u && clock64() - t0 > g_gemv_wait_limit) {
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

}  // namespace gv

struct GemvParams {
  const uint8_t *Wp;          // packed codes
  const uint16_t *A;          // activations, bf16 [M][K]
  const void *scales;         // [K/G][N]
  const uint32_t *zeros;      // [K/G][N/8] or NULL
  void *out;                  // [M][N] (gate+up: [M][N/2])
  float *part;                // [gridDim.x][2][4][16] per-CTA partial sums (shared tiles only)
  unsigned *counters;         // per-tile arrival counters (shared tiles only)
  int M, K, N;
  int split_count, split_mult;   // CTA c owns slots zsplit(split_count, grid, c) * split_mult
  int table_bytes;               // bytes of one consumer warp's scale / zero-point table
  int out_f32;
  int static_w;                  // weights may be read before the preceding kernel ends
  int gate_up;                   // fused gate+up: out[m][j] = silu(col j) * (col N/2 + j)
  int withhold;                  // failure test: withhold consumer 0's first slot
};

namespace gv {
constexpr int kConsumers = 16;                          // consumer warps per CTA
constexpr int kStages = 4;                              // ring stages (one slot per consumer each)
}  // namespace gv

// Shared memory (dynamic, base rounded up to 128 bytes): [bands][ring][tables][pieces]
//   bands   (1 + 2M) rows of act_row_words(K / 64) words: a zero row, then the two exponent
//           bands of each activation row, permuted for the B operands
//   ring    kStages x kConsumers slots of 2 KB of codes
//   tables  per consumer warp, for each of its slots in order: the slot's group scales of the
//           tile's 16 columns [G rows][16], then (INT4 zero points) the two zero-point words of
//           each group row — loaded once, before the main loop
//   pieces  kConsumers x 2 x M x 16 floats: a warp's partial sums of its first and last tile
template <int G, int SC, bool ZP>
__global__ void __launch_bounds__((gv::kConsumers + 1) * 32, 1)
    w4_gemv_kernel(const GemvParams p) {
  using namespace gv;
  constexpr int NC = kConsumers, S = kStages;
  constexpr int ES = SC == kScF32 ? 4 : 2;          // bytes per scale
  constexpr int GPS = kSlotK / G;                   // groups per slot
  constexpr int SPG = G / 16;                       // 16-k MMA steps per group
  constexpr int SCB = GPS * 16 * ES;                // table bytes of a slot's scales
  // table bytes per slot, a multiple of 16 so that every slot's scales start 16-byte aligned
  constexpr int TSB = (SCB + (ZP ? GPS * 2 * 4 : 0) + 15) & ~15;
  typedef typename std::conditional<SC == kScF32, uint32_t, unsigned short>::type sc_t;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  // full_bar[stage][w]: consumer w's slot of the stage landed; empty_bar[stage][w]: consumer
  // w released it.  Each consumer and its producer lane form an independent pipeline.
  __shared__ __align__(8) uint64_t full_bar[S][NC], empty_bar[S][NC];
  __shared__ int s_emax[4], s_emin[4];
  __shared__ int s_last[NC];
  asm volatile("griddepcontrol.launch_dependents;");

  const int M = p.M, K = p.K, N = p.N;
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
  uint8_t *tables = ring + (size_t)S * NC * kSlotCodes;
  float *pieces = reinterpret_cast<float *>(tables + (size_t)NC * p.table_bytes);

  // one (stage, consumer) pair of barriers per thread: initialised by a single thread, the 128
  // barriers held the producer's first copy back by about 1.5 us
  if (threadIdx.x < S * NC) {
    const int s = threadIdx.x / NC, w = threadIdx.x - s * NC;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&full_bar[s][w])) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&empty_bar[s][w])) : "memory");
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
    // lane w < NC streams consumer w's slots [wb, we) through ring slot (stage, w), refilling a
    // stage as soon as that consumer released it
    if (lane < NC) {
      int wb, we;
      zsplit_dev(ce - cb, NC, lane, wb, we);
      wb += cb;
      we += cb;
      const int mine = we - wb;
      const bool withhold = lane == 0 && p.withhold != 0;
      int issued = 0;
      for (int j = 0; j < mine; ++j) {
        const int st = j % S;
        if (j >= S && !wait_phase(saddr(&empty_bar[st][lane]), (uint32_t)((j / S + 1) & 1))) break;
        if (!(withhold && j == 0)) {
          const uint32_t fb = saddr(&full_bar[st][lane]);
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                       "n"(kSlotCodes)
                       : "memory");
          bulk_copy(saddr(ring + ((size_t)st * NC + lane) * kSlotCodes),
                    p.Wp + (size_t)(wb + j) * kSlotCodes, kSlotCodes, fb);
        }
        issued = j + 1;
      }
      // Before the producer leaves, every copy it issued has landed: the CTA's shared memory
      // must not be written after all of its warps are gone (a consumer that gave up never
      // waits for its later slots).  Fill f completed phase f / S of full_bar[f % S][w]; the
      // last fill of each stage is the latest phase that barrier saw.
      for (int f = max(0, issued - S); f < issued; ++f) {
        if (withhold && f == 0) continue;
        if (!wait_phase(saddr(&full_bar[f % S][lane]), (uint32_t)((f / S) & 1))) break;
      }
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

  // ---- this warp's table: for each of its slots, the group scales of the tile's columns (16
  // bytes per cp.async; gate+up: the gate columns 8t.. then the up columns N/2 + 8t..) and the
  // zero-point words; static weights (GQ_STATIC_W) are read before the preceding kernel ends
  uint8_t *tbl = tables + (size_t)warp * p.table_bytes;
  auto load_table = [&]() {
    const size_t srow = (size_t)N * ES;
    const uint8_t *sbase = reinterpret_cast<const uint8_t *>(p.scales);
    constexpr int PPS = GPS * ES;                  // 16-byte scale parts per slot
    for (int e = lane; e < n * PPS; e += 32) {
      const int i = e / PPS, pr = e - i * PPS, g = pr / ES, lp = pr - g * ES;
      const int slot = wb + i, t = slot / SPT, js = slot - t * SPT;
      size_t col_bytes = (size_t)t * kTileN * ES + lp * 16;
      if (p.gate_up)
        col_bytes = lp * 16 < 8 * ES ? (size_t)8 * t * ES + lp * 16
                                     : (size_t)(N / 2 + 8 * t) * ES + (lp * 16 - 8 * ES);
      if (lp * 16 < min(kTileN, N - t * kTileN) * ES)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                         saddr(tbl + (size_t)i * TSB + g * 16 * ES + lp * 16)),
                     "l"(sbase + (size_t)(js * GPS + g) * srow + col_bytes)
                     : "memory");
    }
    if (ZP) {
      const int NW = N >> 3;
      for (int e = lane; e < n * GPS * 2; e += 32) {
        const int i = e / (GPS * 2), pr = e - i * (GPS * 2), g = pr >> 1, h = pr & 1;
        const int slot = wb + i, t = slot / SPT, js = slot - t * SPT;
        const int word = p.gate_up ? (h ? NW / 2 + t : t) : min(2 * t + h, NW - 1);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                         saddr(tbl + (size_t)i * TSB + SCB + (g * 2 + h) * 4)),
                     "l"(p.zeros + (size_t)(js * GPS + g) * NW + word)
                     : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  if (p.static_w) load_table();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!p.static_w) load_table();

  // ---- exponent bands (the consumer warps only; the producer is already streaming).  Each
  // thread reads its 16-byte pieces of A (8 consecutive k of one row) once: for the row's
  // exponent range, then, after one barrier, to convert them (held in registers when every
  // row has at most two pieces per thread, read again from L1 otherwise).
  const int nth = NC * 32, tid = threadIdx.x;
  for (int idx = tid; idx < RS; idx += nth) bands[idx] = 0u;   // zero row 0
  const int ppr = K >> 3;                          // 16-byte pieces per row
  const int per = (ppr + nth - 1) / nth;           // pieces per thread and row
  const uint4 *A4 = reinterpret_cast<const uint4 *>(p.A);
  const bool held_all = per <= 2;
  uint4 held[4][2];
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int pc = tid + i * nth;
      held[m][i] = make_uint4(0u, 0u, 0u, 0u);
      if (held_all && m < M && i < per && pc < ppr) held[m][i] = A4[(size_t)m * ppr + pc];
    }
  auto range_of = [&](const uint4 v, unsigned &mx, unsigned &mn) {
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t mag = wv[e] & 0x7FFF7FFFu;
      const uint32_t lo = mag & 0xFFFFu, hi = mag >> 16;
      mx = max(mx, max(lo, hi));
      mn = min(mn, min(lo ? lo : 0xFFFFu, hi ? hi : 0xFFFFu));   // smallest non-zero
    }
  };
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    if (m >= M) break;
    unsigned mx = 0u, mn = 0xFFFFu;
    if (held_all) {
      range_of(held[m][0], mx, mn);
      range_of(held[m][1], mx, mn);
    } else {
      for (int pc = tid; pc < ppr; pc += nth) range_of(A4[(size_t)m * ppr + pc], mx, mn);
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    mn = __reduce_min_sync(0xffffffffu, mn);
    if (lane == 0) {
      atomicMax(&s_emax[m], (int)(mx >> 7));
      atomicMin(&s_emin[m], (int)(mn >> 7));
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(nth) : "memory");
  // piece pc (k = 8 pc .. 8 pc + 7) of row m, band b: its four words go to base(pc) + 0, 4,
  // 8, 12 of the band row
  auto convert = [&](const uint4 vv, int m, int b, int pc) {
    const int emax = s_emax[m], emin = s_emin[m];
    const int nbu = emin > emax ? 0 : min(2, ((emax - emin) >> 5) + 1);
    const int sb_ = 142 - emax + 32 * b;           // scale exponent of band b
    uint32_t *brw = bands + (1 + 2 * m + b) * RS;
    const bool fast = nbu == 1 && emax < 255;
    const int s1 = sb_ / 2, s2 = sb_ - s1;
    const float c1 = __int_as_float((127 + s1) << 23), c2 = __int_as_float((127 + s2) << 23);
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
  };
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    if (m >= M) break;
    const int emax = s_emax[m], emin = s_emin[m];
    const int nbu = emin > emax ? 0 : min(2, ((emax - emin) >> 5) + 1);
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      if (b >= nbu) break;
      if (held_all) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int pc = tid + i * nth;
          if (i < per && pc < ppr) convert(held[m][i], m, b, pc);
        }
      } else {
        for (int pc = tid; pc < ppr; pc += nth) convert(A4[(size_t)m * ppr + pc], m, b, pc);
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // this lane's table copies landed
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
  auto scale_f = [&](uint32_t bits) -> float {
    if (SC == kScF32) return __uint_as_float(bits);
    if (SC == kScBF16) return __uint_as_float(bits << 16);
    return __half2float(__ushort_as_half((unsigned short)bits));
  };
  const int t_first = wb / SPT;
  int t = t_first, j = wb - t_first * SPT;
  int j0 = j;                                      // first slot of this warp's share of t

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

  const uint8_t *ringw = ring + (size_t)warp * kSlotCodes;
  const uint8_t *ts = tbl;                         // the current slot's table entry
  const uint32_t *bslot = brow + j * (kSlotChunks * 32);
  // the current group's MMA accumulator (a group may span chunks, never a slot: G <= 256;
  // two accumulators alternating by step measured slower here: the consumers are bound by
  // instruction issue, not by the MMA chain's latency)
  float d[4];
  for (int i = 0; i < n; ++i) {
    const int st = i % S;
    if (!wait_phase(saddr(&full_bar[st][warp]), (uint32_t)((i / S) & 1))) break;
    const uint8_t *slot = ringw + (size_t)st * (NC * kSlotCodes);
    const sc_t *sg = reinterpret_cast<const sc_t *>(ts);
    const uint32_t *zt = reinterpret_cast<const uint32_t *>(ts + SCB);
#pragma unroll
    for (int ch = 0; ch < kSlotChunks; ++ch) {
      const uint4 wv = *reinterpret_cast<const uint4 *>(slot + ch * 512 + lane * 16);
      const uint4 blo = *reinterpret_cast<const uint4 *>(bslot + ch * 32);
      const uint4 bhi = *reinterpret_cast<const uint4 *>(bslot + ch * 32 + 16);
      const uint32_t bq[8] = {blo.x, blo.y, blo.z, blo.w, bhi.x, bhi.y, bhi.z, bhi.w};
      const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int stp = ch * 4 + jj;                 // compile-time 16-k step of the slot
        const int gi = stp / SPG;
        // fp16(1024 + z) and fp16(-(64 + z)) in both halves, z of the tile's columns r0 and
        // r0 + 8 (nibble r0 of the group's two zero-point words)
        const uint32_t zl = ZP ? (0x6400u | ((zt[2 * gi] >> (4 * r0)) & 0xFu)) * 0x00010001u : kLoSym;
        const uint32_t zh = ZP ? (0xD400u | (((zt[2 * gi + 1] >> (4 * r0)) & 0xFu) << 4)) * 0x00010001u
                               : kHiSym;
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
          const float fa = scale_f((uint32_t)sg[gi * 16 + r0]);
          const float fb = scale_f((uint32_t)sg[gi * 16 + r0 + 8]);
          acc[0] = fmaf(fa, d[0], acc[0]);
          acc[1] = fmaf(fa, d[1], acc[1]);
          acc[2] = fmaf(fb, d[2], acc[2]);
          acc[3] = fmaf(fb, d[3], acc[3]);
        }
      }
    }
    // every lane has read the slot (its values fed the instructions above): one arrival
    // releases it to the producer lane
    __syncwarp();
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.eq.u32 p, %1, 0;\n\t"
        "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(saddr(&empty_bar[st][warp])),
        "r"(lane)
        : "memory");
    ts += TSB;
    bslot += kSlotChunks * 32;
    if (++j == SPT) {
      flush(SPT);
      ++t;
      j = 0;
      j0 = 0;
      bslot = brow;
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

int table_slot_bytes(int G, int prec) {
  const int es = (prec & GQ_SC_F32) ? 4 : 2, gps = gv::kSlotK / G;
  return (gps * 16 * es + ((prec & GQ_ZP) ? gps * 2 * 4 : 0) + 15) & ~15;
}

}  // namespace

bool gemv_supported(int M, int K, int G, int prec) {
  return (prec & GQ_W4) && !(prec & (GQ_ACT_F32 | GQ_ZP_FLOAT)) && M >= 1 && M <= 4 &&
         K % gv::kSlotK == 0 && G <= gv::kSlotK;
}

// Bytes of one consumer warp's table for a CTA holding at most max_cta_slots slots.
int gemv_table_bytes(int G, int prec, int max_cta_slots) {
  const int per_warp = (max_cta_slots + gv::kConsumers - 1) / gv::kConsumers;
  return (int)(((size_t)per_warp * table_slot_bytes(G, prec) + 15) & ~(size_t)15);
}

size_t gemv_smem_bytes(int M, int K, int G, int prec, int max_cta_slots) {
  const size_t bands = round128((size_t)(1 + 2 * M) * act_row_words(K / kChunkK) * 4);
  const size_t ring = (size_t)gv::kStages * gv::kConsumers * gv::kSlotCodes;
  const size_t tables = (size_t)gv::kConsumers * gemv_table_bytes(G, prec, max_cta_slots);
  const size_t pieces = (size_t)gv::kConsumers * 2 * M * kTileN * 4;
  return 128 + bands + ring + tables + pieces;       // 128: alignment of the dynamic base
}

int gemv_threads() { return (gv::kConsumers + 1) * 32; }

template <int G, int SC, bool ZP>
static cudaError_t launch_gemv_t(const Plan &pl, const GemvParams &gp, cudaStream_t s) {
  auto kern = w4_gemv_kernel<G, SC, ZP>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       pl.smem_bytes);
  if (e != cudaSuccess) return e;
  // programmatic stream serialization: the next kernel may begin launching while this one
  // runs; this kernel reads activations and writes outputs only after griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid_x);
  cfg.blockDim = dim3(gemv_threads());
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, gp);
}

template <int G, int SC>
static cudaError_t launch_gemv_z(const Plan &pl, int prec, const GemvParams &gp, cudaStream_t s) {
  if (prec & GQ_ZP) return launch_gemv_t<G, SC, true>(pl, gp, s);
  return launch_gemv_t<G, SC, false>(pl, gp, s);
}

template <int G>
static cudaError_t launch_gemv_g(const Plan &pl, int prec, const GemvParams &gp, cudaStream_t s) {
  if (prec & GQ_SC_F32) return launch_gemv_z<G, kScF32>(pl, prec, gp, s);
  if (prec & GQ_SC_BF16) return launch_gemv_z<G, kScBF16>(pl, prec, gp, s);
  return launch_gemv_z<G, kScF16>(pl, prec, gp, s);
}

cudaError_t launch_gemv(const Plan &pl, int M, int K, int N, int G, int prec, const void *A,
                        const void *Wq, const void *scales, const void *zeros, void *out,
                        float *part, unsigned *counters, cudaStream_t s) {
  GemvParams gp;
  gp.Wp = reinterpret_cast<const uint8_t *>(Wq);
  gp.A = reinterpret_cast<const uint16_t *>(A);
  gp.scales = scales;
  gp.zeros = reinterpret_cast<const uint32_t *>(zeros);
  gp.out = out;
  gp.part = part;
  gp.counters = counters;
  gp.M = M;
  gp.K = K;
  gp.N = N;
  gp.split_count = pl.split_count;
  gp.split_mult = pl.split_mult;
  gp.table_bytes = pl.table_bytes;
  gp.out_f32 = (prec & GQ_OUT_F32) ? 1 : 0;
  gp.static_w = (prec & GQ_STATIC_W) ? 1 : 0;
  gp.gate_up = (prec & GQ_GATE_UP) ? 1 : 0;
  gp.withhold = g_gemv_withhold.load(std::memory_order_relaxed);
  switch (G) {
    case 32: return launch_gemv_g<32>(pl, prec, gp, s);
    case 64: return launch_gemv_g<64>(pl, prec, gp, s);
    case 128: return launch_gemv_g<128>(pl, prec, gp, s);
    case 256: return launch_gemv_g<256>(pl, prec, gp, s);
    default: return cudaErrorInvalidValue;
  }
}

int gemv_set_wait_limit(long long cycles) {
  return cudaMemcpyToSymbol(g_gemv_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? 0 : -1;
}

int gemv_set_withhold(bool on) {
  g_gemv_withhold.store(on ? 1 : 0, std::memory_order_relaxed);
  return 0;
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

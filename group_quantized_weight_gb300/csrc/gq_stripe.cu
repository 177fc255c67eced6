// Striped small-M decode kernel (M <= 8) of the group-quantized weight-only GEMM.
//
// Work partition.  The packed weights are a sequence of 16-column tiles, each tile's K
// contiguous, so the flattened sequence of (tile, slot) pairs — a slot is 256 consecutive k
// of one tile, 2 KB of codes — is one contiguous byte stream.  CTA c (one per SM) owns a
// contiguous range of slots and its 24 warps split that range into contiguous sub-ranges
// (the striped partitioning of "GPU Kernel 工程（09）：量化与融合 kernel", section 3.3 item 4:
// every SM gets the same amount of work for any shape).  When there are enough tiles the
// CTA ranges are whole tiles, so no tile is shared between SMs; otherwise they are equal
// slot ranges and a tile may be shared by neighbouring CTAs.  Every partial sum is a sum of
// whole scaled groups, combined in a fixed order (warps in order inside a CTA, then CTAs in
// order), so the result is bitwise reproducible.
//
// Streaming.  Each warp owns a ring of S shared-memory slots.  Lane 0 fills a slot with TMA
// bulk copies (cp.async.bulk, completion counted in bytes on the slot's mbarrier): the
// slot's 2 KB of packed codes and, per group, the scales of the tile's 16 columns.  A slot
// is refilled with the slot S ahead as soon as the warp has decoded it.
//
// Decode: the FP16 form of the magic-number trick of section 2.4 of the same page, one
// shift per eight codes: (w & 0x000F000F) | 0x64006400 is fp16(1024 + q) for the codes in
// bits 0-3 and 16-19, one fp16x2 subtraction of fp16(1024 + z) leaves q - z;
// (w & 0x00F000F0) | 0x64006400 is fp16(1024 + 16q) for bits 4-7 and 20-23, and one fp16x2
// FMA with 1/16 and -(64 + z) leaves q - z; w >> 8 exposes the other four codes.  Every
// value is an exact small integer.
//
// The MMA is FP16 x FP16 -> FP32 (mma.sync m16n8k16) with the 16 MMA rows on the tile's 16
// output columns, so the bf16 activations are carried into fp16 exactly by exponent bands:
// for activation row m with largest exponent field Emax, band b (b = 0, 1) holds the
// elements whose exponent field lies in (Emax - 32(b+1), Emax - 32b], scaled by
// 2^(142 - Emax + 32b) so that they land in [2^-16, 2^16) where fp16 represents every bf16
// significand exactly.  Row m's two bands are MMA columns 2m and 2m + 1; the column sums
// are scaled back by the inverse powers of two and added band 0 first.  Every activation
// larger than 2^-64 times its row's largest one is represented exactly; smaller ones are
// treated as zero.  Each group starts a fresh FP32 accumulator (zero input) and is
// multiplied by its scale after its last MMA step.
//
// The kernel is launched with programmatic stream serialization: it lets the next kernel
// in the stream start launching at once, and it reads none of its inputs and writes none
// of its outputs before griddepcontrol.wait (the end of the previous kernel).
#include <type_traits>

#include "gq_device.cuh"

namespace gq {

constexpr int kSlotChunks = 4;                          // 64-k chunks per slot
constexpr int kSlotK = kSlotChunks * kChunkK;           // 256 k
constexpr int kMaxSlots = 3;                            // ring slots per warp
// bounded waits: SM clock cycles before a wait gives up (about two seconds by default;
// gq_set_wait_limit changes it)
static __device__ long long g_stripe_wait_limit = 4000000000ll;

// Sticky device-side status of this kernel (GQ_ERR_TIMEOUT after a bounded wait gave up),
// read by the host through stripe_read_error.
static __device__ int g_stripe_error;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Wait until the mbarrier phase of parity `parity` completes.  Bounded: after about two
// seconds it records GQ_ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool slot_wait(uint32_t bar, uint32_t parity) {
  long long t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (it == 0) {
      t0 = clock64();
    } else if ((it & 63u) == 0u && clock64() - t0 > g_stripe_wait_limit) {
      atomicExch(&g_stripe_error, GQ_ERR_TIMEOUT);
      return false;
    }
  }
}

// decode constants (fp16x2 bit patterns)
constexpr uint32_t kMagic = 0x64006400u;       // 1024 in both halves
constexpr uint32_t kSixteenth = 0x2C002C00u;   // 1/16
constexpr uint32_t kLoSym = 0x64086408u;       // 1024 + 8: the symmetric zero point
constexpr uint32_t kHiSym = 0xD480D480u;       // -(64 + 8)

struct StripeParams {
  const uint8_t *Wp;          // packed codes
  const uint16_t *A;          // activations, bf16 [M][K]
  const void *scales;         // [K/G][N]
  const uint32_t *zeros;      // [K/G][N/8] or NULL
  void *out;                  // [M][N]
  float *part;                // [gridDim.x][2][8][16] per-CTA partial sums of the tile a CTA
                              // starts inside and the tile it ends inside (shared tiles only)
  unsigned *counters;         // per-tile arrival counters (shared tiles only)
  int M, K, N;
  int split_count, split_mult;   // CTA c owns slots zsplit(split_count, grid, c) * split_mult
  int S;                         // ring slots per warp
  int out_f32;
  int static_w;                  // weights may be read before the preceding kernel ends
  int gate_up;                   // fused gate+up: out[m][j] = silu(col j) * (col N/2 + j)
};

// Shared-memory layout (dynamic): [bands][rings][pieces]
//   bands  (1 + 2M) rows of act_row_words(K / 64) words: a zero row, then two exponent
//          bands per activation row, permuted so that a lane gets the B operands of four
//          consecutive 16-k MMA steps with two 16-byte loads
//   rings  kStrWarps x S slots of slot_bytes: 2 KB of codes, then the group scales
//   pieces kStrWarps x 2 x M x 16 floats: a warp's partial sums of its first and last tile
__host__ __device__ constexpr int stripe_groups_per_slot(int G) { return kSlotK / G; }
__host__ __device__ constexpr int stripe_slot_bytes(int G, int es) {
  return kSlotChunks * 512 + stripe_groups_per_slot(G) * 16 * es;
}

template <int G, int SC, bool ZP, int MT>
__global__ void __launch_bounds__(kStrWarps * 32, 1) w4_stripe_kernel(const StripeParams p) {
  constexpr int ES = SC == kScF32 ? 4 : 2;          // bytes per scale
  constexpr int GPS = stripe_groups_per_slot(G);    // groups per slot
  constexpr int SPG = G / 16;                       // 16-k MMA steps per group
  constexpr int SLOTB = stripe_slot_bytes(G, ES);
  constexpr int LPG = ES;                           // 16-byte parts per group's 16 scales
  constexpr int NL = GPS * LPG;                     // lanes copying scales (at most 32)
  static_assert(NL <= 32, "one 16-byte scale part per lane");
  typedef typename std::conditional<SC == kScF32, uint32_t, unsigned short>::type sc_t;

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kStrWarps][kMaxSlots];
  __shared__ int s_emax[8], s_emin[8];
  asm volatile("griddepcontrol.launch_dependents;");

  const int M = p.M, K = p.K, N = p.N, S = p.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = lane >> 2, q = lane & 3;
  const int C = K / kChunkK;                        // chunks per tile
  const int SPT = K / kSlotK;                       // slots per tile
  int cb, ce;                                       // this CTA's slots
  zsplit_dev(p.split_count, gridDim.x, blockIdx.x, cb, ce);
  cb *= p.split_mult;
  ce *= p.split_mult;
  int wb, we;                                       // this warp's slots
  zsplit_dev(ce - cb, kStrWarps, warp, wb, we);
  wb += cb;
  we += cb;
  const int n = we - wb;

  const int RS = act_row_words(C);
  uint32_t *bands = reinterpret_cast<uint32_t *>(smem);
  uint8_t *rings = smem + (((size_t)(1 + 2 * M) * RS * 4 + 127) & ~(size_t)127);
  uint8_t *ring = rings + (size_t)warp * S * SLOTB;
  float *pieces = reinterpret_cast<float *>(rings + (size_t)kStrWarps * S * SLOTB);

  if (threadIdx.x < 8) {
    s_emax[threadIdx.x] = 0;
    s_emin[threadIdx.x] = 255;
  }
  if (lane == 0) {
    for (int s = 0; s < S; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&bars[warp][s])),
                   "n"(1 + NL)
                   : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // inputs written by the preceding kernel are read only after it has ended; static weights
  // (GQ_STATIC_W) start streaming before that
  if (!p.static_w) asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- the load side: the next slot of this warp's range into the next ring slot.  One lane
  // issues the bulk copy of the slot's 2 KB of codes (operands broadcast from lane 0, so the
  // compiler sees them warp-uniform); lanes 0 .. NL-1 each copy 16 bytes of the slot's group
  // scales with cp.async and report completion on the slot's mbarrier
  // (cp.async.mbarrier.arrive.noinc), which therefore expects 1 + NL arrivals per phase.
  // Source pointers advance by a fixed stride per slot and are recomputed at tile changes.
  const size_t srow = (size_t)N * ES;               // bytes per scale row
  const uint8_t *hw = p.Wp + (size_t)wb * (kSlotChunks * 512);
  int ht = wb / SPT, hj = wb - ht * SPT, hs = 0;
  const int lg = lane / LPG, lp = lane - lg * LPG;  // this lane's scale group and 16-byte part
  const uint8_t *lsc = nullptr;                     // this lane's scale source in the head slot
  bool lcopy = false;                               // the part lies inside the tile's columns
  auto head_tile = [&]() {
    // byte offset of this lane's 16-byte part of the tile's scale row: columns 16 ht .. +15,
    // or with gate+up the gate columns 8 ht .. +7 then the up columns N/2 + 8 ht .. +7
    size_t col_bytes = (size_t)ht * kTileN * ES + lp * 16;
    if (p.gate_up && lp * 16 >= 8 * ES) col_bytes = (size_t)(N / 2 + 8 * ht) * ES + (lp * 16 - 8 * ES);
    else if (p.gate_up) col_bytes = (size_t)8 * ht * ES + lp * 16;
    lsc = reinterpret_cast<const uint8_t *>(p.scales) + (size_t)(hj * GPS + lg) * srow + col_bytes;
    lcopy = lane < NL && lp * 16 < min(kTileN, N - ht * kTileN) * ES;
  };
  head_tile();
  auto issue_next = [&]() {
    const uint32_t bar = smem_addr(&bars[warp][hs]);
    const uint32_t dst = smem_addr(ring + hs * SLOTB);
    const uint32_t ubar = __shfl_sync(0xffffffffu, bar, 0);
    const uint32_t udst = __shfl_sync(0xffffffffu, dst, 0);
    const unsigned long long usrc = __shfl_sync(0xffffffffu, (unsigned long long)hw, 0);
    if (lane == 0) {
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(ubar),
                   "n"(kSlotChunks * 512)
                   : "memory");
      asm volatile(
          "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(udst),
          "l"(usrc), "n"(kSlotChunks * 512), "r"(ubar)
          : "memory");
    }
    if (lane < NL) {
      if (lcopy)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + kSlotChunks * 512 + lg * 16 * ES + lp * 16),
                     "l"(lsc)
                     : "memory");
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
    }
    hw += kSlotChunks * 512;
    if (++hj == SPT) {
      hj = 0;
      ++ht;
      head_tile();
    } else {
      lsc += GPS * srow;
    }
    hs = hs + 1 == S ? 0 : hs + 1;
  };
  for (int i = 0; i < S && i < n; ++i) issue_next();
  if (p.static_w) asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- stage A: exponent bands as fp16, permuted for the B operands.  Each thread reads
  // 16-byte pieces of A (8 consecutive k of one row) from global memory: once for the row's
  // exponent range, once more to convert and store them.
  for (int idx = threadIdx.x; idx < RS; idx += blockDim.x) bands[idx] = 0u;   // zero row 0
  const int ppr = K >> 3;                          // pieces per row
  const uint4 *A4 = reinterpret_cast<const uint4 *>(p.A);
  // exponent range of each row: the magnitude bits (bits & 0x7FFF) order like the values
  for (int m = 0; m < M; ++m) {
    unsigned mx = 0u, mn = 0xFFFFu;
    for (int pc = threadIdx.x; pc < ppr; pc += blockDim.x) {
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
  __syncthreads();
  // band row 1 + 2m + b holds band b of activation row m (only if the row needs it).  The
  // four words of piece pc (k = 8 pc .. 8 pc + 7) go to base(pc) + 0, 4, 8, 12 of the row.
  for (int v = 0; v < 2 * M; ++v) {
    const int m = v >> 1, b = v & 1;
    const int emax = s_emax[m], emin = s_emin[m];
    const int nbu = emin > emax ? 0 : min(2, ((emax - emin) >> 5) + 1);
    if (b >= nbu) continue;
    const int sb_ = 142 - emax + 32 * b;           // scale exponent of band b
    uint32_t *brw = bands + (1 + v) * RS;
    const bool fast = nbu == 1 && emax < 255;
    // every non-zero element of a single-band row lies in band 0: scale them all by 2^sb
    // (two exact power-of-two products, each factor a normal float) and round to fp16, which
    // is exact for bf16 significands in [2^-16, 2^16)
    const int s1 = sb_ / 2, s2 = sb_ - s1;
    const float c1 = __int_as_float((127 + s1) << 23), c2 = __int_as_float((127 + s2) << 23);
    for (int pc = threadIdx.x; pc < ppr; pc += blockDim.x) {
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
  __syncthreads();

  // B-operand rows of this lane (MMA column r0 of each block = band r0 % 2 of row r0 / 2),
  // or the zero row
  const uint32_t *brow[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int m = mt * 4 + (r0 >> 1), b = r0 & 1;
    int row = 0;
    if (m < M) {
      const int emax = s_emax[m], emin = s_emin[m];
      const int nbu = emin > emax ? 0 : min(2, ((emax - emin) >> 5) + 1);
      if (b < nbu) row = 1 + 2 * m + b;
    }
    brow[mt] = bands + row * RS + q * 4;
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
  // zero-point words of the slot (tile tz, slot jz of the tile): groups jz * GPS + gi,
  // column words 2 tz and 2 tz + 1
  auto load_zeros = [&](int tz, int jz, uint32_t (&z)[GPS][2]) {
#pragma unroll
    for (int gi = 0; gi < GPS; ++gi) {
      const uint32_t *zr = p.zeros + (size_t)(jz * GPS + gi) * NW;
      // the words of the tile's columns r0 and r0 + 8 (gate+up: gate word tz, up word
      // N/16 + tz)
      z[gi][0] = __ldg(zr + min(p.gate_up ? tz : 2 * tz, NW - 1));
      z[gi][1] = __ldg(zr + min(p.gate_up ? NW / 2 + tz : 2 * tz + 1, NW - 1));
    }
  };
  const int t_first = wb / SPT;
  int t = t_first, j = wb - t_first * SPT;
  int j0 = j;                                      // first slot of this warp's share of t
  uint32_t zcur[GPS][2], znext[GPS][2];
  if (ZP && n > 0) load_zeros(t, j, znext);

  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  // End of the warp's share of tile t (slots j0 .. j1 - 1): combine the bands, then store
  // a whole tile or keep the share's partial sums for the CTA's reduction.
  auto flush = [&](int j1) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      // lane (r0, q) holds columns 2q, 2q + 1 (both bands of row mt * 4 + q) of the tile's
      // columns r0 and r0 + 8
      const int mrow = mt * 4 + q;
      const int emax = mrow < M ? s_emax[mrow] : 127;
      const float v0 = scale_pow2(acc[mt][0], emax - 142) + scale_pow2(acc[mt][1], emax - 174);
      const float v1 = scale_pow2(acc[mt][2], emax - 142) + scale_pow2(acc[mt][3], emax - 174);
      acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      if (mrow >= M) continue;
      if (j0 == 0 && j1 == SPT) {
        if (p.gate_up) {                           // v0 is gate column 8t + r0, v1 its up column
          store_out_rt(p.out, (size_t)mrow * (N / 2) + t * 8 + r0, silu_mul(v0, v1),
                       p.out_f32 != 0);
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
    }
  };

  int s = 0;
  uint32_t ph = 0;
  for (int i = 0; i < n; ++i) {
    slot_wait(smem_addr(&bars[warp][s]), ph);
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
    const uint8_t *slot = ring + (size_t)s * SLOTB;
    const uint8_t *ssc = slot + kSlotChunks * 512;          // the slot's scales
    // a group's MMA accumulators (a group may span chunks; never a slot: G <= 256)
    float d[MT][4];
#pragma unroll
    for (int ch = 0; ch < kSlotChunks; ++ch) {
      const uint4 wv = *reinterpret_cast<const uint4 *>(slot + ch * 512 + lane * 16);
      uint32_t bq[MT][8];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint32_t *bp = brow[mt] + (j * kSlotChunks + ch) * 32;
        const uint4 lo = *reinterpret_cast<const uint4 *>(bp);
        const uint4 hi = *reinterpret_cast<const uint4 *>(bp + 16);
        bq[mt][0] = lo.x; bq[mt][1] = lo.y; bq[mt][2] = lo.z; bq[mt][3] = lo.w;
        bq[mt][4] = hi.x; bq[mt][5] = hi.y; bq[mt][6] = hi.z; bq[mt][7] = hi.w;
      }
      const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
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
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          if (stp % SPG == 0)
            mma_16816_f16_zc(d[mt], a0, a1, a2, a3, bq[mt][2 * jj], bq[mt][2 * jj + 1]);
          else
            mma_16816_f16(d[mt], a0, a1, a2, a3, bq[mt][2 * jj], bq[mt][2 * jj + 1]);
        }
        if ((stp + 1) % SPG == 0) {                 // a whole group: scale it in
          const sc_t *sg = reinterpret_cast<const sc_t *>(ssc + gi * 16 * ES);
          const float fa = scale_f((uint32_t)sg[r0]), fb = scale_f((uint32_t)sg[r0 + 8]);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            acc[mt][0] = fmaf(fa, d[mt][0], acc[mt][0]);
            acc[mt][1] = fmaf(fa, d[mt][1], acc[mt][1]);
            acc[mt][2] = fmaf(fb, d[mt][2], acc[mt][2]);
            acc[mt][3] = fmaf(fb, d[mt][3], acc[mt][3]);
          }
        }
      }
    }
    // every lane has consumed the slot (its shared-memory reads fed the instructions above);
    // order those generic-proxy reads before the bulk copy's writes, then refill
    __syncwarp();
    if (i + S < n) {
      if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue_next();
    }
    if (++s == S) {
      s = 0;
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
  __syncthreads();
  // A tile is reduced by the lowest warp of the CTA that holds part of it: this warp for its
  // first tile unless a lower warp ends inside that tile, and for its last tile when that
  // differs from its first.  A share that covers a whole tile was stored already.
  __shared__ int s_last[kStrWarps];
  for (int pass = 0; pass < 2 && n > 0; ++pass) {
    const int tt = pass == 0 ? t_first : (we - 1) / SPT;
    if (pass == 1 && tt == t_first) break;
    const int tb = tt * SPT, te = tb + SPT;         // the tile's slots
    if (max(tb, wb) == tb && min(te, we) == te) continue;          // stored directly
    if (pass == 0 && wb > cb && wb % SPT != 0) continue;          // a lower warp reduces it
    const bool cta_whole = tb >= cb && te <= ce;
    // region of this CTA's share of tile tt in the partial-sum buffer: one per CTA for the
    // tile it starts inside and one for the tile it ends inside
    const int region = tb < cb ? 0 : 1;
    for (int base = 0; base < M * kTileN; base += 32) {
      const int idx = base + lane;
      const int m = idx / kTileN, nl = idx - m * kTileN;
      float sum = 0.f;
      if (idx < M * kTileN) {
        // the CTA's share: warps warp, warp + 1, ... while they hold slots of the tile
        for (int w2 = warp; w2 < kStrWarps; ++w2) {
          int b2, e2;
          zsplit_dev(ce - cb, kStrWarps, w2, b2, e2);
          b2 += cb;
          e2 += cb;
          if (e2 <= b2 || b2 >= te) break;
          sum += pieces[((w2 * 2 + (b2 / SPT == tt ? 0 : 1)) * M + m) * kTileN + nl];
        }
      }
      if (cta_whole) {
        store_tile_value(tt, idx, m, nl, sum);
      } else if (idx < M * kTileN) {
        __stcg(p.part + ((size_t)blockIdx.x * 2 + region) * (8 * kTileN) + m * kTileN + nl, sum);
      }
    }
    if (cta_whole) continue;
    // Last arriver: every CTA holding part of the tile publishes its share, then adds its slot
    // count to the tile's counter; the CTA whose addition completes the tile's SPT slots adds
    // all shares in CTA order (the same order whichever CTA arrives last), stores the tile
    // and resets the counter.  No CTA waits for another.
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
    // the CTAs holding slots of the tile: a contiguous run of block indices around this one
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
          if (e2 <= b2) continue;                    // a CTA without slots
          const int r2 = tb < b2 ? 0 : 1;           // the region that CTA wrote
          sum += __ldcg(p.part + ((size_t)c2 * 2 + r2) * (8 * kTileN) + m * kTileN + nl);
        }
      }
      store_tile_value(tt, idx, m, nl, sum);
    }
  }
}

template <int G, int SC, bool ZP, int MT>
static cudaError_t launch_stripe_t(const Plan &pl, const StripeParams &sp, cudaStream_t s) {
  auto kern = w4_stripe_kernel<G, SC, ZP, MT>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       pl.smem_bytes);
  if (e != cudaSuccess) return e;
  // programmatic stream serialization: the next kernel may begin launching while this one
  // runs; this kernel touches its inputs and outputs only after griddepcontrol.wait
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
  return cudaLaunchKernelEx(&cfg, kern, sp);
}

template <int G, int SC, bool ZP>
static cudaError_t launch_stripe_m(const Plan &pl, const StripeParams &sp, cudaStream_t s) {
  if (sp.M <= 4) return launch_stripe_t<G, SC, ZP, 1>(pl, sp, s);
  return launch_stripe_t<G, SC, ZP, 2>(pl, sp, s);
}

template <int G, int SC>
static cudaError_t launch_stripe_z(const Plan &pl, int prec, const StripeParams &sp, cudaStream_t s) {
  if (prec & GQ_ZP) return launch_stripe_m<G, SC, true>(pl, sp, s);
  return launch_stripe_m<G, SC, false>(pl, sp, s);
}

template <int G>
static cudaError_t launch_stripe_g(const Plan &pl, int prec, const StripeParams &sp, cudaStream_t s) {
  if (prec & GQ_SC_F32) return launch_stripe_z<G, kScF32>(pl, prec, sp, s);
  if (prec & GQ_SC_BF16) return launch_stripe_z<G, kScBF16>(pl, prec, sp, s);
  return launch_stripe_z<G, kScF16>(pl, prec, sp, s);
}

int stripe_set_wait_limit(long long cycles) {
  return cudaMemcpyToSymbol(g_stripe_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? 0 : -1;
}

int stripe_read_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_stripe_error, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(g_stripe_error, &z, sizeof(int));
  }
  return v;
}

bool stripe_supported(int M, int K, int G, int prec) {
  return (prec & GQ_W4) && !(prec & GQ_ACT_F32) && M >= 1 && M <= 8 && K % kSlotK == 0 &&
         G <= kSlotK;
}

size_t stripe_smem_bytes(int M, int K, int G, int prec, int slots) {
  const int es = (prec & GQ_SC_F32) ? 4 : 2;
  const size_t bands =
      (((size_t)(1 + 2 * M) * act_row_words(K / kChunkK) * 4) + 127) & ~(size_t)127;
  const size_t rings = (size_t)kStrWarps * slots * stripe_slot_bytes(G, es);
  const size_t pieces = (size_t)kStrWarps * 2 * M * kTileN * 4;
  return bands + rings + pieces;
}

int stripe_slots_for(int M, int K, int G, int prec, size_t smem_cap) {
  for (int s = kMaxSlots; s >= 2; --s)
    if (stripe_smem_bytes(M, K, G, prec, s) <= smem_cap) return s;
  return 0;
}

int stripe_slot_k() { return kSlotK; }

cudaError_t launch_stripe_decode(const Plan &pl, int M, int K, int N, int G, int prec,
                                 const void *A, const void *Wq, const void *scales,
                                 const void *zeros, void *out, float *part,
                                 unsigned *counters, cudaStream_t s) {
  StripeParams sp;
  sp.Wp = reinterpret_cast<const uint8_t *>(Wq);
  sp.A = reinterpret_cast<const uint16_t *>(A);
  sp.scales = scales;
  sp.zeros = reinterpret_cast<const uint32_t *>(zeros);
  sp.out = out;
  sp.part = part;
  sp.counters = counters;
  sp.M = M;
  sp.K = K;
  sp.N = N;
  sp.split_count = pl.split_count;
  sp.split_mult = pl.split_mult;
  sp.S = pl.slots;
  sp.out_f32 = (prec & GQ_OUT_F32) ? 1 : 0;
  sp.static_w = (prec & GQ_STATIC_W) ? 1 : 0;
  sp.gate_up = (prec & GQ_GATE_UP) ? 1 : 0;
  switch (G) {
    case 32: return launch_stripe_g<32>(pl, prec, sp, s);
    case 64: return launch_stripe_g<64>(pl, prec, sp, s);
    case 128: return launch_stripe_g<128>(pl, prec, sp, s);
    case 256: return launch_stripe_g<256>(pl, prec, sp, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gq

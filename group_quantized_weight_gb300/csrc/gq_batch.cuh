// Small-batch kernel (M <= 64; rows past the striped decode kernel's reach) of the
// group-quantized weight-only GEMM.
//
// Between the single-token decode and the tensor-core prefill the weights still dominate
// the bytes (the roofline argument of "GPU Kernel 工程（09）：量化与融合 kernel", section
// 3.2: at M = 16 an INT4 layer moves about a quarter of the BF16 bytes), so this kernel,
// like the striped decode kernel, streams the packed codes once with TMA bulk copies and
// decodes them in registers.  What changes with M is the reuse of the activations: every
// 16-column tile needs all of them, so they live in shared memory, and K is cut into
// slices small enough for a 32-row activation slice to fit there.
//
// Grid: (K slice, tile range) pairs x row blocks of 32 activation rows.  CTA (s, c) holds
// activation rows m0 .. m0 + 31 of K slice s in shared memory (bf16, permuted so that a lane
// reads the B operands of four 16-k MMA steps with two 16-byte loads) and computes the
// slice's partial sums for tile range c.  Its warps (32, 24 or 16 as the rows grow) split
// the tile range into whole tiles.  Each warp streams its tiles' slots (256 k, 2 KB of codes) through a shared-memory
// ring: lane 0 issues a cp.async.bulk copy of the codes, lanes 0 .. NL-1 copy the group
// scales with cp.async, and both report on the slot's mbarrier.
//
// Decode: the BF16 form of the magic-number trick of section 2.4 of the same page, with
// each code moved to the low nibble of its 16-bit half first (the high-nibble form is not
// exact in bf16): ((w >> 4i) & 0x000F000F) | 0x43004300 is bf16(128 + q) in both halves and
// one bf16x2 subtraction of bf16(128 + z) leaves the exact integer q - z.  MMA:
// mma.sync m16n8k16 BF16 x BF16 -> FP32, the 16 MMA rows on the tile's columns, the 8 MMA
// columns on activation rows.  Each group's FP32 result is multiplied by its scale after the
// whole group (the group-wise GEMM of "04 · 分组量化 GEMM 内核", section 2).
//
// Float zero points (GQ_ZP_FLOAT; Machete's out = (w_q · w_s − w_z) @ a in section 3.4 of
// the first page): the decode leaves the code q itself, each group's FP32 dot is scaled as
// above, and the zero enters as − zf[g][n] · Σ_{k ∈ g} A[m][k], the group sums of the slice's
// activation rows formed once per CTA from its shared-memory copy.
//
// Slices are combined by the split-K of the same page, section 3.3: every warp writes its
// tile's FP32 partial sums, and the last of the K slices' warps to finish a tile adds them in
// slice order 0, 1, ... (a fixed order: bitwise reproducible).
#pragma once

#include <type_traits>

#include "gq_device.cuh"

namespace gq {

constexpr int kBtSlotK = 256;                        // k per slot (four 64-k chunks)
constexpr int kBtSlotCodes = 2048;                   // bytes of codes per slot
constexpr int kBtMaxSlots = 4;                       // ring slots per warp
constexpr int kBtRows = 32;                          // activation rows per CTA
// bounded waits: SM clock cycles before a wait gives up (about two seconds by default;
// gq_set_wait_limit changes it); one copy per translation unit, like the error word
static __device__ long long g_batch_wait_limit = 4000000000ll;

// Sticky device-side status of this kernel (GQ_ERR_TIMEOUT after a bounded wait gave up); one
// word per translation unit that instantiates the kernel (gq_batch.cu: symmetric and INT4
// zero points; gq_batch_zf.cu: float zero points), read together by batch_read_error.
static __device__ int g_batch_error;

namespace bt {

__device__ __forceinline__ void mma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the same MMA with a zero accumulator input (the first step of a group)
__device__ __forceinline__ void mma_bf16_zc(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// (a & 0x000F000F) | c in one LOP3 (the mask an immediate of the instruction, c a register)
__device__ __forceinline__ uint32_t lo_nibbles(uint32_t a, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(r) : "r"(a), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t saddr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Wait until the mbarrier phase of parity `parity` completes; bounded (about two seconds),
// then GQ_ERR_TIMEOUT is recorded and false returned.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity) {
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
    } else if ((it & 63u) == 0u && clock64() - t0 > g_batch_wait_limit) {
      atomicExch(&g_batch_error, GQ_ERR_TIMEOUT);
      return false;
    }
  }
}

constexpr uint32_t kMagic = 0x43004300u;       // bf16 128 in both halves
constexpr uint32_t kSym = 0x43084308u;         // bf16 (128 + 8): the symmetric zero point

}  // namespace bt

struct BtParams {
  const uint8_t *Wp;          // packed codes
  const uint32_t *A32;        // activations, bf16 [M][K] as pairs
  const void *scales;         // [K/G][N]
  const uint32_t *zeros;      // [K/G][N/8] INT4 zero points (packed form) or NULL
  const void *zf;             // [K/G][N] float zero points in the scales' format (float form)
  void *out;                  // [M][N]
  float *part;                // [KS][M][N] FP32 slice partial sums (KS > 1)
  unsigned *counters;         // per (row block, tile) arrival counters (KS > 1)
  int M, K, N;
  int T;                      // 16-column tiles
  int KS, KSL;                // K slices and k per slice
  int cps;                    // CTAs (tile ranges) per K slice
  int S;                      // ring slots per warp
  int out_f32;
  int static_w;               // weights may be read before the preceding kernel ends
  int gate_up;                // fused gate+up: tile t holds gate columns 8t.. and up columns
                              // N/2 + 8t..; out[m][8t + r] = silu(gate) * up, [M][N/2]
};

// Warps per CTA for MT 8-row MMA blocks of activations: as many as the registers allow
// without spills (64 registers a thread for MT = 1, 80 for MT = 2, 128 above).  The kernel
// is latency-bound (no pipe near saturation), so more warps per SM is what speeds it up.
__host__ __device__ constexpr int batch_warps(int MT) { return MT == 1 ? 32 : MT == 2 ? 24 : 16; }
__host__ __device__ constexpr int batch_mt(int M) {
  return ((M < kBtRows ? M : kBtRows) + 7) / 8;
}

__host__ __device__ constexpr int batch_groups_per_slot(int G) { return kBtSlotK / G; }
__host__ __device__ constexpr int batch_slot_bytes(int G, int es) {
  return kBtSlotCodes + batch_groups_per_slot(G) * 16 * es;
}

// bytes of the activation group sums a CTA keeps with float zero points: (KSL / G) groups x
// 8 MT rows of FP32
__host__ __device__ constexpr size_t batch_asum_bytes(int KSL, int G, int MT) {
  return (((size_t)(KSL / G) * 8 * MT * 4) + 127) & ~(size_t)127;
}

// Zero-point forms (template parameter ZM): the symmetric z = 8, packed INT4 zero points
// (GQ_ZP), float zero points subtracted after scaling (GQ_ZP_FLOAT)
enum { kZmSym = 0, kZmInt4 = 1, kZmFloat = 2 };

// Shared memory (dynamic): [activation slice: min(M, 32) rows x act_row_words(KSL / 64)]
// [float zero points only: the slice's activation group sums] [rings]
template <int G, int SC, int ZM, int MT>
__global__ void __launch_bounds__(batch_warps(MT) * 32, 1) w4_batch_kernel(const BtParams p) {
  constexpr bool ZP = ZM == kZmInt4;
  constexpr bool ZF = ZM == kZmFloat;
  using namespace bt;
  constexpr int ES = SC == kScF32 ? 4 : 2;          // bytes per scale
  constexpr int GPS = batch_groups_per_slot(G);     // groups per slot
  constexpr int SPG = G / 16;                       // 16-k MMA steps per group
  constexpr int SLOTB = batch_slot_bytes(G, ES);
  constexpr int LPG = ES;                           // 16-byte parts of a group's 16 scales
  constexpr int NL = GPS * LPG;                     // lanes copying scales
  static_assert(NL <= 32, "one 16-byte scale part per lane");
  typedef typename std::conditional<SC == kScF32, uint32_t, unsigned short>::type sc_t;

  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NWARP = batch_warps(MT);
  __shared__ __align__(8) uint64_t bars[NWARP][kBtMaxSlots];
  asm volatile("griddepcontrol.launch_dependents;");

  const int M = p.M, K = p.K, N = p.N, S = p.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = lane >> 2, q = lane & 3;
  const int ks = blockIdx.x / p.cps, c = blockIdx.x - ks * p.cps;
  const int m0 = blockIdx.y * kBtRows, Mb = min(kBtRows, M - m0);
  const int SPT = K / kBtSlotK, SPS = p.KSL / kBtSlotK;   // slots per tile, per slice
  const int C = p.KSL / kChunkK;                    // chunks per slice
  const int RS = act_row_words(C);
  int tb, te;                                       // this CTA's tiles
  zsplit_dev(p.T, p.cps, c, tb, te);
  int wtb, wte;                                     // this warp's tiles
  zsplit_dev(te - tb, NWARP, warp, wtb, wte);
  wtb += tb;
  wte += tb;
  const int nloads = (wte - wtb) * SPS;

  const int rows = M < kBtRows ? M : kBtRows;     // activation rows a CTA holds at most
  uint32_t *sA = reinterpret_cast<uint32_t *>(smem);
  const size_t act_bytes = ((size_t)rows * RS * 4 + 127) & ~(size_t)127;
  float *s_asum = reinterpret_cast<float *>(smem + act_bytes);
  uint8_t *ring = smem + act_bytes + (ZF ? batch_asum_bytes(p.KSL, G, MT) : 0) +
                  (size_t)warp * S * SLOTB;

  if (lane == 0) {
    for (int s = 0; s < S; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&bars[warp][s])),
                   "n"(1 + NL)
                   : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // inputs written by the preceding kernel are read only after it has ended; static weights
  // (GQ_STATIC_W) start streaming before that
  if (!p.static_w) asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- the load side: the next slot of this warp's tiles into the next ring slot
  const size_t srow = (size_t)N * ES;               // bytes per scale row
  const int lg = lane / LPG, lp = lane - lg * LPG;  // this lane's scale group and part
  int ht = wtb, hj = 0, hs = 0;                     // head: tile, slot of the slice, ring slot
  auto issue_next = [&]() {
    const int j = ks * SPS + hj;                    // slot within the tile
    const uint32_t bar = saddr(&bars[warp][hs]);
    const uint32_t dst = saddr(ring + hs * SLOTB);
    const uint8_t *src = p.Wp + ((size_t)ht * SPT + j) * kBtSlotCodes;
    if (lane == 0) {                                // ht, hj, hs are uniform across the warp
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                   "n"(kBtSlotCodes)
                   : "memory");
      asm volatile(
          "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
          "l"(src), "n"(kBtSlotCodes), "r"(bar)
          : "memory");
    }
    if (lane < NL) {
      // 16 bytes of group (j * GPS + lg)'s scales of the tile's columns; a ragged last tile
      // (8 columns) copies only the parts inside its columns
      // (gate+up: the first 8 columns' parts from the gate columns 8 ht.., the others from
      // the up columns N/2 + 8 ht..)
      const size_t col_bytes =
          !p.gate_up ? (size_t)ht * kTileN * ES + lp * 16
          : lp * 16 < 8 * ES ? (size_t)8 * ht * ES + lp * 16
                             : (size_t)(N / 2 + 8 * ht) * ES + (lp * 16 - 8 * ES);
      if (lp * 16 < min(kTileN, N - ht * kTileN) * ES)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                         dst + kBtSlotCodes + lg * 16 * ES + lp * 16),
                     "l"(reinterpret_cast<const uint8_t *>(p.scales) + (size_t)(j * GPS + lg) * srow +
                         col_bytes)
                     : "memory");
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
    }
    if (++hj == SPS) {
      hj = 0;
      ++ht;
    }
    hs = hs + 1 == S ? 0 : hs + 1;
  };
  for (int l = 0; l < S && l < nloads; ++l) issue_next();
  if (p.static_w) asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- the activation slice: rows m0 .. m0 + Mb - 1, k = ks KSL .. (ks + 1) KSL - 1, as
  // 16-byte pieces (8 k); the four words of piece pc go to base(pc) + 0, 4, 8, 12 of the row
  {
    // eight pieces per thread in flight at once: one global round trip per batch
    constexpr int kU = 8;
    const int ppr = p.KSL >> 3, npc = Mb * ppr;
    const uint4 *A4 = reinterpret_cast<const uint4 *>(p.A32);
    for (int base = threadIdx.x; base < npc; base += kU * blockDim.x) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = base + u * blockDim.x;
        if (idx < npc) {
          const int m = idx / ppr, pc = idx - m * ppr;
          v[u] = __ldg(A4 + ((size_t)(m0 + m) * K + (size_t)ks * p.KSL) / 8 + pc);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = base + u * blockDim.x;
        if (idx < npc) {
          const int m = idx / ppr, pc = idx - m * ppr;
          uint32_t *dst = sA + m * RS + (pc >> 3) * 32 + ((pc & 7) >> 2) * 16 +
                          ((pc >> 1) & 1) * 2 + (pc & 1);
          dst[0] = v[u].x;
          dst[4] = v[u].y;
          dst[8] = v[u].z;
          dst[12] = v[u].w;
        }
      }
    }
  }
  __syncthreads();
  if (ZF) {
    // Σ_{k ∈ group} A[m][k] of each (group gl of the slice, row ml), one warp per pair in a
    // fixed order.  The slice's chunk permutation keeps each 32-k half chunk in 16
    // consecutive words of the row, so a group is the row's words gl G/2 .. (gl + 1) G/2 - 1.
    constexpr int WPG = G / 2, RW = 8 * MT;
    const int npair = (p.KSL / G) * RW;
    for (int pr = warp; pr < npair; pr += NWARP) {
      const int gl = pr / RW, ml = pr - gl * RW;
      float v = 0.f;
      if (ml < Mb) {
        const uint32_t *w = sA + ml * RS + gl * WPG;
#pragma unroll
        for (int i = 0; i < (WPG + 31) / 32; ++i) {
          const int wi = lane + 32 * i;
          if (wi < WPG) {
            const uint32_t x = w[wi];
            v += __uint_as_float(x << 16) + __uint_as_float(x & 0xFFFF0000u);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      }
      if (lane == 0) s_asum[pr] = v;
    }
    __syncthreads();
  }

  auto zz_of = [&](uint32_t zw) -> uint32_t {      // bf16(128 + z) in both halves
    return (0x4300u | ((zw >> (4 * r0)) & 0xFu)) * 0x00010001u;
  };
  auto scale_f = [&](uint32_t bits) -> float {
    if (SC == kScF32) return __uint_as_float(bits);
    if (SC == kScBF16) return __uint_as_float(bits << 16);
    return __half2float(__ushort_as_half((unsigned short)bits));
  };
  const int NW = N >> 3;
  // zero-point words of slot jz (of the slice) of tile tz: groups, column words 2 tz, 2 tz + 1,
  // loaded a slot ahead (zn) and turned into the decode's subtrahends bf16(128 + z) once per
  // slot (zc), not at every 16-k step
  uint32_t zc[GPS][2], zn[GPS][2];
  auto load_zeros = [&](int tz, int jz) {
#pragma unroll
    for (int gi = 0; gi < GPS; ++gi) {
      const uint32_t *row = p.zeros + (size_t)((ks * SPS + jz) * GPS + gi) * NW;
      // the words of the tile's columns r0 and r0 + 8 (gate+up: gate word tz, up word
      // N/16 + tz)
      zn[gi][0] = __ldg(row + min(p.gate_up ? tz : 2 * tz, NW - 1));
      zn[gi][1] = __ldg(row + min(p.gate_up ? NW / 2 + tz : 2 * tz + 1, NW - 1));
    }
  };
  // float zero points of slot jz (of the slice) of tile tz: the raw bits for this lane's
  // columns 16 tz + r0 and 16 tz + r0 + 8 (a ragged last tile reads column N - 1 instead)
  auto load_zf = [&](int tz, int jz) {
    const sc_t *zfp = reinterpret_cast<const sc_t *>(p.zf);
    const int c0 = min(tz * kTileN + r0, N - 1), c1 = min(tz * kTileN + r0 + 8, N - 1);
#pragma unroll
    for (int gi = 0; gi < GPS; ++gi) {
      const sc_t *row = zfp + (size_t)((ks * SPS + jz) * GPS + gi) * N;
      zn[gi][0] = (uint32_t)__ldg(row + c0);
      zn[gi][1] = (uint32_t)__ldg(row + c1);
    }
  };
  if (ZP && nloads > 0) load_zeros(wtb, 0);
  if (ZF && nloads > 0) load_zf(wtb, 0);

  // B operands: activation row m0 + r0 + 8 mt of the slice, this lane's 8 words of a chunk.
  // A row past the block's last reads row 0 instead: B column r0 only reaches D column r0,
  // an output row that is never stored, so no zero fill is needed.
  const uint32_t *brow[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) brow[mt] = sA + (r0 + 8 * mt < Mb ? r0 + 8 * mt : 0) * RS + q * 4;
  const bool split = p.KS > 1;

  // ---- main loop: this warp's tiles, each over the slice's slots
  int rs = 0;
  uint32_t ph = 0;
  int l = 0;
  for (int t = wtb; t < wte; ++t) {
    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    for (int j = 0; j < SPS; ++j, ++l) {
      wait_phase(saddr(&bars[warp][rs]), ph);
      if (ZP || ZF) {
#pragma unroll
        for (int gi = 0; gi < GPS; ++gi) {
          zc[gi][0] = ZP ? zz_of(zn[gi][0]) : zn[gi][0];
          zc[gi][1] = ZP ? zz_of(zn[gi][1]) : zn[gi][1];
        }
        if (l + 1 < nloads) {
          if (ZP) {
            if (j + 1 < SPS) load_zeros(t, j + 1);
            else load_zeros(t + 1, 0);
          } else {
            if (j + 1 < SPS) load_zf(t, j + 1);
            else load_zf(t + 1, 0);
          }
        }
      }
      const uint8_t *slot = ring + rs * SLOTB;
      const uint8_t *ssc = slot + kBtSlotCodes;
      // a group's MMA accumulators (a group may span chunks; never a slot: G <= 256)
      float d[MT][4];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const uint4 wv = *reinterpret_cast<const uint4 *>(slot + ch * 512 + lane * 16);
        uint32_t bq[MT][8];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t *bp = brow[mt] + (j * 4 + ch) * 32;
          const uint4 lo = *reinterpret_cast<const uint4 *>(bp);
          const uint4 hi = *reinterpret_cast<const uint4 *>(bp + 16);
          bq[mt][0] = lo.x; bq[mt][1] = lo.y; bq[mt][2] = lo.z; bq[mt][3] = lo.w;
          bq[mt][4] = hi.x; bq[mt][5] = hi.y; bq[mt][6] = hi.z; bq[mt][7] = hi.w;
        }
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int stp = ch * 4 + jj;               // 16-k step of the slot
          const int gi = stp / SPG;
          // float zero points: the codes themselves (z = 0); the zero enters after scaling
          const uint32_t z0 = ZP ? zc[gi][0] : ZF ? kMagic : kSym;
          const uint32_t z1 = ZP ? zc[gi][1] : ZF ? kMagic : kSym;
          const uint32_t w = words[jj];
          // pair i of the word (bits 4i and 4i + 16): rows r0 + 8 (i & 1), k half i >> 1
          const uint32_t a0 = bsub2(lo_nibbles(w, kMagic), z0);
          const uint32_t a1 = bsub2(lo_nibbles(w >> 4, kMagic), z1);
          const uint32_t a2 = bsub2(lo_nibbles(w >> 8, kMagic), z0);
          const uint32_t a3 = bsub2(lo_nibbles(w >> 12, kMagic), z1);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if (stp % SPG == 0)
              mma_bf16_zc(d[mt], a0, a1, a2, a3, bq[mt][2 * jj], bq[mt][2 * jj + 1]);
            else
              mma_bf16(d[mt], a0, a1, a2, a3, bq[mt][2 * jj], bq[mt][2 * jj + 1]);
          }
          if ((stp + 1) % SPG == 0) {                // a whole group: scale it in
            const sc_t *sg = reinterpret_cast<const sc_t *>(ssc + gi * 16 * ES);
            const float fa = scale_f((uint32_t)sg[r0]), fb = scale_f((uint32_t)sg[r0 + 8]);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              acc[mt][0] = fmaf(fa, d[mt][0], acc[mt][0]);
              acc[mt][1] = fmaf(fa, d[mt][1], acc[mt][1]);
              acc[mt][2] = fmaf(fb, d[mt][2], acc[mt][2]);
              acc[mt][3] = fmaf(fb, d[mt][3], acc[mt][3]);
            }
            if (ZF) {                                // - zf[g][n] * Σ_{k ∈ g} A[m][k]
              const float za = scale_f(zc[gi][0]), zb = scale_f(zc[gi][1]);
              const float *as = s_asum + (j * GPS + gi) * (8 * MT) + 2 * q;
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                const float a0 = as[8 * mt], a1 = as[8 * mt + 1];
                acc[mt][0] = fmaf(-za, a0, acc[mt][0]);
                acc[mt][1] = fmaf(-za, a1, acc[mt][1]);
                acc[mt][2] = fmaf(-zb, a0, acc[mt][2]);
                acc[mt][3] = fmaf(-zb, a1, acc[mt][3]);
              }
            }
          }
        }
      }
      // every lane has consumed the slot; order those generic-proxy reads before the bulk
      // copy's writes, then refill
      __syncwarp();
      if (l + S < nloads) {
        if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_next();
      }
      if (++rs == S) {
        rs = 0;
        ph ^= 1u;
      }
    }
    // D fragment: e = 0, 1 -> column 16 t + r0, e = 2, 3 -> column 16 t + r0 + 8; rows
    // m0 + 8 mt + 2 q + (e & 1)
    // gate+up: e = 0, 1 hold gate column 8 t + r0 of rows 2 q, 2 q + 1 and e = 2, 3 the matching
    // up column, so each lane stores silu(gate) * up for two rows of out [M][N/2]
    auto store_pairs = [&](const float (&v)[MT][4]) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ml = 8 * mt + 2 * q + e;
          if (ml < Mb)
            store_out_rt(p.out, (size_t)(m0 + ml) * (N / 2) + 8 * t + r0,
                         silu_mul(v[mt][e], v[mt][e + 2]), p.out_f32 != 0);
        }
    };
    if (!split) {
      if (p.gate_up) {
        store_pairs(acc);
        continue;
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = t * kTileN + r0 + 8 * (e >> 1);
          const int ml = 8 * mt + 2 * q + (e & 1);
          if (n < N && ml < Mb)
            store_out_rt(p.out, (size_t)(m0 + ml) * N + n, acc[mt][e], p.out_f32 != 0);
        }
      continue;
    }
    // split K: write this slice's partial sums of tile t; the last of the KS warps (one per
    // K slice) to finish the tile adds the slices in the fixed order 0, 1, ..., so the
    // reduction is spread over the run instead of forming a tail at its end
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = t * kTileN + r0 + 8 * (e >> 1);
        const int ml = 8 * mt + 2 * q + (e & 1);
        if (n < N && ml < Mb) p.part[(size_t)ks * M * N + (size_t)(m0 + ml) * N + n] = acc[mt][e];
      }
    __threadfence();                // this lane's partials visible device-wide
    __syncwarp();
    unsigned last = 0u;
    if (lane == 0) {
      unsigned *ctr = p.counters + (size_t)blockIdx.y * p.T + t;
      last = atomicAdd(ctr, 1u) == (unsigned)(p.KS - 1) ? 1u : 0u;
      if (last) *ctr = 0u;          // every slice of this tile has arrived: reset
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) continue;
    __threadfence();
    float tot[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = t * kTileN + r0 + 8 * (e >> 1);
        const int ml = 8 * mt + 2 * q + (e & 1);
        float sum = 0.f;
        if (n < N && ml < Mb) {
          const size_t o = (size_t)(m0 + ml) * N + n;
#pragma unroll 4
          for (int s2 = 0; s2 < p.KS; ++s2)
            sum += s2 == ks ? acc[mt][e] : __ldcg(p.part + (size_t)s2 * M * N + o);
          if (!p.gate_up) store_out_rt(p.out, o, sum, p.out_f32 != 0);
        }
        tot[mt][e] = sum;
      }
    if (p.gate_up) store_pairs(tot);
  }
}

template <int G, int SC, int ZM, int MT>
static cudaError_t launch_bt_t(const Plan &pl, const BtParams &bp, cudaStream_t s) {
  auto kern = w4_batch_kernel<G, SC, ZM, MT>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       pl.smem_bytes);
  if (e != cudaSuccess) return e;
  // programmatic stream serialization: the next kernel may begin launching while this one
  // runs; this kernel touches its inputs and outputs only after griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid_x, pl.grid_z);
  cfg.blockDim = dim3(batch_warps(MT) * 32);     // the kernel's own warp count
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, bp);
}

template <int G, int SC, int ZM>
static cudaError_t launch_bt_m(const Plan &pl, const BtParams &bp, cudaStream_t s) {
  const int rows = bp.M < kBtRows ? bp.M : kBtRows;
  if (rows <= 8) return launch_bt_t<G, SC, ZM, 1>(pl, bp, s);
  if (rows <= 16) return launch_bt_t<G, SC, ZM, 2>(pl, bp, s);
  if (rows <= 24) return launch_bt_t<G, SC, ZM, 3>(pl, bp, s);
  return launch_bt_t<G, SC, ZM, 4>(pl, bp, s);
}

// float zero points (GQ_ZP_FLOAT): instantiated in their own translation unit
cudaError_t launch_batch_zf(const Plan &pl, int prec, int G, const BtParams &bp, cudaStream_t s);
int batch_zf_read_error(int clear);
int batch_zf_set_wait_limit(long long cycles);

}  // namespace gq

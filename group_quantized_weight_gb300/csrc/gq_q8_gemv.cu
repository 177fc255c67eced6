// Warp-specialized INT8 (Q8_0-style) decode kernel for M <= 4: fp32 activations, or INT8
// activations with a scale per (row, group) (W8A8); fp32 weight scales.
//
// At decode the INT8 path is bound by the bytes of its codes ("GPU Kernel 工程（09）：量化与
// 融合 kernel", section 3.2), and a short problem (the Q8_0 projection reads 28 MB) is set by
// how soon HBM is kept busy and how little is left to do once it is done.  One CTA per SM,
// two roles, as in the W4 decode kernel:
//   producer warp   lane w streams consumer w's 2 KB slots of codes (32 k of one 64-column
//                   block: two 16-k chunk rows of the packed layout) with cp.async.bulk into
//                   a ring of its own, completing on consumer w's "full" mbarrier; with
//                   GQ_STATIC_W it starts before the wait on the previous kernel.
//   consumer warps  copy the group scales of their units into a table of their own, stage
//                   the activations, then per slot: one bounded wait, four 16-byte reads of
//                   codes, the slot released at once (the codes are in registers), and the
//                   products on CUDA cores (FP32, or dp4a for INT8 activations).
// The consumers need about two instructions per code (FP32) or a quarter of one (dp4a), under
// what the SM can issue in the time HBM takes to deliver the bytes, so they keep up with the
// stream and little is left to do when the last copy lands.
//
// Arithmetic: the group-wise product of "04 · 分组量化 GEMM 内核", section 2 in its own order —
// per (column, group) the FP32 dot of the exact codes with the activations (even and odd k in
// two sums, one fma.rn.f32x2 per two products), then the group's scale times that dot added to
// the column's running sum.  An INT8 code c becomes the exact float c by placing (c xor 0x80)
// in the low byte of 2^23 and subtracting 2^23 + 128.  With INT8 activations the group's dot
// is the exact INT32 sum of dp4a products, converted exactly (|dot| <= 128 * 128 * 127 < 2^24)
// and multiplied by the activation scale times the weight scale (the same FMA as the W8A8
// block kernel).
//
// Work partition (the striped partitioning of "量化与融合 kernel", section 3.3 item 4): with N a
// multiple of 64 the packed codes are the units (64-column block b, group g) one after another,
// unit u = b (K / G) + g at byte u · 64 G.  CTA c owns a contiguous range of units (whole
// blocks when there are enough of them, otherwise an equal share) and its sixteen consumer
// warps split that range into contiguous sub-ranges, so every partial sum is a sum of whole
// scaled groups.  A block split between warps is summed in warp order, one split between CTAs
// in CTA order by whichever CTA finishes its part last (an arrival counter), so the result is
// bitwise reproducible.
#include "gq_device.cuh"

namespace gq {

namespace q8g {
constexpr int kConsumers = 16;                  // consumer warps per CTA
constexpr int kStages = 3;                      // ring stages (one slot per consumer each)
constexpr int kSlotBytes = 2048;                // 32 k x 64 columns of codes
constexpr int kSlotK = 32;
constexpr int kCols = 64;                       // columns per block (two per lane)
constexpr int kMaxRows = 4;                     // fp32 activations
constexpr int kMaxRowsA8 = 4;                   // INT8 activations (the same bound)
constexpr int kUnitTable = kCols * 4;           // table bytes per unit: 64 fp32 scales
constexpr int kBatch = 4;                       // partial sums loaded per batch in reductions
}  // namespace q8g

// Sticky device-side status (GQ_ERR_TIMEOUT after a bounded wait gave up) and the wait limit
// in SM clock cycles (about two seconds by default; gq_set_wait_limit changes it).
static __device__ int g_q8g_error;
static __device__ long long g_q8g_wait_limit = 4000000000ll;

struct Q8GemvParams {
  const uint8_t *Wp;          // packed codes, 64-column blocks of K/16 chunk rows
  const float *A;             // [M][K] fp32 activations, or
  const int8_t *Aq;           // [M][K] INT8 activations and
  const float *As;            // [M][K/G] their scales
  const float *S;             // [K/G][N]
  void *out;                  // [M][N] (gate+up: [M][N/2])
  float *part;                // [gridDim.x][2][4][64] per-CTA partial sums (shared blocks)
  unsigned *counters;         // per-block arrival counters (shared blocks)
  int M, K, N, G;
  int split_count, split_mult;   // CTA c owns units zsplit(split_count, grid, c) * split_mult
  int table_bytes;               // bytes of one consumer warp's scale table
  int out_f32;
  int static_w;                  // weights may be read before the preceding kernel ends
  int gate_up;                   // fused gate+up: block b = gate 32b.. and up N/2 + 32b..
};

namespace q8g {

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

// Wait for the phase of parity `parity`; bounded, then GQ_ERR_TIMEOUT and false.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity) {
  if (try_phase(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (try_phase(bar, parity)) return true;
    if ((it & 63u) == 0u && clock64() - t0 > g_q8g_wait_limit) {
      atomicExch(&g_q8g_error, GQ_ERR_TIMEOUT);
      return false;
    }
  }
}

// (z0, z1) += (x0, x1) * (y0, y1), one instruction
__device__ __forceinline__ void fma2(float &z0, float &z1, float x0, float x1, float y0,
                                     float y1) {
  asm("{\n\t.reg .b64 a, b, c;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 c, a, b, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "+f"(z0), "+f"(z1)
      : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

// codes b0 and b1 of w (already xor 0x80 per byte) as the exact floats c0 and c1
__device__ __forceinline__ void codes2(uint32_t w, int b0, float &c0, float &c1) {
  c0 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + b0));
  c1 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + b0 + 1));
  fma2(c0, c1, 1.f, 1.f, -8388736.f, -8388736.f);   // - (2^23 + 128), exact
}

// bytes of the activation area: MR rows of K fp32 values, or MR rows of K INT8 codes and then
// MR rows of K / G fp32 scales
__host__ __device__ inline size_t act_bytes(int MR, int K, int G, bool a8) {
  const size_t b = a8 ? (((size_t)MR * K + 15) & ~(size_t)15) + (size_t)MR * (K / G) * 4
                      : (size_t)MR * K * 4;
  return (b + 127) & ~(size_t)127;
}

__device__ __forceinline__ int dp4a(int a, int b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

}  // namespace q8g

// Shared memory (dynamic, base rounded up to 128 bytes): [act][ring][tables][pieces]
//   act     MR rows of K fp32 activations, or of K INT8 codes followed by MR rows of K / G
//           activation scales (rows past M zero)
//   ring    kStages x kConsumers slots of 2 KB of codes
//   tables  per consumer warp, for each of its units in order: the 64 columns' fp32 scales
//           (lane l's columns l and 32 + l at words l and 32 + l)
//   pieces  kConsumers x 2 x MR x 64 floats: a warp's partial sums of its first and last block
template <int MR, int SPU, bool A8>
__global__ void __launch_bounds__((q8g::kConsumers + 1) * 32, 1)
    q8_gemv_kernel(const Q8GemvParams p) {
  using namespace q8g;
  constexpr int NC = kConsumers, S = kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  __shared__ __align__(8) uint64_t full_bar[S][NC], empty_bar[S][NC];
  __shared__ int s_last[NC];
  asm volatile("griddepcontrol.launch_dependents;");

  const int M = p.M, K = p.K, N = p.N, G = p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int GPB = K / G;                            // units (groups) per block
  const size_t unit_bytes = (size_t)kCols * G;      // SPU slots
  int cb, ce;                                       // this CTA's units
  zsplit_dev(p.split_count, gridDim.x, blockIdx.x, cb, ce);
  cb *= p.split_mult;
  ce *= p.split_mult;
  float *act = reinterpret_cast<float *>(smem);
  const int8_t *acode = reinterpret_cast<const int8_t *>(smem);         // A8: [MR][K]
  float *ascale = reinterpret_cast<float *>(smem + (((size_t)MR * K + 15) & ~(size_t)15));
  uint8_t *ring = smem + act_bytes(MR, K, G, A8);
  uint8_t *tables = ring + (size_t)S * NC * kSlotBytes;
  float *pieces = reinterpret_cast<float *>(tables + (size_t)NC * p.table_bytes);

  if (threadIdx.x < S * NC) {                       // one (stage, consumer) pair per thread
    const int s = threadIdx.x / NC, w = threadIdx.x - s * NC;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&full_bar[s][w])) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&empty_bar[s][w])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ================================================================ producer warp
  if (warp == NC) {
    if (!p.static_w) asm volatile("griddepcontrol.wait;" ::: "memory");
    // lane w < NC streams consumer w's units [wb, we) — one contiguous byte range — as 2 KB
    // slots through ring slot (stage, w), refilling a stage once that consumer released it
    if (lane < NC) {
      int wb, we;
      zsplit_dev(ce - cb, NC, lane, wb, we);
      wb += cb;
      we += cb;
      const int mine = (we - wb) * SPU;
      const uint8_t *src = p.Wp + (size_t)wb * unit_bytes;
      int issued = 0;
      for (int j = 0; j < mine; ++j) {
        const int st = j % S;
        if (j >= S && !wait_phase(saddr(&empty_bar[st][lane]), (uint32_t)((j / S + 1) & 1))) break;
        const uint32_t fb = saddr(&full_bar[st][lane]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                     "n"(kSlotBytes)
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                saddr(ring + ((size_t)st * NC + lane) * kSlotBytes)),
            "l"(src + (size_t)j * kSlotBytes), "n"(kSlotBytes), "r"(fb)
            : "memory");
        issued = j + 1;
      }
      // every copy issued has landed before the producer leaves (the CTA's shared memory must
      // not be written after all of its warps are gone): fill f completed phase f / S of
      // full_bar[f % S][w]
      for (int f = max(0, issued - S); f < issued; ++f)
        if (!wait_phase(saddr(&full_bar[f % S][lane]), (uint32_t)((f / S) & 1))) break;
    }
    return;
  }

  // ================================================================ consumer warps
  int wb, we;                                       // this warp's units
  zsplit_dev(ce - cb, NC, warp, wb, we);
  wb += cb;
  we += cb;
  const int nu = we - wb;

  // ---- this warp's scale table (static weights: before the preceding kernel ends)
  float *tbl = reinterpret_cast<float *>(tables + (size_t)warp * p.table_bytes);
  auto load_table = [&]() {
    for (int e = lane; e < nu * 16; e += 32) {
      const int iu = e >> 4, pc = e & 15;
      const int u = wb + iu, b = u / GPB, g = u - b * GPB;
      size_t col = (size_t)b * kCols + pc * 4;
      if (p.gate_up)
        col = pc < 8 ? (size_t)32 * b + pc * 4 : (size_t)N / 2 + 32 * b + (pc - 8) * 4;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr(tbl + iu * kCols + pc * 4)),
                   "l"(p.S + (size_t)g * N + col)
                   : "memory");
    }
  };
  if (p.static_w) load_table();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!p.static_w) load_table();
  // ---- activations, zero rows past M: [MR][K] fp32, or [MR][K] INT8 codes (16 bytes per
  // copy) and [MR][K / G] scales (4 bytes per copy)
  const int nth = NC * 32;
  if (A8) {
    const int K16 = K >> 4;
    for (int idx = threadIdx.x; idx < MR * K16; idx += nth) {
      const int m = idx / K16, k16 = idx - m * K16;
      uint8_t *dst = smem + (size_t)m * K + 16 * k16;
      if (m < M)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr(dst)),
                     "l"(p.Aq + (size_t)m * K + 16 * k16)
                     : "memory");
      else
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int idx = threadIdx.x; idx < MR * GPB; idx += nth) {
      const int m = idx / GPB, g = idx - m * GPB;
      if (m < M)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(saddr(ascale + idx)),
                     "l"(p.As + (size_t)m * GPB + g)
                     : "memory");
      else
        ascale[idx] = 0.f;
    }
  } else {
    const int K4 = K >> 2;
    for (int idx = threadIdx.x; idx < MR * K4; idx += nth) {
      const int m = idx / K4, k4 = idx - m * K4;
      if (m < M)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr(act + (size_t)m * K + 4 * k4)),
                     "l"(p.A + (size_t)m * K + 4 * k4)
                     : "memory");
      else
        *reinterpret_cast<float4 *>(act + (size_t)m * K + 4 * k4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
  asm volatile("bar.sync 1, %0;" ::"r"(nth) : "memory");

  const int t_first = wb / GPB;
  int bcur = t_first, gcur = wb - t_first * GPB;
  int j0 = gcur;                                   // first unit of this warp's share of bcur
  float acc[MR][2];
#pragma unroll
  for (int m = 0; m < MR; ++m) acc[m][0] = acc[m][1] = 0.f;

  // end of the warp's share of block bcur (units j0 .. j1 - 1): store a whole block or keep
  // the share for the reduction
  auto flush = [&](int j1) {
    if (j0 == 0 && j1 == GPB) {
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        if (m < M) {
          if (p.gate_up) {
            store_out_rt(p.out, (size_t)m * (N / 2) + 32 * bcur + lane,
                         silu_mul(acc[m][0], acc[m][1]), p.out_f32 != 0);
          } else {
            store_out_rt(p.out, (size_t)m * N + bcur * kCols + lane, acc[m][0], p.out_f32 != 0);
            store_out_rt(p.out, (size_t)m * N + bcur * kCols + 32 + lane, acc[m][1],
                         p.out_f32 != 0);
          }
        }
      }
    } else {
      float *pc = pieces + (size_t)(warp * 2 + (bcur == t_first ? 0 : 1)) * MR * kCols;
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        pc[m * kCols + lane] = acc[m][0];
        pc[m * kCols + 32 + lane] = acc[m][1];
      }
    }
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m][0] = acc[m][1] = 0.f;
  };

  const uint8_t *ringw = ring + (size_t)warp * kSlotBytes + lane * 16;
  bool ok = true;
  int i = 0;                                       // slot number within this warp's stream
  for (int iu = 0; iu < nu && ok; ++iu) {
    // the group's dot per row and column: even and odd k (fp32 activations), or INT32 (A8)
    float de[MR][2], dd[MR][2];
    int di[MR][2];
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      de[m][0] = de[m][1] = dd[m][0] = dd[m][1] = 0.f;
      di[m][0] = di[m][1] = 0;
    }
    const float *ag = act + gcur * G;
    const int8_t *aq = acode + gcur * G;
#pragma unroll
    for (int ps = 0; ps < SPU; ++ps, ++i) {
      const int st = i % S;
      if (!wait_phase(saddr(&full_bar[st][warp]), (uint32_t)((i / S) & 1))) {
        ok = false;
        break;
      }
      // chunk row r of the slot: column l's 16 codes at 1024 r + 16 l, column 32 + l's at
      // 1024 r + 512 + 16 l
      const uint8_t *slot = ringw + (size_t)st * (NC * kSlotBytes);
      const uint4 va0 = *reinterpret_cast<const uint4 *>(slot);
      const uint4 vc0 = *reinterpret_cast<const uint4 *>(slot + 512);
      const uint4 va1 = *reinterpret_cast<const uint4 *>(slot + 1024);
      const uint4 vc1 = *reinterpret_cast<const uint4 *>(slot + 1536);
      // the codes are in registers: release the slot to the producer lane now
      __syncwarp();
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.eq.u32 p, %1, 0;\n\t"
          "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(saddr(&empty_bar[st][warp])),
          "r"(lane)
          : "memory");
      const uint32_t wa[8] = {va0.x, va0.y, va0.z, va0.w, va1.x, va1.y, va1.z, va1.w};
      const uint32_t wc[8] = {vc0.x, vc0.y, vc0.z, vc0.w, vc1.x, vc1.y, vc1.z, vc1.w};
      if (A8) {
        // word q of a column: k = 4q .. 4q + 3 of the slot; the row's codes of k = 16h ..
        // 16h + 15 in one 16-byte broadcast
#pragma unroll
        for (int m = 0; m < MR; ++m) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 av = *reinterpret_cast<const uint4 *>(aq + (size_t)m * K + ps * kSlotK + 16 * h);
            const int aw[4] = {(int)av.x, (int)av.y, (int)av.z, (int)av.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              di[m][0] = dp4a((int)wa[4 * h + e], aw[e], di[m][0]);
              di[m][1] = dp4a((int)wc[4 * h + e], aw[e], di[m][1]);
            }
          }
        }
        continue;
      }
      const float *ak = ag + ps * kSlotK;
#pragma unroll
      for (int q = 0; q < 8; ++q) {                // k = 4q .. 4q + 3 of the slot
        const uint32_t xa = wa[q] ^ 0x80808080u, xc = wc[q] ^ 0x80808080u;
        float a0, a1, a2, a3, c0, c1, c2, c3;
        codes2(xa, 0, a0, a1);
        codes2(xa, 2, a2, a3);
        codes2(xc, 0, c0, c1);
        codes2(xc, 2, c2, c3);
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          const float4 x = *reinterpret_cast<const float4 *>(ak + (size_t)m * K + 4 * q);
          fma2(de[m][0], dd[m][0], a0, a1, x.x, x.y);
          fma2(de[m][0], dd[m][0], a2, a3, x.z, x.w);
          fma2(de[m][1], dd[m][1], c0, c1, x.x, x.y);
          fma2(de[m][1], dd[m][1], c2, c3, x.z, x.w);
        }
      }
    }
    if (!ok) break;
    // a whole group: its scale times its dot
    const float sa = tbl[iu * kCols + lane], sc = tbl[iu * kCols + 32 + lane];
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      if (A8) {
        const float as = ascale[m * GPB + gcur];
        acc[m][0] = fmaf(as * sa, (float)di[m][0], acc[m][0]);
        acc[m][1] = fmaf(as * sc, (float)di[m][1], acc[m][1]);
      } else {
        acc[m][0] = fmaf(sa, de[m][0] + dd[m][0], acc[m][0]);
        acc[m][1] = fmaf(sc, de[m][1] + dd[m][1], acc[m][1]);
      }
    }
    if (++gcur == GPB) {
      flush(GPB);
      ++bcur;
      gcur = 0;
      j0 = 0;
    }
  }
  if (nu > 0 && gcur != 0) flush(gcur);

  // Final sums of block tt, row m, column pair (c, 32 + c), lane c: stored, or with gate+up
  // silu(gate) * up.
  auto store_block = [&](int tt, int m, float sa, float sc) {
    if (m >= M) return;
    if (p.gate_up) {
      store_out_rt(p.out, (size_t)m * (N / 2) + 32 * tt + lane, silu_mul(sa, sc), p.out_f32 != 0);
    } else {
      store_out_rt(p.out, (size_t)m * N + tt * kCols + lane, sa, p.out_f32 != 0);
      store_out_rt(p.out, (size_t)m * N + tt * kCols + 32 + lane, sc, p.out_f32 != 0);
    }
  };

  // ---- reduction of the blocks shared between warps (shared memory) and CTAs (global)
  asm volatile("bar.sync 1, %0;" ::"r"(nth) : "memory");
  for (int pass = 0; pass < 2 && nu > 0; ++pass) {
    const int tt = pass == 0 ? t_first : (we - 1) / GPB;
    if (pass == 1 && tt == t_first) break;
    const int tb = tt * GPB, te = tb + GPB;         // the block's units
    if (max(tb, wb) == tb && min(te, we) == te) continue;          // stored directly
    if (pass == 0 && wb > cb && wb % GPB != 0) continue;          // a lower warp reduces it
    const bool cta_whole = tb >= cb && te <= ce;
    const int region = tb < cb ? 0 : 1;
    // the warps of this CTA holding units of the block: warp .. w_hi
    int w_hi = warp;
    for (int w2 = warp + 1; w2 < NC; ++w2) {
      int b2, e2;
      zsplit_dev(ce - cb, NC, w2, b2, e2);
      if (e2 <= b2 || b2 + cb >= te) break;
      w_hi = w2;
    }
    // their shares added in warp order; the loads of kBatch warps are issued before their adds
    float sa[MR], sc[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) sa[m] = sc[m] = 0.f;
    for (int w0 = warp; w0 <= w_hi; w0 += kBatch) {
      float va[kBatch][MR], vc[kBatch][MR];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int w2 = min(w0 + j, w_hi);
        int b2, e2;
        zsplit_dev(ce - cb, NC, w2, b2, e2);
        const float *pc = pieces + (size_t)(w2 * 2 + ((b2 + cb) / GPB == tt ? 0 : 1)) * MR * kCols;
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          va[j][m] = pc[m * kCols + lane];
          vc[j][m] = pc[m * kCols + 32 + lane];
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (w0 + j > w_hi) break;
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          sa[m] += va[j][m];
          sc[m] += vc[j][m];
        }
      }
    }
    for (int m = 0; m < M; ++m) {
      if (cta_whole) {
        store_block(tt, m, sa[m], sc[m]);
      } else {
        float *dst = p.part + ((size_t)blockIdx.x * 2 + region) * (kMaxRows * kCols) + m * kCols;
        __stcg(dst + lane, sa[m]);
        __stcg(dst + 32 + lane, sc[m]);
      }
    }
    if (cta_whole) continue;
    // last arriver over the CTAs holding units of the block (no CTA waits for another)
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      const unsigned mine = (unsigned)(min(te, ce) - max(tb, cb));
      const unsigned prev = atomicAdd(p.counters + tt, mine);
      const bool last = prev + mine == (unsigned)GPB;
      if (last) p.counters[tt] = 0u;
      s_last[warp] = last ? 1 : 0;
    }
    __syncwarp();
    if (!s_last[warp]) continue;
    __threadfence();
    // the CTAs holding units of the block: c_lo .. c_hi (a CTA's range may be empty)
    int c_lo = blockIdx.x, c_hi = blockIdx.x;
    for (;;) {
      if (c_lo == 0) break;
      int b2, e2;
      zsplit_dev(p.split_count, gridDim.x, c_lo - 1, b2, e2);
      if (e2 * p.split_mult <= tb) break;
      --c_lo;
    }
    for (;;) {
      if (c_hi + 1 >= (int)gridDim.x) break;
      int b2, e2;
      zsplit_dev(p.split_count, gridDim.x, c_hi + 1, b2, e2);
      if (b2 * p.split_mult >= te) break;
      ++c_hi;
    }
    // their partial sums added in CTA order; the L2 reads of kBatch CTAs are issued before
    // their adds (one round trip per batch, not per CTA)
#pragma unroll
    for (int m = 0; m < MR; ++m) sa[m] = sc[m] = 0.f;
    for (int c0 = c_lo; c0 <= c_hi; c0 += kBatch) {
      float va[kBatch][MR], vc[kBatch][MR];
      bool use[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int c2 = min(c0 + j, c_hi);
        int b2, e2;
        zsplit_dev(p.split_count, gridDim.x, c2, b2, e2);
        b2 *= p.split_mult;
        e2 *= p.split_mult;
        use[j] = c0 + j <= c_hi && e2 > b2;
        const int r2 = tb < b2 ? 0 : 1;           // the region that CTA wrote
        const float *src = p.part + ((size_t)c2 * 2 + r2) * (kMaxRows * kCols);
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          va[j][m] = use[j] ? __ldcg(src + m * kCols + lane) : 0.f;
          vc[j][m] = use[j] ? __ldcg(src + m * kCols + 32 + lane) : 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (!use[j]) continue;
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          sa[m] += va[j][m];
          sc[m] += vc[j][m];
        }
      }
    }
    for (int m = 0; m < M; ++m) store_block(tt, m, sa[m], sc[m]);
  }
}

// ------------------------------------------------------------------ host side

namespace {
bool is_a8(int prec) { return (prec & GQ_ACT_I8) != 0; }
// template rows: 1, 2 or 4
int q8_gemv_rows(int M, int) { return M <= 1 ? 1 : M <= 2 ? 2 : 4; }
}  // namespace

bool q8_gemv_supported(int M, int K, int N, int G, int prec) {
  const bool a8 = is_a8(prec);
  const bool acts = a8 ? !(prec & (GQ_ACT_F32 | GQ_GATE_UP)) && M <= q8g::kMaxRowsA8
                       : (prec & GQ_ACT_F32) && M <= q8g::kMaxRows;
  return !(prec & GQ_W4) && acts && (prec & GQ_SC_F32) && !(prec & (GQ_ZP | GQ_ZP_FLOAT)) &&
         M >= 1 && N > 0 && N % q8g::kCols == 0 && G % q8g::kSlotK == 0 && G <= 128 &&
         K % G == 0;
}

int q8_gemv_table_bytes(int max_cta_units) {
  const int per_warp = (max_cta_units + q8g::kConsumers - 1) / q8g::kConsumers;
  return per_warp * q8g::kUnitTable;
}

size_t q8_gemv_smem_bytes(int M, int K, int G, int prec, int max_cta_units) {
  const int mr = q8_gemv_rows(M, prec);
  const size_t act = q8g::act_bytes(mr, K, G, is_a8(prec));
  const size_t ring = (size_t)q8g::kStages * q8g::kConsumers * q8g::kSlotBytes;
  const size_t tables = (size_t)q8g::kConsumers * q8_gemv_table_bytes(max_cta_units);
  const size_t pieces = (size_t)q8g::kConsumers * 2 * mr * q8g::kCols * 4;
  return 128 + act + ring + tables + pieces;         // 128: alignment of the dynamic base
}

int q8_gemv_threads() { return (q8g::kConsumers + 1) * 32; }

// per-CTA partial sums of the blocks shared between CTAs
size_t q8_gemv_part_bytes(int grid) {
  return (size_t)grid * 2 * q8g::kMaxRows * q8g::kCols * sizeof(float);
}

template <int MR, int SPU, bool A8>
static cudaError_t launch_q8g_t(const Plan &pl, const Q8GemvParams &qp, cudaStream_t s) {
  auto kern = q8_gemv_kernel<MR, SPU, A8>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), pl.smem_bytes);
  if (e != cudaSuccess) return e;
  // programmatic stream serialization: this kernel reads activations and writes outputs only
  // after griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid_x);
  cfg.blockDim = dim3(q8_gemv_threads());
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, qp);
}

template <int MR, bool A8>
static cudaError_t launch_q8g_g(const Plan &pl, const Q8GemvParams &qp, cudaStream_t s) {
  switch (qp.G) {
    case 32: return launch_q8g_t<MR, 1, A8>(pl, qp, s);
    case 64: return launch_q8g_t<MR, 2, A8>(pl, qp, s);
    case 128: return launch_q8g_t<MR, 4, A8>(pl, qp, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_q8_gemv(const Plan &pl, int M, int K, int N, int G, int prec, const void *A,
                           const float *a_scales, const void *Wq, const void *scales,
                           void *out, float *part, unsigned *counters, cudaStream_t s) {
  if (!q8_gemv_supported(M, K, N, G, prec)) return cudaErrorInvalidValue;
  const bool a8 = is_a8(prec);
  if (a8 && !a_scales) return cudaErrorInvalidValue;
  Q8GemvParams qp;
  qp.Wp = reinterpret_cast<const uint8_t *>(Wq);
  qp.A = a8 ? nullptr : reinterpret_cast<const float *>(A);
  qp.Aq = a8 ? reinterpret_cast<const int8_t *>(A) : nullptr;
  qp.As = a8 ? a_scales : nullptr;
  qp.S = reinterpret_cast<const float *>(scales);
  qp.out = out;
  qp.part = part;
  qp.counters = counters;
  qp.M = M;
  qp.K = K;
  qp.N = N;
  qp.G = G;
  qp.split_count = pl.split_count;
  qp.split_mult = pl.split_mult;
  qp.table_bytes = pl.table_bytes;
  qp.out_f32 = (prec & GQ_OUT_F32) ? 1 : 0;
  qp.static_w = (prec & GQ_STATIC_W) ? 1 : 0;
  qp.gate_up = (prec & GQ_GATE_UP) ? 1 : 0;
  switch (q8_gemv_rows(M, prec)) {
    case 1: return a8 ? launch_q8g_g<1, true>(pl, qp, s) : launch_q8g_g<1, false>(pl, qp, s);
    case 2: return a8 ? launch_q8g_g<2, true>(pl, qp, s) : launch_q8g_g<2, false>(pl, qp, s);
    default: return a8 ? launch_q8g_g<4, true>(pl, qp, s) : launch_q8g_g<4, false>(pl, qp, s);
  }
}

int q8_gemv_set_wait_limit(long long cycles) {
  return cudaMemcpyToSymbol(g_q8g_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? 0 : -1;
}

int q8_gemv_read_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_q8g_error, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(g_q8g_error, &z, sizeof(int));
  }
  return v;
}

}  // namespace gq

// Striped small-M decode kernel (M <= 8) of the group-quantized weight-only GEMM.
#include <type_traits>
#include <utility>

#include "gq_device.cuh"

namespace gq {

// ------------------------------------------------------------------ W4, striped variant

// Persistent decode kernel for M <= 8.  The flattened space of (16-column tile, K unit)
// pairs is cut into W contiguous, equal stripes, one per warp (the striped partitioning of
// "GPU Kernel 工程（09）：量化与融合 kernel", section 3.3 item 4: every SM gets the same amount
// of work for any shape, at the price of a few cross-warp reductions).  The packed layout
// stores each tile's chunks contiguously and the tiles one after another, so a stripe is
// one contiguous range of memory that the warp streams front to back.  A K unit is
// max(G, 64) values of k, a whole number of groups, so every partial sum is a sum of whole
// scaled groups.  A tile covered by one warp is stored directly; a tile split between
// warps w_a < ... < w_b is summed by the warp that completes it, adding the partials in
// warp order w_a, ..., w_b (fixed order: bitwise reproducible).
//
// Streaming: each lane keeps kStages chunks (16 bytes each) of its stripe in flight in a
// register ring, loaded kStages chunks ahead of use; the scales and zero-point words of a
// unit are loaded together with the unit's weights.
//
// Decode: the FP16 form of the magic-number trick of section 2.4 of the same page, which
// needs one shift per eight codes: (w & 0x000F000F) | 0x64006400 is fp16(1024 + q) for the
// codes in bits 0-3 and 16-19, one fp16x2 subtraction of fp16(1024 + z) leaves q - z;
// (w & 0x00F000F0) | 0x64006400 is fp16(1024 + 16q) for bits 4-7 and 20-23, and one fp16x2
// FMA with 1/16 and -(64 + z) leaves q - z; w >> 8 exposes the other four codes.  Every
// value is an exact small integer.
//
// The MMA is FP16 x FP16 -> FP32 with the 16 MMA rows on output columns n, so the bf16
// activations are carried into fp16 exactly by exponent bands: for activation row m with
// largest exponent field Emax, band b (b = 0, 1) holds the elements whose exponent field
// lies in (Emax - 32(b+1), Emax - 32b], scaled by 2^(142 - Emax + 32b) so that they land in
// [2^-16, 2^16) where fp16 represents every bf16 significand exactly.  Row m's two bands
// are MMA columns 2m and 2m + 1; the column sums are scaled back by the inverse powers of
// two and added band 0 first.  Every activation larger than 2^-64 times its row's largest
// one is represented exactly; smaller ones are treated as zero.
//
// Each group's accumulator is scaled into the tile sums one group later (accumulators
// alternate by group parity), so the FP32 scaling never waits on the MMA chain.
//
// The kernel is launched with programmatic stream serialization: it lets the next kernel
// in the stream start launching at once, and it reads none of its inputs and writes none
// of its outputs before griddepcontrol.wait (the end of the previous kernel).

constexpr int kStages = 8;    // chunks in flight per lane (register ring)

__device__ __forceinline__ int warp_of_unit(int u, int U, int W) {
  const int base = U / W, rem = U % W;
  const int big = rem * (base + 1);
  return u < big ? u / (base + 1) : rem + (u - big) / base;
}

__device__ __forceinline__ void mma_16816_f16(float d[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// (a & b) | c in one LOP3
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Decode constants, passed as a kernel parameter: the instructions read them from the
// parameter bank instead of materializing immediates around every use.
struct DecodeConsts {
  uint32_t lo_mask;     // 0x000F000F: codes in bits 0-3 and 16-19
  uint32_t hi_mask;     // 0x00F000F0: codes in bits 4-7 and 20-23
  uint32_t magic;       // 0x64006400: fp16 1024 in both halves
  uint32_t sixteenth;   // 0x2C002C00: fp16 1/16 in both halves
  uint32_t lo_sym;      // 0x64086408: fp16 (1024 + 8), symmetric zero point
  uint32_t hi_sym;      // 0xD480D480: fp16 -(64 + 8)
};

// Fix-up of a tile that a stripe covers only in part.  `val` holds the lane's combined
// value for rows m = lane_row(...) (set by the caller), columns n0 and n0 + 8.
__device__ __forceinline__ void stripe_fixup(float v0, float v1, int mrow, bool owner,
                                             float *part, unsigned *counters, void *out,
                                             int M, int N, int t, int slot, int gw,
                                             int held_units, int Cu, int U, int W,
                                             bool out_f32) {
  const int lane = threadIdx.x & 31, r0 = lane >> 2;
  float *pp = part + ((size_t)gw * 2 + slot) * (kTileN * 8);
  if (owner && mrow < M) {
    pp[mrow * kTileN + r0] = v0;
    pp[mrow * kTileN + r0 + 8] = v1;
  }
  // __syncwarp orders the lanes' partial stores before lane 0's release; the acq_rel
  // read-modify-write publishes them and, in the last arriver, makes every other
  // contributor's partials visible to the loads below
  __syncwarp();
  unsigned last = 0;
  if (lane == 0) {
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;"
                 : "=r"(prev)
                 : "l"(counters + t), "r"((unsigned)held_units)
                 : "memory");
    last = (prev + (unsigned)held_units == (unsigned)Cu) ? 1u : 0u;
    if (last) counters[t] = 0u;     // every contributor has arrived: leave it at zero
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  const int wa = warp_of_unit(t * Cu, U, W), wb = warp_of_unit(t * Cu + Cu - 1, U, W);
  for (int idx = lane; idx < M * kTileN; idx += 32) {
    const int m = idx / kTileN, nl = idx - m * kTileN;
    float s = 0.f;
    for (int w2 = wa; w2 <= wb; ++w2) {
      int b2, e2;
      zsplit_dev(U, W, w2, b2, e2);
      const int sl = (b2 / Cu == t) ? 0 : 1;
      s += __ldcg(part + ((size_t)w2 * 2 + sl) * (kTileN * 8) + m * kTileN + nl);
    }
    const int n = t * kTileN + nl;
    if (n < N) store_out_rt(out, (size_t)m * N + n, s, out_f32);
  }
}

// MT: n8 MMA blocks (1 for M <= 4, 2 for M <= 8); UG: a K unit is UG * max(G, 64) values
// of k (UG = 2 halves the per-unit work when K allows it).
template <int G, int SC, bool ZP, int MT, int UG>
__global__ void __launch_bounds__(kStrWarps * 32, 1)
w4_stripe_kernel(const uint4 *__restrict__ Wp, const uint16_t *__restrict__ A,
                 const void *__restrict__ scales, const uint32_t *__restrict__ zeros,
                 void *__restrict__ out, float *__restrict__ part,
                 unsigned *__restrict__ counters, int M, int K, int N, int W, int out_f32,
                 const DecodeConsts dk) {
  constexpr int UK = (G > kChunkK ? G : kChunkK) * UG;   // k per unit
  constexpr int UCH = UK / kChunkK;               // chunks per unit
  constexpr int GPU = UK / G;                     // groups per unit
  constexpr int SPG = G / 16;                     // 16-k MMA steps per group
  constexpr int PF = kStages / UCH;               // units in flight (kStages chunks)
  constexpr int ES = SC == kScF32 ? 4 : 2;        // bytes per scale
  static_assert(kStages % UCH == 0, "the register ring holds whole units");
  typedef typename std::conditional<SC == kScF32, uint32_t, unsigned short>::type sc_t;

  extern __shared__ __align__(16) uint32_t smem[];
  __shared__ int s_emax[8], s_emin[8];
  asm volatile("griddepcontrol.launch_dependents;");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kStrWarps + warp;
  const int C = K / kChunkK;
  const int Cu = K / UK;
  const int T = (N + kTileN - 1) / kTileN;
  const int U = T * Cu;
  const int NW = N >> 3;
  int u0 = 0, u1 = 0;
  if (gw < W) zsplit_dev(U, W, gw, u0, u1);
  const int nu = u1 - u0;                          // units in this warp's stripe
  const int r0 = lane >> 2, q = lane & 3;
  if (threadIdx.x < 8) {
    s_emax[threadIdx.x] = 0;
    s_emin[threadIdx.x] = 255;
  }
  // shared memory: [band rows][raw A]
  const int RS = act_row_words(C);
  uint32_t *bands = smem;
  uint32_t *araw = bands + (1 + 2 * M) * RS;     // zero row + two band rows per row

  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- the load side: weights of PF units ahead in registers, with their scales
  const uint4 *wsrc = Wp + (size_t)u0 * UCH * 32 + lane;
  const size_t srow = (size_t)N;                   // elements per scale row
  int ht = u0 / Cu, hu = u0 - ht * Cu;             // tile and unit of the load head
  const sc_t *hsa = reinterpret_cast<const sc_t *>(scales) + min(ht * kTileN + r0, N - 1);
  const sc_t *hsb = reinterpret_cast<const sc_t *>(scales) + min(ht * kTileN + r0 + 8, N - 1);
  const uint32_t *hza = zeros + min(2 * ht, NW - 1), *hzb = zeros + min(2 * ht + 1, NW - 1);
  size_t hg = (size_t)hu * GPU;                    // group index of the head unit
  uint4 buf[PF][UCH];
  uint32_t sr[PF][GPU][2], zr[PF][GPU][2];
  auto load_unit = [&](auto slot, int k) {         // unit k of the stripe into ring slot P
    constexpr int P = decltype(slot)::value;
#pragma unroll
    for (int ch = 0; ch < UCH; ++ch)
      buf[P][ch] = ld_stream(wsrc + (size_t)(k * UCH + ch) * 32);
#pragma unroll
    for (int gi = 0; gi < GPU; ++gi) {
      sr[P][gi][0] = (uint32_t)__ldg(hsa + (hg + gi) * srow);
      sr[P][gi][1] = (uint32_t)__ldg(hsb + (hg + gi) * srow);
      if (ZP) {
        zr[P][gi][0] = __ldg(hza + (hg + gi) * NW);
        zr[P][gi][1] = __ldg(hzb + (hg + gi) * NW);
      }
    }
    hg += GPU;
    if (++hu == Cu) {
      hu = 0;
      hg = 0;
      ++ht;
      hsa = reinterpret_cast<const sc_t *>(scales) + min(ht * kTileN + r0, N - 1);
      hsb = reinterpret_cast<const sc_t *>(scales) + min(ht * kTileN + r0 + 8, N - 1);
      hza = zeros + min(2 * ht, NW - 1);
      hzb = zeros + min(2 * ht + 1, NW - 1);
    }
  };
  auto prefetch = [&](auto slot) {
    constexpr int P = decltype(slot)::value;
    if (P < nu) load_unit(slot, P);
  };
  [&]<int... P>(std::integer_sequence<int, P...>) {
    (prefetch(std::integral_constant<int, P>()), ...);
  }(std::make_integer_sequence<int, PF>());

  // ---- stage A: exponent bands as fp16, permuted for the B operands
  {
    const int n16 = (M * K) >> 3;                  // 16-byte pieces of A
    const uint32_t dst0 = (uint32_t)__cvta_generic_to_shared(araw);
    for (int i = threadIdx.x; i < n16; i += blockDim.x)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst0 + 16u * i),
                   "l"(reinterpret_cast<const uint4 *>(A) + i)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int idx = threadIdx.x; idx < RS; idx += blockDim.x) bands[idx] = 0u;   // zero row 0
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();                                 // raw A visible; s_emax / s_emin set
  const int wpr = K >> 1;                          // bf16 pairs per row
  for (int m = 0; m < M; ++m) {
    int emx = 0, emn = 255;
    for (int w = threadIdx.x; w < wpr; w += blockDim.x) {
      const uint32_t raw = araw[m * wpr + w];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t bits = (raw >> (16 * h)) & 0xFFFFu;
        if (bits & 0x7FFFu) {
          const int e = (bits >> 7) & 0xFF;
          emx = max(emx, e);
          emn = min(emn, e);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      emx = max(emx, __shfl_xor_sync(0xffffffffu, emx, o));
      emn = min(emn, __shfl_xor_sync(0xffffffffu, emn, o));
    }
    if (lane == 0) {
      atomicMax(&s_emax[m], emx);
      atomicMin(&s_emin[m], emn);
    }
  }
  __syncthreads();
  // band row 1 + 2m + b holds band b of activation row m (only if the row needs it)
  for (int v = 0; v < 2 * M; ++v) {
    const int m = v >> 1, b = v & 1;
    const int emax = s_emax[m], emin = s_emin[m];
    const int nbu = emin > emax ? 0 : min(2, ((emax - emin) >> 5) + 1);
    if (b >= nbu) continue;
    const int sb = 142 - emax + 32 * b;            // scale exponent of band b
    for (int w = threadIdx.x; w < wpr; w += blockDim.x) {
      const uint32_t raw = araw[m * wpr + w];
      uint32_t pair = 0u;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t bits = (raw >> (16 * h)) & 0xFFFFu;
        const int ex = (bits >> 7) & 0xFF;
        if ((bits & 0x7FFFu) && ((emax - ex) >> 5) == b) {
          float f;
          if (ex == 255)
            f = __uint_as_float(bits << 16);                       // inf / nan stay so
          else if (ex == 0)
            f = ldexpf(__uint_as_float(bits << 16), sb);           // bf16 subnormal
          else
            f = __uint_as_float((bits << 16) + ((uint32_t)sb << 23));  // exponent + sb
          pair |= (uint32_t)__half_as_ushort(__float2half_rn(f)) << (16 * h);
        }
      }
      const int kk = 2 * w;
      const int c = kk >> 6, r = kk & 63, j = r >> 4, hh = (r >> 3) & 1, qq = (r & 7) >> 1;
      bands[(1 + v) * RS + c * 32 + (j >> 1) * 16 + qq * 4 + (j & 1) * 2 + hh] = pair;
    }
  }
  __syncthreads();
  if (nu <= 0) return;

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

  int t = u0 / Cu, ul = u0 - t * Cu;               // tile and unit being computed
  const int t_first = t;
  int tile_u0 = ul;
  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  // one unit from ring slot P; the slot is refilled with unit k + PF first
  auto step = [&](auto slot, int k) {
    constexpr int P = decltype(slot)::value;
    uint4 cur[UCH];
    uint32_t sv[GPU][2], zw[GPU][2];
#pragma unroll
    for (int ch = 0; ch < UCH; ++ch) cur[ch] = buf[P][ch];
#pragma unroll
    for (int gi = 0; gi < GPU; ++gi) {
      sv[gi][0] = sr[P][gi][0];
      sv[gi][1] = sr[P][gi][1];
      if (ZP) { zw[gi][0] = zr[P][gi][0]; zw[gi][1] = zr[P][gi][1]; }
    }
    if (k + PF < nu) load_unit(slot, k + PF);

    uint32_t zl = ZP ? zlo_of(zw[0][0]) : dk.lo_sym, zh = ZP ? zhi_of(zw[0][1]) : dk.hi_sym;
    float d[MT][4];
    const uint32_t *bp[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) bp[mt] = brow[mt] + ul * (UCH * 32);
#pragma unroll
    for (int ch = 0; ch < UCH; ++ch) {
      uint32_t bq[MT][8];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint4 lo = *reinterpret_cast<const uint4 *>(bp[mt] + ch * 32);
        const uint4 hi = *reinterpret_cast<const uint4 *>(bp[mt] + ch * 32 + 16);
        bq[mt][0] = lo.x; bq[mt][1] = lo.y; bq[mt][2] = lo.z; bq[mt][3] = lo.w;
        bq[mt][4] = hi.x; bq[mt][5] = hi.y; bq[mt][6] = hi.z; bq[mt][7] = hi.w;
      }
      const uint32_t words[4] = {cur[ch].x, cur[ch].y, cur[ch].z, cur[ch].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int stp = ch * 4 + j;                   // compile-time
        const uint32_t w = words[j], w8 = w >> 8;
        const uint32_t a0 = hsub2_u(lop3_and_or(w, dk.lo_mask, dk.magic), zl);
        const uint32_t a1 = hfma2_u(lop3_and_or(w, dk.hi_mask, dk.magic), dk.sixteenth, zh);
        const uint32_t a2 = hsub2_u(lop3_and_or(w8, dk.lo_mask, dk.magic), zl);
        const uint32_t a3 = hfma2_u(lop3_and_or(w8, dk.hi_mask, dk.magic), dk.sixteenth, zh);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          if (stp % SPG == 0) d[mt][0] = d[mt][1] = d[mt][2] = d[mt][3] = 0.f;
          mma_16816_f16(d[mt], a0, a1, a2, a3, bq[mt][2 * j], bq[mt][2 * j + 1]);
        }
        if ((stp + 1) % SPG == 0) {                // a whole group: scale it in
          const int gi = stp / SPG;
          const float fa = scale_f(sv[gi][0]), fb = scale_f(sv[gi][1]);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            acc[mt][0] = fmaf(fa, d[mt][0], acc[mt][0]);
            acc[mt][1] = fmaf(fa, d[mt][1], acc[mt][1]);
            acc[mt][2] = fmaf(fb, d[mt][2], acc[mt][2]);
            acc[mt][3] = fmaf(fb, d[mt][3], acc[mt][3]);
          }
          if (ZP && gi + 1 < GPU) {
            zl = zlo_of(zw[gi + 1 < GPU ? gi + 1 : 0][0]);
            zh = zhi_of(zw[gi + 1 < GPU ? gi + 1 : 0][1]);
          }
        }
      }
    }

    // end of a tile, or of the stripe: combine the bands, then store or fix up
    ++ul;
    if (ul == Cu || k + 1 == nu) {
      const bool whole = (tile_u0 == 0 && ul == Cu);
      float *pp = part + ((size_t)gw * 2 + (t == t_first ? 0 : 1)) * (kTileN * 8);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        // lane (r0, q) holds columns 2q, 2q + 1 (both bands of row mt * 4 + q) of rows
        // n0 = r0 and r0 + 8
        const int mrow = mt * 4 + q;
        const int emax = mrow < M ? s_emax[mrow] : 127;
        const float v0 = ldexpf(acc[mt][0], emax - 142) + ldexpf(acc[mt][1], emax - 174);
        const float v1 = ldexpf(acc[mt][2], emax - 142) + ldexpf(acc[mt][3], emax - 174);
        if (mrow < M) {
          if (whole) {
            const int n0 = t * kTileN + r0;
            if (n0 < N) store_out_rt(out, (size_t)mrow * N + n0, v0, out_f32 != 0);
            if (n0 + 8 < N) store_out_rt(out, (size_t)mrow * N + n0 + 8, v1, out_f32 != 0);
          } else {
            pp[mrow * kTileN + r0] = v0;
            pp[mrow * kTileN + r0 + 8] = v1;
          }
        }
        acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      }
      if (!whole)
        stripe_fixup(0.f, 0.f, 0, false, part, counters, out, M, N, t, t == t_first ? 0 : 1,
                     gw, ul - tile_u0, Cu, U, W, out_f32 != 0);
      if (ul == Cu) { ul = 0; ++t; tile_u0 = 0; }
    }
  };

  for (int k0 = 0; k0 < nu; k0 += PF) {
    [&]<int... P>(std::integer_sequence<int, P...>) {
      ((k0 + P < nu ? (step(std::integral_constant<int, P>(), k0 + P), 0) : 0), ...);
    }(std::make_integer_sequence<int, PF>());
  }
}

template <int G, int SC, bool ZP, int MT, int UG>
static cudaError_t launch_stripe_t(const Plan &p, int prec, int M, int K, int N,
                                   const void *A, const void *Wq, const void *scales,
                                   const void *zeros, void *out, float *part,
                                   unsigned *counters, cudaStream_t s) {
  auto kern = w4_stripe_kernel<G, SC, ZP, MT, UG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)p.smem_bytes);
  if (e != cudaSuccess) return e;
  const int out_f32 = (prec & GQ_OUT_F32) ? 1 : 0;
  // programmatic stream serialization: the next kernel may begin launching while this one
  // runs; this kernel touches its inputs and outputs only after griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid_x);
  cfg.blockDim = dim3(p.block_threads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4 *>(Wq),
                            reinterpret_cast<const uint16_t *>(A), scales,
                            reinterpret_cast<const uint32_t *>(zeros), out, part, counters,
                            M, K, N, p.nsplit, out_f32,
                            DecodeConsts{0x000F000Fu, 0x00F000F0u, 0x64006400u, 0x2C002C00u,
                                         0x64086408u, 0xD480D480u});
}

// units of two groups when K allows it (G = 64, 128), one group otherwise
int stripe_unit_groups(int K, int G) {
  const int base = G > kChunkK ? G : kChunkK;
  return ((G == 64 || G == 128) && K % (2 * base) == 0) ? 2 : 1;
}

template <int G, int SC, bool ZP, int UG>
static cudaError_t launch_stripe_m(const Plan &p, int prec, int M, int K, int N,
                                   const void *A, const void *Wq, const void *scales,
                                   const void *zeros, void *out, float *part, unsigned *cnt,
                                   cudaStream_t s) {
  if (M <= 4) return launch_stripe_t<G, SC, ZP, 1, UG>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, cnt, s);
  return launch_stripe_t<G, SC, ZP, 2, UG>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, cnt, s);
}

template <int G, int SC, bool ZP>
static cudaError_t launch_stripe_u(const Plan &p, int prec, int M, int K, int N,
                                   const void *A, const void *Wq, const void *scales,
                                   const void *zeros, void *out, float *part, unsigned *cnt,
                                   cudaStream_t s) {
  if constexpr (G == 64 || G == 128) {
    if (stripe_unit_groups(K, G) == 2)
      return launch_stripe_m<G, SC, ZP, 2>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, cnt, s);
  }
  return launch_stripe_m<G, SC, ZP, 1>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, cnt, s);
}

template <int G, int SC>
static cudaError_t launch_stripe_z(const Plan &p, int prec, int M, int K, int N,
                                   const void *A, const void *Wq, const void *scales,
                                   const void *zeros, void *out, float *part, unsigned *cnt,
                                   cudaStream_t s) {
  if (prec & GQ_ZP)
    return launch_stripe_u<G, SC, true>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, cnt, s);
  return launch_stripe_u<G, SC, false>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, cnt, s);
}

template <int G>
static cudaError_t launch_stripe_g(const Plan &p, int prec, int M, int K, int N,
                                   const void *A, const void *Wq, const void *scales,
                                   const void *zeros, void *out, float *part, unsigned *cnt,
                                   cudaStream_t s) {
  if (prec & GQ_SC_F32)
    return launch_stripe_z<G, kScF32>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, cnt, s);
  if (prec & GQ_SC_BF16)
    return launch_stripe_z<G, kScBF16>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, cnt, s);
  return launch_stripe_z<G, kScF16>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, cnt, s);
}

size_t stripe_smem_bytes(int M, int K, int G, int prec) {
  (void)G;
  (void)prec;
  const size_t bands = (size_t)(1 + 2 * M) * (K / kChunkK * 32 + 16) * 4;
  return bands + (size_t)M * K * 2;
}

cudaError_t launch_stripe_decode(const Plan &p, int M, int K, int N, int G, int prec,
                                 const void *A, const void *Wq, const void *scales,
                                 const void *zeros, void *out, float *part,
                                 unsigned *counters, cudaStream_t s) {
  switch (G) {
    case 32: return launch_stripe_g<32>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, counters, s);
    case 64: return launch_stripe_g<64>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, counters, s);
    case 128: return launch_stripe_g<128>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, counters, s);
    case 256: return launch_stripe_g<256>(p, prec, M, K, N, A, Wq, scales, zeros, out, part, counters, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gq

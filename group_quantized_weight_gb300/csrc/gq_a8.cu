// INT8-activation variant: per-group dynamic quantization of the activations and the exact
// integer group dots of "04 · 分组量化 GEMM 内核", section 2:
//
//     out[m][n] = Σ_g a_scale[m][g] · b_scale[g][n] · ( Σ_{k ∈ g} Aq[m][k] · Wq[k][n] )
//
// The integer dot of a whole group is finished (exact, INT32) before either scale is applied.
//
// gq_quantize_act: a_scale[m][g] = max_{k ∈ g} |A[m][k]| / 127 (FP32 division) and
// Aq[m][k] = rint(A[m][k] / a_scale[m][g]) (FP32 division, ties to even), clamped to
// [-127, 127]; a group of zeros gets scale 0 and codes 0.  (The absmax reduction and cast of
// "量化与融合 kernel" section 四.5, with 127 for INT8 and one scale per group.)
//
// q8a8_kernel: CTA = 8 warps over one 64-column block (W8 packed layout) and one K slice of
// whole groups, up to 32 activation rows (blockIdx.y selects the row block).  Lane l owns
// columns l and 32 + l; warps split the rows into RB blocks of RT and the slice into 8 / RB
// parts.  The INT8 codes need no decode: the 16 bytes of a chunk are 16 consecutive k of one
// column, so four dp4a against the row's 16 activation codes (one 16-byte shared-memory
// broadcast) give the chunk's dot.  Codes stream through a per-lane cp.async ring.  K parts
// are added in part order through shared memory, K slices by the last CTA of the block in
// slice order (fixed order: bitwise reproducible).
#include "gq_device.cuh"

namespace gq {

constexpr int kA8Threads = 256;
constexpr int kA8Warps = 8;
constexpr int kA8Cols = 64;
constexpr int kA8MaxRows = 32;                 // rows per CTA (more rows: more row blocks)
constexpr size_t kA8SmemCap = 113u << 10;      // two CTAs per SM

namespace a8 {

__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ int dp4a(int a, int b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

}  // namespace a8

// ------------------------------------------------------------------ activation quantizer

// One warp per (row, group): lanes stride the group's G values.
template <bool F32>
__global__ void __launch_bounds__(256) quantize_act_kernel(const void *__restrict__ A,
                                                           int8_t *__restrict__ Aq,
                                                           float *__restrict__ a_scales, int M,
                                                           int K, int G) {
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int ng = K / G;
  if (wid >= (long long)M * ng) return;
  const int m = (int)(wid / ng), g = (int)(wid - (long long)m * ng);
  const size_t base = (size_t)m * K + (size_t)g * G;
  auto load = [&](int k) -> float {
    if (F32) return reinterpret_cast<const float *>(A)[base + k];
    return __uint_as_float((uint32_t)reinterpret_cast<const unsigned short *>(A)[base + k] << 16);
  };
  float amax = 0.f;
  for (int k = lane; k < G; k += 32) amax = fmaxf(amax, fabsf(load(k)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.f);
  for (int k = lane; k < G; k += 32) {
    int q = 0;
    if (s > 0.f) {
      const float r = rintf(__fdiv_rn(load(k), s));
      q = (int)fminf(fmaxf(r, -127.f), 127.f);
    }
    Aq[base + k] = (int8_t)q;
  }
  if (lane == 0) a_scales[(size_t)m * ng + g] = s;
}

cudaError_t launch_quantize_act(int M, int K, int G, bool f32, const void *A, int8_t *Aq,
                                float *a_scales, cudaStream_t s) {
  const long long warps = (long long)M * (K / G);
  const long long blocks = (warps + 7) / 8;
  if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  if (f32)
    quantize_act_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(A, Aq, a_scales, M, K, G);
  else
    quantize_act_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(A, Aq, a_scales, M, K, G);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ W8A8 group GEMM

struct A8Params {
  const uint4 *Wp;            // packed codes, 64-column blocks of K/16 chunk rows
  const int8_t *Aq;           // [M][K]
  const float *As;            // [M][K/G]
  const float *S;             // [K/G][N]
  void *out;                  // [M][N]
  float *part;                // [KS][M][N] FP32 slice partial sums (KS > 1)
  unsigned *counters;         // per (row block, column block) (KS > 1)
  int M, K, N, G;
  int KS, NB;
  int out_f32;
};

__host__ __device__ inline int a8_rt(int Mb) {
  int rt = 1;
  while (rt < Mb && rt < 8) rt *= 2;
  return rt;
}
__host__ __device__ inline int a8_rb(int Mb) {
  int rb = 1;
  while (rb * 8 < Mb) rb *= 2;
  return rb;
}
__host__ __device__ inline int a8_pd(int rt) { return rt <= 2 ? 8 : rt == 4 ? 6 : 4; }
// shared memory: [activation codes MR x W bytes][activation scales MR x ngw floats]
// [K-part reduction KP x MR x 64 floats][8 warps x PD ring slots of 1 KiB]
__host__ __device__ inline size_t a8_codes_bytes(int mr, int W) { return ((size_t)mr * W + 15) / 16 * 16; }
__host__ __device__ inline size_t a8_scale_bytes(int mr, int ngw) {
  return ((size_t)mr * ngw * 4 + 15) / 16 * 16;    // keeps the ring 16-byte aligned
}
__host__ __device__ inline size_t a8_smem_bytes(int Mb, int K, int G, int KS) {
  const int rt = a8_rt(Mb), rb = a8_rb(Mb), mr = rt * rb, kp = kA8Warps / rb;
  const int ngw = (K / G + KS - 1) / KS, W = ngw * G;
  return a8_codes_bytes(mr, W) + a8_scale_bytes(mr, ngw) + (size_t)kp * mr * kA8Cols * 4 +
         (size_t)kA8Warps * a8_pd(rt) * 1024;
}

template <int RT, int PD>
__global__ void __launch_bounds__(kA8Threads, 2) q8a8_kernel(const A8Params p) {
  using namespace a8;
  extern __shared__ __align__(16) unsigned char sa[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = blockIdx.x / p.NB, nb = blockIdx.x - ks * p.NB;
  const int m0 = blockIdx.y * kA8MaxRows;
  const int Mb = min(kA8MaxRows, p.M - m0);        // rows of this row block
  const int K = p.K, N = p.N, G = p.G;
  const int RB = a8_rb(Mb), KP = kA8Warps / RB, MR = RB * RT;
  const int rb = warp % RB, kp = warp / RB;
  const int n0 = nb * kA8Cols, wb = min(kA8Cols, N - n0);
  const int groups = K / G, ngw = (groups + p.KS - 1) / p.KS, W = ngw * G;
  int gs0, gs1;
  zsplit_dev(groups, p.KS, ks, gs0, gs1);
  int gp0, gp1;
  zsplit_dev(gs1 - gs0, KP, kp, gp0, gp1);
  gp0 += gs0;
  gp1 += gs0;
  const int k0 = gs0 * G, ksl = (gs1 - gs0) * G;
  const int cpg = G / kChunkK8;
  const int c0 = gp0 * cpg, nch = (gp1 - gp0) * cpg;

  int8_t *acode = reinterpret_cast<int8_t *>(sa);                          // [MR][W]
  float *ascale = reinterpret_cast<float *>(sa + a8_codes_bytes(MR, W));    // [MR][ngw]
  float *red = reinterpret_cast<float *>(sa + a8_codes_bytes(MR, W) + a8_scale_bytes(MR, ngw));
  const size_t off_ring = a8_codes_bytes(MR, W) + a8_scale_bytes(MR, ngw) +
                          (size_t)KP * MR * kA8Cols * 4;                    // [KP][MR][64] above
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(sa) + (uint32_t)off_ring +
                          (uint32_t)(warp * PD * 1024 + lane * 16);
  const uint4 *ringp = reinterpret_cast<const uint4 *>(sa + off_ring + warp * PD * 1024 + lane * 16);

  // codes of columns n0 + l and n0 + 32 + l (clamped in a narrow block)
  const int ja = min(lane, wb - 1), jc = min(32 + lane, wb - 1);
  const uint4 *blk = p.Wp + (size_t)nb * (kA8Cols / kChunkK8) * K + (size_t)c0 * wb;
  const uint4 *wa = blk + ja, *wc = blk + jc;
#pragma unroll
  for (int j = 0; j < PD; ++j) {
    if (j < nch) {
      cp16(ring_s + j * 1024, wa + (size_t)j * wb);
      cp16(ring_s + j * 1024 + 512, wc + (size_t)j * wb);
    }
    cp_commit();
  }

  // the slice's activation codes (16 bytes per thread step) and scales, zero rows padded
  const int q16 = ksl >> 4;
  for (int idx = threadIdx.x; idx < MR * q16; idx += blockDim.x) {
    const int m = idx / q16, k = (idx - m * q16) * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m < Mb) v = __ldg(reinterpret_cast<const uint4 *>(p.Aq + (size_t)(m0 + m) * K + k0 + k));
    *reinterpret_cast<uint4 *>(acode + (size_t)m * W + k) = v;
  }
  for (int idx = threadIdx.x; idx < MR * (gs1 - gs0); idx += blockDim.x) {
    const int m = idx / (gs1 - gs0), gg = idx - m * (gs1 - gs0);
    ascale[(size_t)m * ngw + gg] = m < Mb ? __ldg(p.As + (size_t)(m0 + m) * groups + gs0 + gg) : 0.f;
  }
  __syncthreads();

  const float *sca = p.S + n0 + ja, *scc = p.S + n0 + jc;
  float acc[RT][2];
  int da[RT], dc[RT];                              // the current group's integer dots
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    acc[r][0] = acc[r][1] = 0.f;
    da[r] = dc[r] = 0;
  }
  const int8_t *arow = acode + (size_t)(rb * RT) * W + (gp0 * G - k0);
  const float *srow = ascale + (size_t)(rb * RT) * ngw + (gp0 - gs0);
  int grp = gp0, st = 0;
  for (int base = 0; base < nch; base += PD) {
#pragma unroll
    for (int j = 0; j < PD; ++j) {
      const int c = base + j;
      if (c < nch) {
        cp_wait<PD - 1>();                         // this lane's copies of chunk c landed
        const uint4 va = ringp[j * 64], vc = ringp[j * 64 + 32];
        const int xa[4] = {(int)va.x, (int)va.y, (int)va.z, (int)va.w};
        const int xc[4] = {(int)vc.x, (int)vc.y, (int)vc.z, (int)vc.w};
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          const uint4 av = *reinterpret_cast<const uint4 *>(arow + (size_t)r * W + c * 16);
          const int aw[4] = {(int)av.x, (int)av.y, (int)av.z, (int)av.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            da[r] = dp4a(xa[e], aw[e], da[r]);
            dc[r] = dp4a(xc[e], aw[e], dc[r]);
          }
        }
        // the slot's data is consumed: refill it with chunk c + PD
        if (c + PD < nch) {
          cp16(ring_s + j * 1024, wa + (size_t)(c + PD) * wb);
          cp16(ring_s + j * 1024 + 512, wc + (size_t)(c + PD) * wb);
        }
        cp_commit();
        if (++st == cpg) {                         // a whole group: scale its exact dots in
          st = 0;
          const float ba = __ldg(sca + (size_t)grp * N), bc = __ldg(scc + (size_t)grp * N);
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const float as = srow[(size_t)r * ngw + (grp - gp0)];
            acc[r][0] = fmaf(as * ba, (float)da[r], acc[r][0]);
            acc[r][1] = fmaf(as * bc, (float)dc[r], acc[r][1]);
            da[r] = dc[r] = 0;
          }
          ++grp;
        }
      }
    }
  }
  cp_wait<0>();

  // K parts in part order: red[kp][m][64]
  __syncthreads();
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    const int m = rb * RT + r;
    red[((size_t)kp * MR + m) * kA8Cols + lane] = acc[r][0];
    red[((size_t)kp * MR + m) * kA8Cols + 32 + lane] = acc[r][1];
  }
  __syncthreads();
  const bool split = p.KS > 1;
  for (int idx = threadIdx.x; idx < Mb * kA8Cols; idx += blockDim.x) {
    const int m = idx / kA8Cols, c = idx - m * kA8Cols, n = n0 + c;
    float sum = 0.f;
    for (int q = 0; q < KP; ++q) sum += red[((size_t)q * MR + m) * kA8Cols + c];
    if (c < wb) {
      if (split)
        p.part[((size_t)ks * p.M + m0 + m) * N + n] = sum;
      else
        store_out_rt(p.out, (size_t)(m0 + m) * N + n, sum, p.out_f32 != 0);
    }
  }
  if (!split) return;
  if (!last_arriver(p.counters + (size_t)blockIdx.y * p.NB + nb, p.KS)) return;
  for (int idx = threadIdx.x; idx < Mb * kA8Cols; idx += blockDim.x) {
    const int m = idx / kA8Cols, c = idx - m * kA8Cols, n = n0 + c;
    if (c >= wb) continue;
    float sum = 0.f;
    for (int s2 = 0; s2 < p.KS; ++s2)
      sum += __ldcg(p.part + ((size_t)s2 * p.M + m0 + m) * N + n);
    store_out_rt(p.out, (size_t)(m0 + m) * N + n, sum, p.out_f32 != 0);
  }
}

// K slices: up to 8 rows the fewest whose shared memory fits two CTAs per SM (load-latency
// bound); above, the fewest waves of two CTAs per SM with 5% charged per slice.  Every warp of
// a split CTA keeps a group.
int q8a8_slices(int M, int K, int N, int G, int sms, size_t part_cap, int forced) {
  const int Mb = M < kA8MaxRows ? M : kA8MaxRows;
  const int groups = K / G, kp = kA8Warps / a8_rb(Mb);
  const long ctas1 = (long)((N + kA8Cols - 1) / kA8Cols) * ((M + kA8MaxRows - 1) / kA8MaxRows);
  int best = 0, largest = 0;
  double best_cost = 0.0;
  for (int ks = 1; ks <= groups; ++ks) {
    if (ks > 1 && groups / ks < kp) break;
    if (ks > 1 && (size_t)ks * M * N * 4 > part_cap) break;
    if (a8_smem_bytes(Mb, K, G, ks) > kA8SmemCap) continue;
    largest = ks;
    if (forced != 0) {
      if (forced == ks) return ks;
      continue;
    }
    if (Mb <= 8) return ks;
    const long waves = (ctas1 * ks + 2L * sms - 1) / (2L * sms);
    const double cost = (double)waves / ks * (1.0 + 0.05 * ks);
    if (best == 0 || cost < best_cost * (1.0 - 1e-9)) {
      best = ks;
      best_cost = cost;
    }
  }
  if (forced == -1) return largest;
  return forced != 0 ? 0 : best;
}

size_t q8a8_smem_bytes(int M, int K, int G, int KS) {
  return a8_smem_bytes(M < kA8MaxRows ? M : kA8MaxRows, K, G, KS);
}

cudaError_t launch_q8a8(const Plan &pl, int M, int K, int N, int G, int prec, const int8_t *Aq,
                        const float *As, const void *Wq, const void *scales, void *out,
                        float *part, unsigned *counters, cudaStream_t s) {
  A8Params ap;
  ap.Wp = reinterpret_cast<const uint4 *>(Wq);
  ap.Aq = Aq;
  ap.As = As;
  ap.S = reinterpret_cast<const float *>(scales);
  ap.out = out;
  ap.part = part;
  ap.counters = counters;
  ap.M = M;
  ap.K = K;
  ap.N = N;
  ap.G = G;
  ap.KS = pl.nsplit;
  ap.NB = (N + kA8Cols - 1) / kA8Cols;
  ap.out_f32 = (prec & GQ_OUT_F32) ? 1 : 0;
  const dim3 grid(pl.grid_x, pl.grid_z);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                         pl.smem_bytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kA8Threads, pl.smem_bytes, s>>>(ap);
    return cudaGetLastError();
  };
  // every row block but the last has 32 rows: all of them run with RT of the first block
  switch (a8_rt(M < kA8MaxRows ? M : kA8MaxRows)) {
    case 1: return go(q8a8_kernel<1, 8>);
    case 2: return go(q8a8_kernel<2, 8>);
    case 4: return go(q8a8_kernel<4, 6>);
    case 8: return go(q8a8_kernel<8, 4>);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gq

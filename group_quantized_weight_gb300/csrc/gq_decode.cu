// Small-M ("decode") kernels of the group-quantized weight-only GEMM.
//
// Both kernels stream the packed weights once with 16-byte loads (a warp reads 512
// contiguous bytes per instruction), decode the codes in registers, multiply by the
// activations in FP32, apply each group's scale after the whole group's dot product, and
// split K over whole groups in a single launch (the z-split of "04 · 分组量化 GEMM 内核",
// section 3.3).  Split partial sums go to a scratch buffer; the last CTA to finish a tile
// (per-tile arrival counter) adds the partials in slice order 0, 1, ..., nsplit-1, so the
// result is bitwise reproducible from run to run (same section: the fixed-order reduction
// is what makes the result deterministic).
//
// W4 (path 0): tensor cores via mma.sync m16n8k16 with the roles swapped — the 16 MMA rows
// are 16 output columns n (weights, decoded in registers) and the 8 MMA columns are rows
// m of A — so that a single activation row wastes 7/8 of an MMA that is nearly free, while
// the decode stays at about one instruction per code (the magic-number decode of
// "GPU Kernel 工程（09）：量化与融合 kernel", section 2.4, in its BF16 form: the two codes of
// a pair sit in the low nibbles of the two 16-bit halves, OR 0x4300 makes bf16(128 + q),
// and one bf16x2 subtraction of bf16(128 + z) leaves the exact integer q − z).  Products
// of integers |q − z| ≤ 15 with bf16 activations are exact and accumulate in FP32.
//
// W8 (path 1): CUDA cores, one output column per thread (the "each thread owns columns and
// scans K" mapping of "分组量化 GEMM 内核", section 3.2, with activations broadcast from
// shared memory).  An INT8 code c becomes the exact float c by placing (c xor 0x80) in the
// low byte of 2^23 and subtracting 2^23 + 128.
#include "gq_device.cuh"

namespace gq {

// ------------------------------------------------------------------ W4, tensor cores

constexpr int kPF = 4;   // packed chunks in flight per lane (16 B each)


template <int MT, int SC, bool ZP, bool OUTF32>
__global__ void __launch_bounds__(kDecWarps * 32)
w4_mma_decode_kernel(const uint4 *__restrict__ Wp, const uint32_t *__restrict__ A32,
                     const void *__restrict__ scales, const uint32_t *__restrict__ zeros,
                     void *__restrict__ out, float *__restrict__ part,
                     unsigned *__restrict__ counters, int M, int K, int N, int G,
                     int nsplit, int units, int unit_k) {
  extern __shared__ __align__(16) uint32_t sA[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int z = blockIdx.y;
  const int m0 = blockIdx.z * (8 * MT);
  const int Mb = min(8 * MT, M - m0);
  int ub, ue;
  zsplit_dev(units, nsplit, z, ub, ue);
  const int kb = ub * unit_k, ke = ue * unit_k;
  const int nchunks = (ke - kb) / kChunkK;
  const int RS = act_row_words(nchunks);

  {  // stage the activation slice
    const int wpr = (ke - kb) >> 1;
    for (int idx = threadIdx.x; idx < Mb * wpr; idx += blockDim.x) {
      const int m = idx / wpr, w = idx - m * wpr;
      const int kk = 2 * w;
      const int c = kk >> 6, r = kk & 63, j = r >> 4, h = (r >> 3) & 1, q = (r & 7) >> 1;
      sA[m * RS + c * 32 + (j >> 1) * 16 + q * 4 + (j & 1) * 2 + h] =
          A32[(((size_t)(m0 + m) * K + kb) >> 1) + w];
    }
  }
  __syncthreads();

  const int n0 = (blockIdx.x * kDecWarps + warp) * kTileN;
  const int r0 = lane >> 2, q = lane & 3;
  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;

  if (n0 < N) {
    const uint4 *wp = Wp + ((size_t)(n0 / kTileN) * (K / kChunkK) + kb / kChunkK) * 32 + lane;
    const int na = min(n0 + r0, N - 1), nb = min(n0 + r0 + 8, N - 1);
    const int spg = G / 16;
    const int g_end = ke / G;
    int g = kb / G;
    const int NW = N >> 3;
    const int zwa = min(n0 >> 3, NW - 1), zwb = min((n0 >> 3) + 1, NW - 1);

    // scales (and zero-point words) of groups g, g+1, g+2 in flight
    uint32_t sa0 = ld_scale_bits<SC>(scales, (size_t)g * N + na);
    uint32_t sb0 = ld_scale_bits<SC>(scales, (size_t)g * N + nb);
    uint32_t sa1 = 0, sb1 = 0, sa2 = 0, sb2 = 0;
    if (g + 1 < g_end) {
      sa1 = ld_scale_bits<SC>(scales, (size_t)(g + 1) * N + na);
      sb1 = ld_scale_bits<SC>(scales, (size_t)(g + 1) * N + nb);
    }
    if (g + 2 < g_end) {
      sa2 = ld_scale_bits<SC>(scales, (size_t)(g + 2) * N + na);
      sb2 = ld_scale_bits<SC>(scales, (size_t)(g + 2) * N + nb);
    }
    uint32_t za0 = 0, zb0 = 0, za1 = 0, zb1 = 0, za2 = 0, zb2 = 0;
    if (ZP) {
      za0 = __ldg(zeros + (size_t)g * NW + zwa);
      zb0 = __ldg(zeros + (size_t)g * NW + zwb);
      if (g + 1 < g_end) {
        za1 = __ldg(zeros + (size_t)(g + 1) * NW + zwa);
        zb1 = __ldg(zeros + (size_t)(g + 1) * NW + zwb);
      }
      if (g + 2 < g_end) {
        za2 = __ldg(zeros + (size_t)(g + 2) * NW + zwa);
        zb2 = __ldg(zeros + (size_t)(g + 2) * NW + zwb);
      }
    }
    auto zz_of = [&](uint32_t zw) -> uint32_t {
      if (!ZP) return 0x43084308u;                 // bf16(128 + 8) in both halves
      const uint32_t zc = (zw >> (4 * r0)) & 0xFu;
      return (0x4300u | zc) * 0x00010001u;         // bf16(128 + z) in both halves
    };
    uint32_t zz0 = zz_of(za0), zz1 = zz_of(zb0);

    float d[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) d[mt][e] = 0.f;
    int ks = 0;

    uint4 buf[kPF];
#pragma unroll
    for (int i = 0; i < kPF; ++i)
      buf[i] = (i < nchunks) ? ld_stream(wp + (size_t)i * 32) : make_uint4(0, 0, 0, 0);

    for (int c0 = 0; c0 < nchunks; c0 += kPF) {
#pragma unroll
      for (int i = 0; i < kPF; ++i) {
        const int c = c0 + i;
        if (c >= nchunks) break;
        const uint4 cur = buf[i];
        if (c + kPF < nchunks) buf[i] = ld_stream(wp + (size_t)(c + kPF) * 32);

        uint32_t bq[MT][8];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int m = r0 + 8 * mt;
          if (m < Mb) {
            const uint4 lo = *reinterpret_cast<const uint4 *>(sA + m * RS + c * 32 + q * 4);
            const uint4 hi = *reinterpret_cast<const uint4 *>(sA + m * RS + c * 32 + 16 + q * 4);
            bq[mt][0] = lo.x; bq[mt][1] = lo.y; bq[mt][2] = lo.z; bq[mt][3] = lo.w;
            bq[mt][4] = hi.x; bq[mt][5] = hi.y; bq[mt][6] = hi.z; bq[mt][7] = hi.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) bq[mt][e] = 0u;
          }
        }
        const uint32_t words[4] = {cur.x, cur.y, cur.z, cur.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w = words[j];
          const uint32_t a0 = bf16x2_sub(nib_pair(w), zz0);
          const uint32_t a1 = bf16x2_sub(nib_pair(w >> 4), zz1);
          const uint32_t a2 = bf16x2_sub(nib_pair(w >> 8), zz0);
          const uint32_t a3 = bf16x2_sub(nib_pair(w >> 12), zz1);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            mma_16816(d[mt], a0, a1, a2, a3, bq[mt][2 * j], bq[mt][2 * j + 1]);
          if (++ks == spg) {   // a whole group is done: scale it into the FP32 sums
            ks = 0;
            const float fa = scale_value<SC>(sa0), fb = scale_value<SC>(sb0);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              acc[mt][0] = fmaf(fa, d[mt][0], acc[mt][0]);
              acc[mt][1] = fmaf(fa, d[mt][1], acc[mt][1]);
              acc[mt][2] = fmaf(fb, d[mt][2], acc[mt][2]);
              acc[mt][3] = fmaf(fb, d[mt][3], acc[mt][3]);
              d[mt][0] = d[mt][1] = d[mt][2] = d[mt][3] = 0.f;
            }
            ++g;
            sa0 = sa1; sb0 = sb1; sa1 = sa2; sb1 = sb2;
            if (g + 2 < g_end) {
              sa2 = ld_scale_bits<SC>(scales, (size_t)(g + 2) * N + na);
              sb2 = ld_scale_bits<SC>(scales, (size_t)(g + 2) * N + nb);
            }
            if (ZP) {
              za0 = za1; zb0 = zb1; za1 = za2; zb1 = zb2;
              if (g + 2 < g_end) {
                za2 = __ldg(zeros + (size_t)(g + 2) * NW + zwa);
                zb2 = __ldg(zeros + (size_t)(g + 2) * NW + zwb);
              }
              zz0 = zz_of(za0);
              zz1 = zz_of(zb0);
            }
          }
        }
      }
    }

    // D fragment: e = 0,1 -> column n0 + r0; e = 2,3 -> n0 + r0 + 8; rows m0 + 8mt + 2q + (e & 1)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = n0 + r0 + 8 * (e >> 1);
        const int ml = 8 * mt + 2 * q + (e & 1);
        if (n < N && ml < Mb) {
          const int m = m0 + ml;
          if (nsplit == 1)
            store_out<OUTF32>(out, (size_t)m * N + n, acc[mt][e]);
          else
            part[((size_t)z * M + m) * N + n] = acc[mt][e];
        }
      }
  }

  if (nsplit > 1) {
    if (last_arriver(counters + blockIdx.z * gridDim.x + blockIdx.x, nsplit))
      reduce_tile<OUTF32>(part, out, M, N, nsplit, m0, Mb, blockIdx.x * kDecWarps * kTileN,
                          kDecWarps * kTileN);
  }
}

// ------------------------------------------------------------------ W8, CUDA cores

template <int MR, bool OUTF32>
__global__ void __launch_bounds__(kQ8Threads)
q8_decode_kernel(const uint4 *__restrict__ Wp, const float *__restrict__ A,
                 const float *__restrict__ S, void *__restrict__ out, float *__restrict__ part,
                 unsigned *__restrict__ counters, int M, int K, int N, int G, int nsplit,
                 int units, int unit_k) {
  extern __shared__ __align__(16) float sAf[];
  const int z = blockIdx.y;
  const int m0 = blockIdx.z * MR;
  const int Mb = min(MR, M - m0);
  int ub, ue;
  zsplit_dev(units, nsplit, z, ub, ue);
  const int kb = ub * unit_k, ke = ue * unit_k;
  const int KS = ke - kb;

  for (int idx = threadIdx.x; idx < Mb * (KS >> 2); idx += blockDim.x) {
    const int m = idx / (KS >> 2), v = idx - m * (KS >> 2);
    reinterpret_cast<float4 *>(sAf)[idx] =
        __ldg(reinterpret_cast<const float4 *>(A + (size_t)(m0 + m) * K + kb) + v);
  }
  __syncthreads();

  const int n = blockIdx.x * kQ8Threads + threadIdx.x;
  float acc[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) acc[m] = 0.f;

  if (n < N) {
    const uint4 *wp = Wp + w8_chunk_index(K, N, n, kb / kChunkK8);
    const int rs = w8_chunk_index(K, N, n, 1) - w8_chunk_index(K, N, n, 0);   // row stride
    const int nch = KS / kChunkK8;
    const int cpg = G / kChunkK8;
    const int g_end = ke / G;
    int g = kb / G;
    float s0 = __ldg(S + (size_t)g * N + n);
    float s1 = (g + 1 < g_end) ? __ldg(S + (size_t)(g + 1) * N + n) : 0.f;
    float s2 = (g + 2 < g_end) ? __ldg(S + (size_t)(g + 2) * N + n) : 0.f;
    float2 p[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) p[m] = make_float2(0.f, 0.f);
    int cg = 0;

    uint4 buf[kPF];
#pragma unroll
    for (int i = 0; i < kPF; ++i)
      buf[i] = (i < nch) ? ld_stream(wp + (size_t)i * rs) : make_uint4(0, 0, 0, 0);

    for (int c0 = 0; c0 < nch; c0 += kPF) {
#pragma unroll
      for (int i = 0; i < kPF; ++i) {
        const int c = c0 + i;
        if (c >= nch) break;
        const uint4 cur = buf[i];
        if (c + kPF < nch) buf[i] = ld_stream(wp + (size_t)(c + kPF) * rs);
        const uint32_t words[4] = {cur.x ^ 0x80808080u, cur.y ^ 0x80808080u,
                                   cur.z ^ 0x80808080u, cur.w ^ 0x80808080u};
        float f[16];
#pragma unroll
        for (int b = 0; b < 16; ++b)
          f[b] = __uint_as_float(__byte_perm(words[b >> 2], 0x4B000000u, 0x7540u + (b & 3))) -
                 8388736.0f;   // 2^23 + 128
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          if (m < Mb) {
            const float4 *a4 = reinterpret_cast<const float4 *>(sAf + m * KS + c * kChunkK8);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const float4 a = a4[v];
              p[m] = ffma2(make_float2(f[4 * v], f[4 * v + 1]), make_float2(a.x, a.y), p[m]);
              p[m] = ffma2(make_float2(f[4 * v + 2], f[4 * v + 3]), make_float2(a.z, a.w), p[m]);
            }
          }
        }
        if (++cg == cpg) {
          cg = 0;
#pragma unroll
          for (int m = 0; m < MR; ++m) {
            acc[m] = fmaf(s0, p[m].x + p[m].y, acc[m]);
            p[m] = make_float2(0.f, 0.f);
          }
          ++g;
          s0 = s1; s1 = s2;
          if (g + 2 < g_end) s2 = __ldg(S + (size_t)(g + 2) * N + n);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      if (m < Mb) {
        if (nsplit == 1)
          store_out<OUTF32>(out, (size_t)(m0 + m) * N + n, acc[m]);
        else
          part[((size_t)z * M + m0 + m) * N + n] = acc[m];
      }
    }
  }

  if (nsplit > 1) {
    if (last_arriver(counters + blockIdx.z * gridDim.x + blockIdx.x, nsplit))
      reduce_tile<OUTF32>(part, out, M, N, nsplit, m0, Mb, blockIdx.x * kQ8Threads, kQ8Threads);
  }
}

// ------------------------------------------------------------------ launchers

template <int MT, int SC, bool ZP, bool OUTF32>
static cudaError_t launch_w4_t(const Plan &p, int M, int K, int N, int G, const void *A,
                               const void *Wq, const void *scales, const void *zeros,
                               void *out, float *part, unsigned *counters, cudaStream_t s) {
  auto kern = w4_mma_decode_kernel<MT, SC, ZP, OUTF32>;
  if (p.smem_bytes > 48 * 1024) {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                         p.smem_bytes);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(p.grid_x, p.grid_y, p.grid_z);
  kern<<<grid, p.block_threads, p.smem_bytes, s>>>(
      reinterpret_cast<const uint4 *>(Wq), reinterpret_cast<const uint32_t *>(A), scales,
      reinterpret_cast<const uint32_t *>(zeros), out, part, counters, M, K, N, G, p.nsplit,
      p.units, p.unit_k);
  return cudaGetLastError();
}

template <int MT, int SC, bool ZP>
static cudaError_t launch_w4_o(const Plan &p, int prec, int M, int K, int N, int G,
                               const void *A, const void *Wq, const void *scales,
                               const void *zeros, void *out, float *part, unsigned *cnt,
                               cudaStream_t s) {
  if (prec & GQ_OUT_F32)
    return launch_w4_t<MT, SC, ZP, true>(p, M, K, N, G, A, Wq, scales, zeros, out, part, cnt, s);
  return launch_w4_t<MT, SC, ZP, false>(p, M, K, N, G, A, Wq, scales, zeros, out, part, cnt, s);
}

template <int MT, int SC>
static cudaError_t launch_w4_z(const Plan &p, int prec, int M, int K, int N, int G,
                               const void *A, const void *Wq, const void *scales,
                               const void *zeros, void *out, float *part, unsigned *cnt,
                               cudaStream_t s) {
  if (prec & GQ_ZP)
    return launch_w4_o<MT, SC, true>(p, prec, M, K, N, G, A, Wq, scales, zeros, out, part, cnt, s);
  return launch_w4_o<MT, SC, false>(p, prec, M, K, N, G, A, Wq, scales, zeros, out, part, cnt, s);
}

template <int MT>
static cudaError_t launch_w4_s(const Plan &p, int prec, int M, int K, int N, int G,
                               const void *A, const void *Wq, const void *scales,
                               const void *zeros, void *out, float *part, unsigned *cnt,
                               cudaStream_t s) {
  if (prec & GQ_SC_F32)
    return launch_w4_z<MT, kScF32>(p, prec, M, K, N, G, A, Wq, scales, zeros, out, part, cnt, s);
  if (prec & GQ_SC_BF16)
    return launch_w4_z<MT, kScBF16>(p, prec, M, K, N, G, A, Wq, scales, zeros, out, part, cnt, s);
  return launch_w4_z<MT, kScF16>(p, prec, M, K, N, G, A, Wq, scales, zeros, out, part, cnt, s);
}

cudaError_t launch_mma_decode(const Plan &p, int M, int K, int N, int G, int prec,
                              const void *A, const void *Wq, const void *scales,
                              const void *zeros, void *out, float *part, unsigned *counters,
                              cudaStream_t s) {
  switch (p.mt) {
    case 1: return launch_w4_s<1>(p, prec, M, K, N, G, A, Wq, scales, zeros, out, part, counters, s);
    case 2: return launch_w4_s<2>(p, prec, M, K, N, G, A, Wq, scales, zeros, out, part, counters, s);
    case 3: return launch_w4_s<3>(p, prec, M, K, N, G, A, Wq, scales, zeros, out, part, counters, s);
    case 4: return launch_w4_s<4>(p, prec, M, K, N, G, A, Wq, scales, zeros, out, part, counters, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int MR, bool OUTF32>
static cudaError_t launch_q8_t(const Plan &p, int M, int K, int N, int G, const void *A,
                               const void *Wq, const void *scales, void *out, float *part,
                               unsigned *counters, cudaStream_t s) {
  auto kern = q8_decode_kernel<MR, OUTF32>;
  if (p.smem_bytes > 48 * 1024) {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                         p.smem_bytes);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(p.grid_x, p.grid_y, p.grid_z);
  kern<<<grid, p.block_threads, p.smem_bytes, s>>>(
      reinterpret_cast<const uint4 *>(Wq), reinterpret_cast<const float *>(A),
      reinterpret_cast<const float *>(scales), out, part, counters, M, K, N, G, p.nsplit,
      p.units, p.unit_k);
  return cudaGetLastError();
}

template <int MR>
static cudaError_t launch_q8_o(const Plan &p, int prec, int M, int K, int N, int G,
                               const void *A, const void *Wq, const void *scales, void *out,
                               float *part, unsigned *counters, cudaStream_t s) {
  if (prec & GQ_OUT_F32)
    return launch_q8_t<MR, true>(p, M, K, N, G, A, Wq, scales, out, part, counters, s);
  return launch_q8_t<MR, false>(p, M, K, N, G, A, Wq, scales, out, part, counters, s);
}

cudaError_t launch_q8_decode(const Plan &p, int M, int K, int N, int G, int prec,
                             const void *A, const void *Wq, const void *scales, void *out,
                             float *part, unsigned *counters, cudaStream_t s) {
  switch (p.m_tile) {
    case 1: return launch_q8_o<1>(p, prec, M, K, N, G, A, Wq, scales, out, part, counters, s);
    case 2: return launch_q8_o<2>(p, prec, M, K, N, G, A, Wq, scales, out, part, counters, s);
    case 4: return launch_q8_o<4>(p, prec, M, K, N, G, A, Wq, scales, out, part, counters, s);
    case 8: return launch_q8_o<8>(p, prec, M, K, N, G, A, Wq, scales, out, part, counters, s);
    case 16: return launch_q8_o<16>(p, prec, M, K, N, G, A, Wq, scales, out, part, counters, s);
    case 32: return launch_q8_o<32>(p, prec, M, K, N, G, A, Wq, scales, out, part, counters, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gq

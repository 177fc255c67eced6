// INT8 (Q8_0-style) kernel of the group-quantized weight-only GEMM for M <= 32, on CUDA cores.
//
// The FP32 output tolerance leaves no room for tensor-core arithmetic on fp32 activations
// (TF32 rounds them), so every product is an FP32 FMA on CUDA cores.  The group-wise
// product of "04 · 分组量化 GEMM 内核", section 2 (activation scale fixed to 1) is
// reassociated: a code is first turned into the exact float c and multiplied by its group's
// scale (one rounding), and the scaled weights meet the activations in FP32 FMAs.  That is
// the same sum over k as scaling per-group sums, within one FP32 rounding per weight.
//
// Blocking.  A CTA of 8 warps owns 64 columns and one K slice (a contiguous run of whole
// groups).  Lane l of every warp owns columns n0 + l and n0 + 32 + l: per 16 k it loads two
// 16-byte code chunks, one contiguous KiB per warp, and in the column-block-major packed
// layout a warp's k range is one contiguous run of memory.  The warps split the CTA's rows into RB blocks of RT rows and its K slice
// into KP = 8 / RB parts of whole groups.  Products are paired along k: one fma.rn.f32x2
// multiplies the weights of k and k+1 of a column with the activations of k and k+1 of a row
// (one 16-byte shared-memory broadcast holds four k of a row) into separate even-k and odd-k
// sums, added at the end.  An INT8 code c becomes the exact float c by placing (c xor 0x80)
// in the low byte of 2^23 and subtracting 2^23 + 128.  A register ring keeps the next PD
// chunk pairs of the warp, and the scales of the groups they open, in flight.
//
// Reduction in a fixed order (bitwise reproducible): the K parts of a CTA are added in part
// order through shared memory; with several K slices every CTA writes FP32 partial sums and
// the last CTA of a column block (arrival counter) adds them in slice order — the split-K of
// "04 · 分组量化 GEMM 内核", section 3.3.
#include "gq_device.cuh"

namespace gq {

constexpr int kQbThreads = 256;              // 8 warps
constexpr int kQbWarps = 8;
constexpr int kQbCols = 64;                  // columns per CTA (2 per lane)
constexpr size_t kQbSmemCap = 113u << 10;    // two CTAs per SM

namespace qb {

// (z0, z1) += (x0, x1) * (y0, y1), one instruction
__device__ __forceinline__ void fma2(float &z0, float &z1, float x0, float x1, float y0,
                                     float y1) {
  asm("{\n\t.reg .b64 a, b, c;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 c, a, b, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "+f"(z0), "+f"(z1)
      : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

// byte b of word w (codes xor 0x80) placed in the low byte of 2^23: the float 2^23 + byte
__device__ __forceinline__ float biased(uint32_t w, int b) {
  return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + b));
}

// (x0, x1) *= (y, y)
__device__ __forceinline__ void mul2(float &x0, float &x1, float y) {
  asm("{\n\t.reg .b64 a, b;\n\t"
      "mov.b64 a, {%0, %1};\n\tmov.b64 b, {%2, %2};\n\t"
      "mul.rn.f32x2 a, a, b;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(x0), "+f"(x1)
      : "f"(y));
}

// (x0, x1) - (2^23 + 128): the signed codes, exact
__device__ __forceinline__ void unbias2(float &x0, float &x1) {
  fma2(x0, x1, 1.f, 1.f, -8388736.f, -8388736.f);
}

// 16-byte asynchronous copy global -> shared (L2 only), and its group bookkeeping
__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace qb

struct QbParams {
  const uint4 *Wp;            // packed codes, 64-column blocks of K/16 chunk rows
  const float *A;             // [M][K]
  const float *S;             // [K/G][N]
  void *out;                  // [M][N]
  float *part;                // [KS][M][N] FP32 slice partial sums (KS > 1)
  unsigned *counters;         // per column block (KS > 1)
  int M, K, N, G;
  int KS;                     // K slices (groups split as evenly as possible)
  int NB;                     // column blocks of 64
  int out_f32;
  int gate_up;                // fused gate+up: block b = gate columns 32b.. then up N/2 + 32b..;
                              // out [M][N/2] = silu(gate) * up
};

// Rows per warp RT (1, 2, 4 or 8) and row blocks RB (1, 2 or 4) for M rows.
__host__ __device__ inline int q8_rt(int M) {
  int rt = 1;
  while (rt < M && rt < 8) rt *= 2;
  return rt;
}
__host__ __device__ inline int q8_rb(int M) {
  int rb = 1;
  while (rb * 8 < M) rb *= 2;
  return rb;
}

// activation slice [MR][W] (or the K-part reduction, whichever is larger)
__host__ __device__ inline size_t q8_block_area_bytes(int M, int K, int G, int KS) {
  const int rt = q8_rt(M), rb = q8_rb(M), mr = rb * rt, kp = kQbWarps / rb;
  const int groups = K / G, widest = (groups + KS - 1) / KS;
  const size_t act = (size_t)mr * widest * G * 4, red = (size_t)kp * mr * kQbCols * 4;
  return act > red ? act : red;
}

// chunk pairs in flight per warp (shared-memory ring slots of 1 KiB)
__host__ __device__ inline int q8_block_pd(int M) {
  const int rt = q8_rt(M);
  return rt <= 2 ? 8 : rt == 4 ? 6 : 3;
}

// Shared memory: the K slice's activations as [MR][W] fp32 (MR = RB * RT rows, zero rows
// padded; W = the widest slice's k), reused at the end for the K-part reduction [KP][MR][64].
template <int RT, int PD>
__global__ void __launch_bounds__(kQbThreads, 2) q8_block_kernel(const QbParams p) {
  using namespace qb;
  extern __shared__ __align__(16) float sq[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = blockIdx.x / p.NB, nb = blockIdx.x - ks * p.NB;
  const int n0 = nb * kQbCols;
  const int M = p.M, K = p.K, N = p.N, G = p.G;
  const int RB = q8_rb(M), KP = kQbWarps / RB, MR = RB * RT;
  const int rb = warp % RB, kp = warp / RB;
  const int groups = K / G;
  const int W = (groups + p.KS - 1) / p.KS * G;   // row stride of the activation slice

  int gs0, gs1;                                    // the CTA's groups
  zsplit_dev(groups, p.KS, ks, gs0, gs1);
  int gp0, gp1;                                    // this warp's groups
  zsplit_dev(gs1 - gs0, KP, kp, gp0, gp1);
  gp0 += gs0;
  gp1 += gs0;
  const int k0 = gs0 * G, ksl = (gs1 - gs0) * G;

  const int wb = min(kQbCols, N - n0);             // columns of this block (chunk row stride)
  const int ja = min(lane, wb - 1), jc = min(32 + lane, wb - 1);
  const int cpg = G / kChunkK8;                    // 16-k chunks per group (a power of two)
  const int c0 = gp0 * cpg, nch = (gp1 - gp0) * cpg;
  const uint4 *blk = p.Wp + (size_t)nb * (kQbCols / kChunkK8) * K + (size_t)c0 * wb;
  const uint4 *wa = blk + ja, *wc = blk + jc;
  // scales of this lane's two columns (gate+up: gate column 32 nb + lane, up N/2 + 32 nb + lane)
  const float *sca = p.S + (p.gate_up ? 32 * nb + ja : n0 + ja);
  const float *scc = p.S + (p.gate_up ? N / 2 + 32 * nb + (jc - 32) : n0 + jc);

  // the first PD chunk pairs (and the scales of the groups they open) go out before the
  // activations are staged.  Ring slot j of this warp: [2 columns][32 lanes][16 bytes] after
  // the activation / reduction area; each lane copies and later reads only its own pieces.
  const size_t area = q8_block_area_bytes(M, K, G, p.KS);
  const uint32_t ring = (uint32_t)__cvta_generic_to_shared(sq) + (uint32_t)area +
                        (uint32_t)(warp * PD * 1024 + lane * 16);
  const uint4 *ringp = reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(sq) + area +
                                                       warp * PD * 1024 + lane * 16);
  float sa[PD], sc[PD];
#pragma unroll
  for (int j = 0; j < PD; ++j) {
    sa[j] = sc[j] = 0.f;
    if (j < nch) {
      cp16(ring + j * 1024, wa + (size_t)j * wb);
      cp16(ring + j * 1024 + 512, wc + (size_t)j * wb);
      if ((j & (cpg - 1)) == 0) {
        const size_t g = (size_t)(c0 + j) / cpg;
        sa[j] = __ldg(sca + g * N);
        sc[j] = __ldg(scc + g * N);
      }
    }
    cp_commit();
  }

  // activations of the slice: sq[m * W + k], four k per thread
  const int q4 = ksl >> 2;
  for (int idx = threadIdx.x; idx < MR * q4; idx += blockDim.x) {
    const int m = idx / q4, k = (idx - m * q4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m < M) v = __ldg(reinterpret_cast<const float4 *>(p.A + (size_t)m * K + k0 + k));
    *reinterpret_cast<float4 *>(sq + (size_t)m * W + k) = v;
  }
  __syncthreads();

  float ae[RT][2], ao[RT][2];                      // per row, columns a and c: even / odd k
#pragma unroll
  for (int r = 0; r < RT; ++r) ae[r][0] = ae[r][1] = ao[r][0] = ao[r][1] = 0.f;
  const float *arow = sq + (size_t)(rb * RT) * W + (gp0 * G - k0);
  float ga = 0.f, gc = 0.f;                        // scales of the current group

  for (int base = 0; base < nch; base += PD) {
#pragma unroll
    for (int j = 0; j < PD; ++j) {
      const int c = base + j;
      if (c < nch) {
        cp_wait<PD - 1>();                         // this lane's copies of chunk c have landed
        const uint4 va = ringp[j * 64], vc = ringp[j * 64 + 32];
        if ((c & (cpg - 1)) == 0) {                // the chunk opens a group
          ga = sa[j];
          gc = sc[j];
        }
        const int cn = c + PD;
        if (cn < nch && (cn & (cpg - 1)) == 0) {
          const size_t g = (size_t)(c0 + cn) / cpg;
          sa[j] = __ldg(sca + g * N);
          sc[j] = __ldg(scc + g * N);
        }
        const uint32_t xa[4] = {va.x ^ 0x80808080u, va.y ^ 0x80808080u, va.z ^ 0x80808080u,
                                va.w ^ 0x80808080u};
        const uint32_t xc[4] = {vc.x ^ 0x80808080u, vc.y ^ 0x80808080u, vc.z ^ 0x80808080u,
                                vc.w ^ 0x80808080u};
#pragma unroll
        for (int q = 0; q < 4; ++q) {              // k = 16c + 4q .. +3
          float fa[4], fc[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            fa[b] = biased(xa[q], b);
            fc[b] = biased(xc[q], b);
          }
          unbias2(fa[0], fa[1]);
          unbias2(fa[2], fa[3]);
          unbias2(fc[0], fc[1]);
          unbias2(fc[2], fc[3]);
          mul2(fa[0], fa[1], ga);
          mul2(fa[2], fa[3], ga);
          mul2(fc[0], fc[1], gc);
          mul2(fc[2], fc[3], gc);
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const float4 a4 =
                *reinterpret_cast<const float4 *>(arow + (size_t)r * W + c * 16 + q * 4);
            fma2(ae[r][0], ao[r][0], fa[0], fa[1], a4.x, a4.y);
            fma2(ae[r][0], ao[r][0], fa[2], fa[3], a4.z, a4.w);
            fma2(ae[r][1], ao[r][1], fc[0], fc[1], a4.x, a4.y);
            fma2(ae[r][1], ao[r][1], fc[2], fc[3], a4.z, a4.w);
          }
        }
        // the slot's data is consumed: refill it with chunk c + PD (an empty group past the
        // end keeps the group count uniform)
        if (cn < nch) {
          cp16(ring + j * 1024, wa + (size_t)cn * wb);
          cp16(ring + j * 1024 + 512, wc + (size_t)cn * wb);
        }
        cp_commit();
      }
    }
  }
  cp_wait<0>();

  // the K parts of the CTA, added in part order: red[kp][m][64 columns]
  __syncthreads();                                 // every warp is done with the activations
  float *red = sq;
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    const int m = rb * RT + r;
    red[((size_t)kp * MR + m) * kQbCols + lane] = ae[r][0] + ao[r][0];
    red[((size_t)kp * MR + m) * kQbCols + 32 + lane] = ae[r][1] + ao[r][1];
  }
  __syncthreads();
  const bool split = p.KS > 1;
  if (p.gate_up && !split) {
    // gate column c < 32 of the block and its up column c + 32: out[m][32 nb + c]
    for (int idx = threadIdx.x; idx < M * 32; idx += blockDim.x) {
      const int m = idx >> 5, c = idx & 31;
      float g = 0.f, u = 0.f;
      for (int q = 0; q < KP; ++q) {
        g += red[((size_t)q * MR + m) * kQbCols + c];
        u += red[((size_t)q * MR + m) * kQbCols + 32 + c];
      }
      store_out_rt(p.out, (size_t)m * (N / 2) + 32 * nb + c, silu_mul(g, u), p.out_f32 != 0);
    }
    return;
  }
  for (int idx = threadIdx.x; idx < M * kQbCols; idx += blockDim.x) {
    const int m = idx / kQbCols, c = idx - m * kQbCols, n = n0 + c;
    float sum = 0.f;
    for (int q = 0; q < KP; ++q) sum += red[((size_t)q * MR + m) * kQbCols + c];
    if (n < N) {
      if (split)
        p.part[((size_t)ks * M + m) * N + n] = sum;
      else
        store_out_rt(p.out, (size_t)m * N + n, sum, p.out_f32 != 0);
    }
  }
  if (!split) return;
  // the last CTA of this column block adds the K slices in slice order
  if (!last_arriver(p.counters + nb, p.KS)) return;
  if (p.gate_up) {
    for (int idx = threadIdx.x; idx < M * 32; idx += blockDim.x) {
      const int m = idx >> 5, c = idx & 31;
      float g = 0.f, u = 0.f;
      for (int s2 = 0; s2 < p.KS; ++s2) {
        g += __ldcg(p.part + ((size_t)s2 * M + m) * N + n0 + c);
        u += __ldcg(p.part + ((size_t)s2 * M + m) * N + n0 + 32 + c);
      }
      store_out_rt(p.out, (size_t)m * (N / 2) + 32 * nb + c, silu_mul(g, u), p.out_f32 != 0);
    }
    return;
  }
  for (int idx = threadIdx.x; idx < M * kQbCols; idx += blockDim.x) {
    const int m = idx / kQbCols, n = n0 + idx - m * kQbCols;
    if (n >= N) continue;
    float sum = 0.f;
    for (int s2 = 0; s2 < p.KS; ++s2) sum += __ldcg(p.part + ((size_t)s2 * M + m) * N + n);
    store_out_rt(p.out, (size_t)m * N + n, sum, p.out_f32 != 0);
  }
}

// ------------------------------------------------------------------ tensor cores
//
// The same GEMM on BF16 tensor cores, exactly: every INT8 code is an integer of at most 8
// bits, exact in BF16, and every fp32 activation is the exact sum of three BF16 parts
// (a0 = bf16(a), a1 = bf16(a - a0), a2 = a - a0 - a1, each rounding to nearest), so each
// product code x part is exact in FP32 and the MMA only adds.  Per group the MMAs start
// from zero and the group's FP32 sum is multiplied by its scale after the whole group, as
// the group-wise GEMM of "04 · 分组量化 GEMM 内核", section 2 orders it.
//
// CTA = 8 warps over one 64-column block and one K slice: warp (mi, kp) owns the 16 columns
// mi·16 .. +15 (the rows of its m16n8k16 MMAs) and half the slice's groups (kp).  The MMA's
// 16 k slots are mapped onto the 16 k of a code chunk so that lane (g, t) needs bytes 4t ..
// 4t+3 of the chunks of columns g and g + 8 (A operand) and activations 4t .. 4t+3 of row g
// (B operand, one 8-byte load per part): slot 2t + e <-> k = 4t + e, slot 2t + 8 + e <->
// k = 4t + 2 + e.  A code byte c (two's complement) becomes a BF16 pair element as
// bf16(128 + (c & 0x7F)) - bf16(128 + (c & 0x80)), both halves built by one LOP3 each.

constexpr int kQmThreads = 256;
constexpr int kQmPD = 8;                       // ring slots per warp (2 code steps each)
constexpr int kQmMaxM = 32;

struct QmParams {
  const uint4 *Wp;            // packed codes, 64-column blocks of K/16 chunk rows
  const float *A;             // [M][K]
  const float *S;             // [K/G][N]
  void *out;                  // [M][N]
  float *part;                // [KS][M][N] FP32 slice partial sums (KS > 1)
  unsigned *counters;         // per column block (KS > 1)
  int M, K, N, G;
  int KS, NB;
  int out_f32;
  int gate_up;                // fused gate+up (as QbParams)
};

__host__ __device__ inline int q8m_rows8(int M) { return (M + 7) / 8 * 8; }
// bf16 elements per activation-plane row: the widest slice plus 16 (32 bytes: the eight
// rows a fragment load touches start in different bank quarters)
__host__ __device__ inline int q8m_row_stride(int K, int G, int KS) {
  return ((K / G) + KS - 1) / KS * G + 16;
}
__host__ __device__ inline size_t q8m_area_bytes(int M, int K, int G, int KS) {
  const size_t planes = (size_t)3 * q8m_rows8(M) * q8m_row_stride(K, G, KS) * 2;
  const size_t red = (size_t)2 * q8m_rows8(M) * 64 * 4;
  const size_t a = planes > red ? planes : red;
  return (a + 15) / 16 * 16;
}
// the slice's scales for the CTA's 64 columns: [widest slice's groups][64] fp32
__host__ __device__ inline size_t q8m_scale_bytes(int K, int G, int KS) {
  return (size_t)(((K / G) + KS - 1) / KS) * 64 * 4;
}

namespace qm {

__device__ __forceinline__ void mma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
               "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
  return d;
}

// codes in bytes 0 and 2 of x (two's complement) -> the BF16 pair (code0, code1)
__device__ __forceinline__ uint32_t codes_bf16x2(uint32_t x) {
  const uint32_t hi = and_or<0x007F007Fu>(x, 0x43004300u);   // 128 + (c & 0x7F)
  const uint32_t lo = and_or<0x00800080u>(x, 0x43004300u);   // 128 or 256
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(hi), "r"(lo));
  return d;
}

}  // namespace qm

template <int NB8>
__global__ void __launch_bounds__(kQmThreads, 2) q8_mma_kernel(const QmParams p) {
  using namespace qm;
  using namespace qb;
  extern __shared__ __align__(16) unsigned char smq[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int ks = blockIdx.x / p.NB, nb = blockIdx.x - ks * p.NB;
  const int M = p.M, K = p.K, N = p.N, G = p.G;
  const int n0 = nb * 64, wb = min(64, N - n0);
  const int mi = warp & 3, kp = warp >> 2;
  constexpr int MR8 = NB8 * 8;
  const int groups = K / G, Wp = q8m_row_stride(K, G, p.KS);
  int gs0, gs1;                                    // the CTA's groups
  zsplit_dev(groups, p.KS, ks, gs0, gs1);
  int gp0, gp1;                                    // this warp's groups
  zsplit_dev(gs1 - gs0, 2, kp, gp0, gp1);
  gp0 += gs0;
  gp1 += gs0;
  const int k0 = gs0 * G, ksl = (gs1 - gs0) * G;
  const int cpg = G / kChunkK8;                    // 16-k steps per group (2 .. 16)
  const int nslot = (gp1 - gp0) * cpg / 2;         // ring slots of this warp (2 steps each)

  // codes: lane copies column mi·16 + (lane & 15) of step (2·slot + lane / 16)
  const size_t area = q8m_area_bytes(M, K, G, p.KS);
  const size_t sbytes = q8m_scale_bytes(K, G, p.KS);
  const uint32_t smq_s = (uint32_t)__cvta_generic_to_shared(smq);
  // the slice's scales for the block's columns (one commit group, the oldest); pieces past
  // a narrow block's last column repeat its last four columns
  const float *ssm = reinterpret_cast<const float *>(smq + area);
  for (int idx = threadIdx.x; idx < (gs1 - gs0) * 16; idx += blockDim.x) {
    const int gr = idx >> 4, q = idx & 15, col = min(q * 4, wb - 4);
    // gate+up: block columns 0 .. 31 are gate columns 32 nb.., 32 .. 63 up columns N/2 + 32 nb..
    const int src = !p.gate_up ? n0 + col : col < 32 ? 32 * nb + col : N / 2 + 32 * nb + (col - 32);
    cp16(smq_s + (uint32_t)(area + gr * 256 + q * 16), p.S + (size_t)(gs0 + gr) * N + src);
  }
  cp_commit();
  const uint32_t ring_s = smq_s + (uint32_t)(area + sbytes) + (uint32_t)(warp * kQmPD * 512);
  const unsigned char *ring = smq + area + sbytes + warp * kQmPD * 512;
  const int ccol = min(mi * 16 + (lane & 15), wb - 1);
  const uint4 *csrc = p.Wp + (size_t)nb * (64 / kChunkK8) * K +
                      (size_t)(gp0 * cpg + (lane >> 4)) * wb + ccol;
  const uint32_t cdst = ring_s + (lane >> 4) * 256 + (lane & 15) * 16;
#pragma unroll
  for (int j = 0; j < kQmPD; ++j) {
    if (j < nslot) cp16(cdst + j * 512, csrc + (size_t)2 * j * wb);
    cp_commit();
  }

  // activations of the slice as three BF16 planes [3][MR8][Wp]
  __nv_bfloat16 *pl = reinterpret_cast<__nv_bfloat16 *>(smq);
  const int q4 = ksl >> 2, nq = MR8 * q4;
  for (int base = threadIdx.x; base < nq; base += 4 * kQmThreads) {
    float4 vv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {                  // four independent loads in flight
      const int idx = base + u * kQmThreads, m = idx / q4;
      vv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (idx < nq && m < M)
        vv[u] = __ldg(reinterpret_cast<const float4 *>(p.A + (size_t)m * K + k0 +
                                                      (idx - m * q4) * 4));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * kQmThreads;
      if (idx >= nq) break;
      const int m = idx / q4, k = (idx - m * q4) * 4;
      const float a[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
      uint32_t w[3][2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float r0 = a[2 * h], r1 = a[2 * h + 1];
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const __nv_bfloat162 bb = __floats2bfloat162_rn(r0, r1);
          w[part][h] = *reinterpret_cast<const uint32_t *>(&bb);
          r0 -= __bfloat162float(bb.x);
          r1 -= __bfloat162float(bb.y);
        }
      }
#pragma unroll
      for (int part = 0; part < 3; ++part)
        *reinterpret_cast<uint2 *>(pl + ((size_t)part * MR8 + m) * Wp + k) =
            make_uint2(w[part][0], w[part][1]);
    }
  }
  cp_wait<kQmPD>();                                // the scales (older than the ring) landed
  __syncthreads();

  // scales of the lane's two columns (MMA rows g and g + 8)
  const int cg = min(mi * 16 + g, wb - 1), cg8 = min(mi * 16 + g + 8, wb - 1);
  const float *s_g = ssm - (size_t)gs0 * 64 + cg, *s_g8 = ssm - (size_t)gs0 * 64 + cg8;
  float acc[NB8][4], d[NB8][4];
#pragma unroll
  for (int b = 0; b < NB8; ++b) acc[b][0] = acc[b][1] = acc[b][2] = acc[b][3] = 0.f;
  int grp = gp0;
  float sc0 = 0.f, sc8 = 0.f;
  if (gp0 < gp1) {
    sc0 = s_g[(size_t)grp * 64];
    sc8 = s_g8[(size_t)grp * 64];
  }
  const unsigned char *bbase = reinterpret_cast<const unsigned char *>(pl) +
                               ((size_t)g * Wp + (gp0 * G - k0) + 4 * t) * 2;
  int st = 0;                                      // step within the group
  for (int base = 0; base < nslot; base += kQmPD) {
#pragma unroll
    for (int j = 0; j < kQmPD; ++j) {
      const int sl = base + j;
      if (sl < nslot) {
        cp_wait<kQmPD - 1>();                      // this lane's copy of slot sl landed
        __syncwarp();                              // and so did every other lane's
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const unsigned char *cs = ring + j * 512 + h * 256;
          const uint32_t wg = *reinterpret_cast<const uint32_t *>(cs + g * 16 + 4 * t);
          const uint32_t wg8 = *reinterpret_cast<const uint32_t *>(cs + (g + 8) * 16 + 4 * t);
          const uint32_t a0 = codes_bf16x2(__byte_perm(wg, 0, 0x4140));
          const uint32_t a2 = codes_bf16x2(__byte_perm(wg, 0, 0x4342));
          const uint32_t a1 = codes_bf16x2(__byte_perm(wg8, 0, 0x4140));
          const uint32_t a3 = codes_bf16x2(__byte_perm(wg8, 0, 0x4342));
          if (st == 0) {
#pragma unroll
            for (int b = 0; b < NB8; ++b) d[b][0] = d[b][1] = d[b][2] = d[b][3] = 0.f;
          }
          const int kk = (2 * sl + h) * 16;        // k of this step from the warp's first
#pragma unroll
          for (int b = 0; b < NB8; ++b) {
#pragma unroll
            for (int part = 0; part < 3; ++part) {
              const uint2 bv = *reinterpret_cast<const uint2 *>(
                  bbase + (((size_t)part * MR8 + b * 8) * Wp + kk) * 2);
              mma_bf16(d[b], a0, a1, a2, a3, bv.x, bv.y);
            }
          }
          if (++st == cpg) {                       // the group is complete: scale it in
            st = 0;
#pragma unroll
            for (int b = 0; b < NB8; ++b) {
              acc[b][0] = fmaf(sc0, d[b][0], acc[b][0]);
              acc[b][1] = fmaf(sc0, d[b][1], acc[b][1]);
              acc[b][2] = fmaf(sc8, d[b][2], acc[b][2]);
              acc[b][3] = fmaf(sc8, d[b][3], acc[b][3]);
            }
            if (++grp < gp1) {
              sc0 = s_g[(size_t)grp * 64];
              sc8 = s_g8[(size_t)grp * 64];
            }
          }
        }
        __syncwarp();                              // every lane has read slot j
        if (sl + kQmPD < nslot) cp16(cdst + j * 512, csrc + (size_t)2 * (sl + kQmPD) * wb);
        cp_commit();
      }
    }
  }
  cp_wait<0>();

  // the two K parts, added in part order: red[kp][row][64 columns]
  __syncthreads();                                 // every warp is done with the planes
  float *red = reinterpret_cast<float *>(smq);
#pragma unroll
  for (int b = 0; b < NB8; ++b)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = b * 8 + 2 * t + (e & 1), col = mi * 16 + g + 8 * (e >> 1);
      red[((size_t)kp * MR8 + row) * 64 + col] = acc[b][e];
    }
  __syncthreads();
  const bool split = p.KS > 1;
  if (p.gate_up && !split) {
    // gate column c < 32 of the block and its up column c + 32: out[m][32 nb + c]
    for (int idx = threadIdx.x; idx < M * 32; idx += blockDim.x) {
      const int m = idx >> 5, c = idx & 31;
      const float g = red[(size_t)m * 64 + c] + red[((size_t)MR8 + m) * 64 + c];
      const float u = red[(size_t)m * 64 + 32 + c] + red[((size_t)MR8 + m) * 64 + 32 + c];
      store_out_rt(p.out, (size_t)m * (N / 2) + 32 * nb + c, silu_mul(g, u), p.out_f32 != 0);
    }
    return;
  }
  for (int idx = threadIdx.x; idx < M * 64; idx += blockDim.x) {
    const int m = idx >> 6, c = idx & 63, n = n0 + c;
    const float sum = red[(size_t)m * 64 + c] + red[((size_t)MR8 + m) * 64 + c];
    if (c < wb) {
      if (split)
        p.part[((size_t)ks * M + m) * N + n] = sum;
      else
        store_out_rt(p.out, (size_t)m * N + n, sum, p.out_f32 != 0);
    }
  }
  if (!split) return;
  if (!last_arriver(p.counters + nb, p.KS)) return;
  if (p.gate_up) {
    for (int idx = threadIdx.x; idx < M * 32; idx += blockDim.x) {
      const int m = idx >> 5, c = idx & 31;
      float g = 0.f, u = 0.f;
      for (int s2 = 0; s2 < p.KS; ++s2) {
        g += __ldcg(p.part + ((size_t)s2 * M + m) * N + n0 + c);
        u += __ldcg(p.part + ((size_t)s2 * M + m) * N + n0 + 32 + c);
      }
      store_out_rt(p.out, (size_t)m * (N / 2) + 32 * nb + c, silu_mul(g, u), p.out_f32 != 0);
    }
    return;
  }
  for (int idx = threadIdx.x; idx < M * 64; idx += blockDim.x) {
    const int m = idx >> 6, c = idx & 63, n = n0 + c;
    if (c >= wb) continue;
    float sum = 0.f;
    for (int s2 = 0; s2 < p.KS; ++s2) sum += __ldcg(p.part + ((size_t)s2 * M + m) * N + n);
    store_out_rt(p.out, (size_t)m * N + n, sum, p.out_f32 != 0);
  }
}

bool q8_mma_supported(int M, int K, int G, int prec) {
  return !(prec & GQ_W4) && (prec & GQ_ACT_F32) && (prec & GQ_SC_F32) && M >= 1 &&
         M <= kQmMaxM && G % kChunkK8 == 0 && K % G == 0;
}

size_t q8_mma_smem_bytes(int M, int K, int G, int KS) {
  return q8m_area_bytes(M, K, G, KS) + q8m_scale_bytes(K, G, KS) + (size_t)8 * kQmPD * 512;
}

// K slices: as for the CUDA-core kernel, counted against this kernel's shared memory and
// its two K parts per CTA.
int q8_mma_slices(int M, int K, int N, int G, int sms, size_t part_cap, int forced) {
  const int groups = K / G;
  const int nb = (N + 63) / 64;
  int best = 0, largest = 0;
  double best_cost = 0.0;
  for (int ks = 1; ks <= groups; ++ks) {
    if (ks > 1 && groups / ks < 2) break;          // both K parts keep a group
    if (ks > 1 && (size_t)ks * M * N * 4 > part_cap) break;
    if (q8_mma_smem_bytes(M, K, G, ks) > kQbSmemCap) continue;
    largest = ks;
    if (forced != 0) {
      if (forced == ks) return ks;
      continue;
    }
    if (M <= 8) return ks;
    const long waves = ((long)nb * ks + 2L * sms - 1) / (2L * sms);
    const double cost = (double)waves / ks * (1.0 + 0.05 * ks);
    if (best == 0 || cost < best_cost * (1.0 - 1e-9)) {
      best = ks;
      best_cost = cost;
    }
  }
  if (forced == -1) return largest;
  return forced != 0 ? 0 : best;
}

cudaError_t launch_q8_mma(const Plan &pl, int M, int K, int N, int G, int prec, const void *A,
                          const void *Wq, const void *scales, void *out, float *part,
                          unsigned *counters, cudaStream_t s) {
  QmParams qp;
  qp.Wp = reinterpret_cast<const uint4 *>(Wq);
  qp.A = reinterpret_cast<const float *>(A);
  qp.S = reinterpret_cast<const float *>(scales);
  qp.gate_up = (prec & GQ_GATE_UP) ? 1 : 0;
  qp.out = out;
  qp.part = part;
  qp.counters = counters;
  qp.M = M;
  qp.K = K;
  qp.N = N;
  qp.G = G;
  qp.KS = pl.nsplit;
  qp.NB = (N + 63) / 64;
  qp.out_f32 = (prec & GQ_OUT_F32) ? 1 : 0;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                         pl.smem_bytes);
    if (e != cudaSuccess) return e;
    kern<<<pl.grid_x, kQmThreads, pl.smem_bytes, s>>>(qp);
    return cudaGetLastError();
  };
  switch ((M + 7) / 8) {
    case 1: return go(q8_mma_kernel<1>);
    case 2: return go(q8_mma_kernel<2>);
    case 3: return go(q8_mma_kernel<3>);
    case 4: return go(q8_mma_kernel<4>);
    default: return cudaErrorInvalidValue;
  }
}

bool q8_block_supported(int M, int K, int G, int prec) {
  return !(prec & GQ_W4) && (prec & GQ_ACT_F32) && (prec & GQ_SC_F32) && M >= 1 &&
         M <= kQ8BlockMaxM && G % kChunkK8 == 0 && K % G == 0;
}

size_t q8_block_smem_bytes(int M, int K, int G, int KS) {
  return q8_block_area_bytes(M, K, G, KS) + (size_t)kQbWarps * q8_block_pd(M) * 1024;
}

int q8_block_cols() { return kQbCols; }
int q8_block_threads() { return kQbThreads; }

// K slices for NB column blocks on `sms` SMs, among the counts whose shared memory fits two
// CTAs per SM and whose partial sums stay within part_cap bytes, every warp of a split CTA
// keeping at least one group.  Up to 8 rows the kernel is bound by load latency, which every
// extra wave of CTAs pays again: the fewest slices that fit.  Above 8 rows it is bound by
// the FP32 pipes: the count with the least work per SM counted in waves of two CTAs per SM,
// each slice charged 5% for its partial sums and its CTAs' fixed costs (fewer on ties).
int q8_block_slices(int M, int K, int N, int G, int sms, size_t part_cap, int forced) {
  const int groups = K / G, rb = q8_rb(M), kp = kQbWarps / rb;
  const int nb = (N + kQbCols - 1) / kQbCols;
  int best = 0, largest = 0;
  double best_cost = 0.0;
  for (int ks = 1; ks <= groups; ++ks) {
    if (ks > 1 && groups / ks < kp) break;        // a CTA's warps would run out of groups
    if (ks > 1 && (size_t)ks * M * N * 4 > part_cap) break;
    if (q8_block_smem_bytes(M, K, G, ks) > kQbSmemCap) continue;
    largest = ks;
    if (forced != 0) {
      if (forced == ks) return ks;
      continue;
    }
    if (M <= 8) return ks;
    const long waves = ((long)nb * ks + 2L * sms - 1) / (2L * sms);
    const double cost = (double)waves / ks * (1.0 + 0.05 * ks);
    if (best == 0 || cost < best_cost * (1.0 - 1e-9)) {
      best = ks;
      best_cost = cost;
    }
  }
  if (forced == -1) return largest;
  return forced != 0 ? 0 : best;
}

cudaError_t launch_q8_block(const Plan &pl, int M, int K, int N, int G, int prec, const void *A,
                            const void *Wq, const void *scales, void *out, float *part,
                            unsigned *counters, cudaStream_t s) {
  QbParams qp;
  qp.Wp = reinterpret_cast<const uint4 *>(Wq);
  qp.A = reinterpret_cast<const float *>(A);
  qp.gate_up = (prec & GQ_GATE_UP) ? 1 : 0;
  qp.S = reinterpret_cast<const float *>(scales);
  qp.out = out;
  qp.part = part;
  qp.counters = counters;
  qp.M = M;
  qp.K = K;
  qp.N = N;
  qp.G = G;
  qp.KS = pl.nsplit;
  qp.NB = (N + kQbCols - 1) / kQbCols;
  qp.out_f32 = (prec & GQ_OUT_F32) ? 1 : 0;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                         pl.smem_bytes);
    if (e != cudaSuccess) return e;
    kern<<<pl.grid_x, kQbThreads, pl.smem_bytes, s>>>(qp);
    return cudaGetLastError();
  };
  const int rt = q8_rt(M);
  switch (rt) {
    case 1: return go(q8_block_kernel<1, 8>);
    case 2: return go(q8_block_kernel<2, 8>);
    case 4: return go(q8_block_kernel<4, 6>);
    case 8: return go(q8_block_kernel<8, 3>);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gq

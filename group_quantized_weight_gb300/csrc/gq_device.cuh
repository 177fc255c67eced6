// Device helpers shared by the small-M decode kernels (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gq_internal.h"

namespace gq {

// ------------------------------------------------------------------------------ helpers

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int SC>
__device__ __forceinline__ uint32_t ld_scale_bits(const void *s, size_t idx) {
  if (SC == kScF32) return __float_as_uint(__ldg(reinterpret_cast<const float *>(s) + idx));
  return (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(s) + idx);
}

template <int SC>
__device__ __forceinline__ float scale_value(uint32_t bits) {
  if (SC == kScF32) return __uint_as_float(bits);
  if (SC == kScBF16) return __uint_as_float(bits << 16);
  return __half2float(__ushort_as_half((unsigned short)bits));
}

// (w & 0x000F000F) | 0x43004300: the two codes become bf16(128 + q) in both halves
__device__ __forceinline__ uint32_t nib_pair(uint32_t w) {
  return (w & 0x000F000Fu) | 0x43004300u;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162 *>(&b);
  __nv_bfloat162 r = __hsub2(x, y);
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ void mma_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

template <bool OUTF32>
__device__ __forceinline__ void store_out(void *out, size_t idx, float v) {
  if (OUTF32)
    reinterpret_cast<float *>(out)[idx] = v;
  else
    reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ void zsplit_dev(int units, int nsplit, int z, int &ub, int &ue) {
  const int base = units / nsplit, rem = units % nsplit;
  ub = z * base + (z < rem ? z : rem);
  ue = ub + base + (z < rem ? 1 : 0);
}

// Called by every thread of the CTA after it wrote its split partials.  Returns true in
// the one CTA (per output tile) that arrives last; that CTA then owns the reduction.
__device__ __forceinline__ bool last_arriver(unsigned *counter, int nsplit) {
  __shared__ unsigned s_last;
  __threadfence();                 // make this thread's partials visible device-wide
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(counter, 1u);
    const bool last = (prev == (unsigned)(nsplit - 1));
    if (last) *counter = 0u;       // every other CTA of this tile has arrived: reset
    s_last = last ? 1u : 0u;
  }
  __syncthreads();
  const bool last = s_last != 0u;
  if (last) __threadfence();
  return last;
}

// Sum partials of rows [m0, m0+Mb) x columns [nb0, nb0+NT) in slice order, then store.
template <bool OUTF32>
__device__ __forceinline__ void reduce_tile(const float *part, void *out, int M, int N,
                                            int nsplit, int m0, int Mb, int nb0, int NT) {
  for (int idx = threadIdx.x; idx < Mb * NT; idx += blockDim.x) {
    const int m = m0 + idx / NT;
    const int n = nb0 + idx % NT;
    if (n >= N) continue;
    float s = 0.f;
    for (int z = 0; z < nsplit; ++z) s += __ldcg(part + ((size_t)z * M + m) * N + n);
    store_out<OUTF32>(out, (size_t)m * N + n, s);
  }
}


// runtime-typed scale access (fp16 / bf16 / fp32)
__device__ __forceinline__ uint32_t ld_scale_bits_rt(const void *s, size_t idx, int sc) {
  if (sc == kScF32) return __float_as_uint(__ldg(reinterpret_cast<const float *>(s) + idx));
  return (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(s) + idx);
}

__device__ __forceinline__ float scale_value_rt(uint32_t bits, int sc) {
  if (sc == kScF32) return __uint_as_float(bits);
  if (sc == kScBF16) return __uint_as_float(bits << 16);
  return __half2float(__ushort_as_half((unsigned short)bits));
}

__device__ __forceinline__ void store_out_rt(void *out, size_t idx, float v, bool f32) {
  if (f32)
    reinterpret_cast<float *>(out)[idx] = v;
  else
    reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

// ------------------------------------------------------------------ FP16 decode and MMA
// (the striped and warp-specialized small-M kernels)

__device__ __forceinline__ void mma_16816_f16(float d[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the same MMA with a zero accumulator input (the first step of a group)
__device__ __forceinline__ void mma_16816_f16_zc(float d[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
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

// (a & MASK) | c in one LOP3: the mask is an immediate of the instruction and c a register
// (with both constants taken from memory operands the compiler emits two instructions)
template <uint32_t MASK>
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "n"(MASK), "r"(c));
  return r;
}

// x * 2^e for e in [-174, 127], rounded once.  2^e is a normal float for e >= -126; below
// that, x is first scaled by 2^-64 (exact unless |x| < 2^-62, in which case the result is
// below 2^-188 and rounds to zero either way) and then by 2^(e + 64).
__device__ __forceinline__ float scale_pow2(float x, int e) {
  if (e >= -126) return x * __int_as_float((127 + e) << 23);
  return x * __int_as_float((127 - 64) << 23) * __int_as_float((127 + 64 + e) << 23);
}

// silu(g) * u = g / (1 + e^-g) * u in FP32 (CUDA's expf and IEEE division)
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Shared-memory image of the CTA's activation slice, permuted so that lane (m, q) gets
// the B operands of four consecutive 16-k MMA steps with two 16-byte loads:
//   word(m, chunk c, half h2, q, e) = A[m][kb + 64c + 16(2*h2 + e/2) + 8(e%2) + 2q .. +1]
// Rows are padded by 16 words so that two rows read in one phase hit different banks.
__host__ __device__ constexpr int act_row_words(int nchunks) { return nchunks * 32 + 16; }

}  // namespace gq

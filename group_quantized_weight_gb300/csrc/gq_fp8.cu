// FP8 W8A8 GEMM with 128 x 128 block scales ("GPU Kernel 工程（09）：量化与融合 kernel",
// section 四.3): activations and weights are FP8 E4M3, activations carry one scale per row
// and 128-k block, weights one per 128 x 128 block, and
//
//     out[m][n] = Σ_b a_scale[b][m] · w_scale[n / 128][b] · Σ_{k ∈ block b} A[m][k] · W[n][k].
//
// The scale of a block depends on k, so it cannot move to the epilogue: every 128-k block's
// tensor-core sum is multiplied by its two scales and added into FP32 running sums inside the
// K loop (the page's "promote").  Roles inside one persistent CTA per SM (20 warps):
//   warp 0          TMA producer: per 128-k block, the 128 x 128-byte weight tile and the
//                   256 x 128-byte activation tile (both 128-byte swizzle) into a 4-stage
//                   ring;
//   warp 1          TMEM allocator and MMA issuer: tcgen05.mma.cta_group::1.kind::f8f6f4,
//                   E4M3 x E4M3 -> FP32, M = 128 weight rows (n) x N = 256 activation rows (m)
//                   x K = 32, four per block, into one of two TMEM accumulators (one per block
//                   parity);
//   warps 2-3       idle (the weights need no dequantization);
//   warpgroups 1-4  promotion: warp (lane quarter q, column quarter c) reads its 32 TMEM
//                   lanes x 64 columns of a finished block, times a_scale · w_scale (one
//                   product per activation row, staged in shared memory; w_scale is one per
//                   tile and block), into 64 FP32 running sums per thread with paired FMAs;
//                   epilogue.
// Every mbarrier wait is bounded; a wait that gives up records GQ_ERR_TIMEOUT in a device
// error word, every role then leaves its loop, and TMEM is released before the CTA exits.
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>

#include "gq_internal.h"
#include "gq_tma_host.h"

namespace gq {

constexpr int kF8Stages = 4;                 // TMA ring depth (128-k blocks)
constexpr int kF8TileN = 128;                // weight rows per tile (TMEM lanes) = one block
constexpr int kF8TileM = 256;                // activation rows per tile (TMEM columns)
constexpr int kF8Block = 128;                // k per scale block
constexpr int kF8Threads = 640;              // 20 warps = 5 warpgroups
constexpr int kF8SumWarps = 16;              // warpgroups 1-4
constexpr uint32_t kF8WBytes = kF8TileN * kF8Block;          // 16 KB per stage
constexpr uint32_t kF8ABytes = kF8TileM * kF8Block;          // 32 KB per stage
constexpr uint32_t kF8StageBytes = kF8ABytes + kF8WBytes;    // 48 KB
// bounded waits: SM clock cycles before a wait gives up (about two seconds by default;
// gq_set_wait_limit changes it)
static __device__ long long g_f8_wait_limit = 4000000000ll;

static __device__ int g_fp8_error;           // sticky status (GQ_ERR_TIMEOUT), read by the host
static __device__ unsigned g_fp8_abort;      // token of the launch that gave up

namespace f8 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
// Bounded wait for phase `parity`: false once another role of this launch gave up, or after
// g_f8_wait_limit SM clock cycles, recording GQ_ERR_TIMEOUT and this launch's token.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned token) {
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 255u) == 0u) {
      if (*(volatile unsigned *)&g_fp8_abort == token) return false;
      if (clock64() - t0 > g_f8_wait_limit) {
        atomicExch(&g_fp8_abort, token);
        atomicExch(&g_fp8_error, GQ_ERR_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
  d |= (uint64_t)1 << 16;                          // leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset
  d |= (uint64_t)1 << 46;                          // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f8f6f4: FP32 accumulator (bit 4), A and B E4M3 (type code 0
// at bits 7 and 10), both K-major, N / 8 at bit 17, M / 16 at bit 24.
__host__ __device__ constexpr uint32_t idesc_e4m3(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float v[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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
// the 512 promotion threads (named barrier 1)
__device__ __forceinline__ void sum_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

}  // namespace f8

__global__ void __launch_bounds__(kF8Threads, 1)
fp8_block_gemm_kernel(const __grid_constant__ CUtensorMap map_w,
                      const __grid_constant__ CUtensorMap map_a,
                      const float *__restrict__ a_scales, const float *__restrict__ w_scales,
                      __nv_bfloat16 *__restrict__ out_bf16, float *__restrict__ out_f32,
                      int M, int K, int N, int out_f32_flag, unsigned token) {
  using namespace f8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kF8Stages], bar_empty[kF8Stages], bar_acc_full[2],
      bar_acc_empty[2];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(16) float s_ascale[2][kF8TileM];     // a_scale of the tile's rows, 2 blocks
  __shared__ int s_fail;                                     // a promotion thread's wait gave up
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  auto a_at = [&](int s) { return smem + (size_t)s * kF8StageBytes; };               // 32 KB
  auto w_at = [&](int s) { return smem + (size_t)s * kF8StageBytes + kF8ABytes; };   // 16 KB

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  const int nb = K / kF8Block;                     // k blocks
  const int tiles_n = (N + kF8TileN - 1) / kF8TileN;
  const int tiles_m = (M + kF8TileM - 1) / kF8TileM;
  const int tiles = tiles_n * tiles_m;

  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int s = 0; s < kF8Stages; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);       // the MMA's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_acc_full[b]), 1);
      mbar_init(smem_u32(&bar_acc_empty[b]), kF8SumWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {   // TMEM: two accumulators of 256 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = s_tmem;

  // Register budgets: the block is launched with 640 threads x 96 registers = 61,440 (the
  // launch bound's allocation, checked by the host before the launch), and setmaxnreg.inc
  // draws on that pool: roles 32 for warpgroup 0, promotion 112 for warpgroups 1-4:
  // 4,096 + 4 x 14,336 = 61,440.
  if (wg == 0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 32;" ::: "memory");
    if (warp == 0) {
      // -------------------------------------------------------------- TMA producer
      if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&map_w) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&map_a) : "memory");
        uint32_t i = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
          const int tn = tile % tiles_n, tm = tile / tiles_n;
          for (int kb = 0; kb < nb && ok; ++kb, ++i) {
            const int s = i % kF8Stages;
            ok = mbar_wait(smem_u32(&bar_empty[s]), ((i / kF8Stages) & 1) ^ 1, token);
            if (!ok) break;
            const uint32_t fb = smem_u32(&bar_full[s]);
            mbar_expect_tx(fb, kF8StageBytes);
            tma_load_2d(smem_u32(w_at(s)), &map_w, fb, kb * kF8Block, tn * kF8TileN);
            tma_load_2d(smem_u32(a_at(s)), &map_a, fb, kb * kF8Block, tm * kF8TileM);
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // -------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3(kF8TileN, kF8TileM);
        uint32_t i = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
          for (int kb = 0; kb < nb && ok; ++kb, ++i) {
            const int b = i & 1, s = i % kF8Stages;
            ok = mbar_wait(smem_u32(&bar_acc_empty[b]), ((i >> 1) & 1) ^ 1, token) &&
                 mbar_wait(smem_u32(&bar_full[s]), (i / kF8Stages) & 1, token);
            if (!ok) break;
            fence_after();
            // both operands K-major with 128-byte swizzle: 32 k = 32 bytes = 2 units
            const uint64_t da = desc_sw128(smem_u32(w_at(s)));
            const uint64_t db = desc_sw128(smem_u32(a_at(s)));
#pragma unroll
            for (int k = 0; k < kF8Block / 32; ++k)
              mma_e4m3(tmem + (uint32_t)b * kF8TileM, da + 2 * k, db + 2 * k, idesc,
                       k != 0 ? 1u : 0u);
            mma_commit(smem_u32(&bar_empty[s]));     // the stage is consumed
            mma_commit(smem_u32(&bar_acc_full[b]));  // the block's sum is in TMEM
          }
        }
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 112;" ::: "memory");
    // ---------------------------------------------------------------- promotion, epilogue
    const int wq = warp - 4;                       // 0..15
    const int lq = warp & 3;                       // TMEM lane quarter this warp may access
    const int cq = wq >> 2;                        // activation-row quarter of the tile
    const int row = lq * 32 + lane;                // TMEM lane = weight row within the tile
    const int st = threadIdx.x - 128;              // 0..511: threads below 256 stage row st
    const bool stager = st < kF8TileM;
    const bool odd = (lane & 1) != 0;
    float sum[64];
    uint32_t i = 0;
    bool ok = true;
    // the product a_scale[kb][m] · w_scale[tile][kb] of tile row st (the staging thread's
    // row) is staged in s_ascale[slot][st] one block ahead: a load issued a block early, one
    // multiply, one shared store
    auto load_ascale = [&](int tm, int kb) -> float {
      if (!stager) return 0.f;
      return __ldg(a_scales + (size_t)kb * M + min(tm * kF8TileM + st, M - 1));
    };
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      const int tn = tile % tiles_n, tm = tile / tiles_n;
#pragma unroll
      for (int c = 0; c < 64; ++c) sum[c] = 0.f;
      float as_next = load_ascale(tm, 0), ws_next = __ldg(w_scales + (size_t)tn * nb);
      for (int kb = 0; kb < nb; ++kb, ++i) {
        const int b = i & 1;
        if (stager) s_ascale[b][st] = as_next * ws_next;   // the block's scale of row st
        if (kb + 1 < nb) {                         // one block ahead
          as_next = load_ascale(tm, kb + 1);
          ws_next = __ldg(w_scales + (size_t)tn * nb + kb + 1);
        }
        // the block's sum is in TMEM (one lane per warp polls); the decision to give up is
        // taken by all 512 promotion threads together (all of them reach the named barrier)
        bool got = true;
        if (lane == 0) got = mbar_wait(smem_u32(&bar_acc_full[b]), (i >> 1) & 1, token);
        got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        if (!got && lane == 0) s_fail = 1;
        sum_sync();                                // scales of block kb stored; s_fail seen
        ok = *(volatile int *)&s_fail == 0;
        if (!ok) break;
        fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)b * kF8TileM +
                               (uint32_t)cq * 64;
        const float *sc = &s_ascale[b][cq * 64];
        // two 32-column TMEM loads, each waited for, then the scales from shared memory (four
        // 16-column loads with the scale reads in their shadow measured 1.6% slower: four
        // load latencies in series)
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          float v[32];
          tmem_ld32(taddr + c2 * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 s4 = *reinterpret_cast<const float4 *>(sc + c2 * 32 + 4 * q);
            float *z = &sum[c2 * 32 + 4 * q];
            fma2(z[0], z[1], s4.x, s4.y, v[4 * q], v[4 * q + 1]);
            fma2(z[2], z[3], s4.z, s4.w, v[4 * q + 2], v[4 * q + 3]);
          }
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_acc_empty[b]));
        // s_ascale[b] is refilled two blocks later, by a thread that has passed the next
        // block's barrier, which every reader of this block reaches only after these reads
      }
      if (!ok) break;
      // output column n = tn * 128 + row, rows m = tm * 256 + cq * 64 + c; lanes pair up
      // (lane, lane ^ 1) to store two adjacent columns (N is even)
      const int n = tn * kF8TileN + row;
      const int mb = tm * kF8TileM + cq * 64;
      const int ncol0 = n - (odd ? 1 : 0);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float mine_keep = odd ? sum[c + 1] : sum[c];
        const float mine_send = odd ? sum[c] : sum[c + 1];
        const float other = __shfl_xor_sync(0xffffffffu, mine_send, 1);
        const float lo = odd ? other : mine_keep, hi = odd ? mine_keep : other;
        const int m = mb + c + (odd ? 1 : 0);
        if (m < M && ncol0 < N) {
          if (out_f32_flag)
            *reinterpret_cast<float2 *>(out_f32 + (size_t)m * N + ncol0) = make_float2(lo, hi);
          else
            *reinterpret_cast<__nv_bfloat162 *>(out_bf16 + (size_t)m * N + ncol0) =
                __floats2bfloat162_rn(lo, hi);
        }
      }
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

// ------------------------------------------------------------------ activation quantizer

// Dynamic FP8 quantization of activations ("量化与融合 kernel" section 四.5, with 1 x 128
// blocks): scale = max_{k in block} |x| / 448 (binary32 division), code = E4M3(x / scale)
// (binary32 division, then the hardware's round-to-nearest-even conversion with saturation
// to ±448); a block of zeros gets scale 0 and codes 0.  One warp per (row, block): lane l
// holds k = 4l .. 4l + 3.
template <bool F32>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const void *__restrict__ A,
                                                           uint8_t *__restrict__ Aq,
                                                           float *__restrict__ scales, int M,
                                                           int K) {
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int nb = K / kF8Block;
  if (wid >= (long long)M * nb) return;
  const int m = (int)(wid / nb), b = (int)(wid - (long long)m * nb);
  const size_t base = (size_t)m * K + (size_t)b * kF8Block + 4 * lane;
  float x[4];
  if (F32) {
    const float4 v = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(A) + base);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2 *>(reinterpret_cast<const unsigned short *>(A) + base);
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xFFFF0000u);
  }
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 448.f);
  uint32_t word = 0;
  if (s > 0.f) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(__fdiv_rn(x[1], s)), "f"(__fdiv_rn(x[0], s)));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(__fdiv_rn(x[3], s)), "f"(__fdiv_rn(x[2], s)));
    word = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  *reinterpret_cast<uint32_t *>(Aq + base) = word;
  if (lane == 0) scales[(size_t)b * M + m] = s;   // [K/128][M], the GEMM's layout
}

int launch_quantize_fp8(int M, int K, bool f32, const void *A, void *Aq, void *scales,
                        cudaStream_t s) {
  const long long warps = (long long)M * (K / kF8Block);
  const long long blocks = (warps + 7) / 8;
  if (blocks > 0x7FFFFFFFll) return GQ_ERR_INVALID_ARG;
  if (f32)
    quantize_fp8_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(A, (uint8_t *)Aq, (float *)scales, M, K);
  else
    quantize_fp8_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(A, (uint8_t *)Aq, (float *)scales, M, K);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    note_cuda_error("launch(fp8 quantizer)", e);
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

// ------------------------------------------------------------------ host side

// rows x K bytes, K contiguous: boxes of 128 k x box_rows rows, 128-byte swizzle
static int f8_encode(CUtensorMap *map, const void *base, int rows, int K, int box_rows,
                     const char *what) {
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) {
    note_cuda_error_code("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", -1);
    return GQ_ERR_CUDA;
  }
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t str[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {(cuuint32_t)kF8Block, (cuuint32_t)box_rows};
  const cuuint32_t ones[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                         str, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    note_cuda_error_code(what, (int)r);
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

static unsigned f8_next_token() {
  static std::atomic<unsigned> t{0};
  return t.fetch_add(1u) + 1u;
}

size_t fp8_smem_bytes() { return (size_t)kF8Stages * kF8StageBytes + 1024; }

int fp8_block_plan(int M, int N, int sms, int *grid) {
  const int tiles = ((N + kF8TileN - 1) / kF8TileN) * ((M + kF8TileM - 1) / kF8TileM);
  *grid = tiles < sms ? tiles : sms;
  return GQ_OK;
}

int launch_fp8_block(int M, int K, int N, int prec, const void *A, const void *a_scales,
                     const void *W, const void *w_scales, void *out, int grid, cudaStream_t s) {
  CUtensorMap mw, ma;
  int st = f8_encode(&mw, W, N, K, kF8TileN, "cuTensorMapEncodeTiled(fp8 weights)");
  if (st != GQ_OK) return st;
  st = f8_encode(&ma, A, M, K, kF8TileM, "cuTensorMapEncodeTiled(fp8 activations)");
  if (st != GQ_OK) return st;
  const size_t smem = fp8_smem_bytes();
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(fp8_block_gemm_kernel), smem);
  if (e != cudaSuccess) {
    note_cuda_error("cudaFuncSetAttribute(fp8 shared memory)", e);
    return GQ_ERR_CUDA;
  }
  // the setmaxnreg split inside the kernel adds up to 640 threads x 96 registers: a build
  // whose launch allocation differs would make setmaxnreg.inc wait, so it is refused here
  static int regs = -1;
  if (regs < 0) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, fp8_block_gemm_kernel) != cudaSuccess) {
      cudaGetLastError();
      return GQ_ERR_CUDA;
    }
    regs = fa.numRegs;
  }
  if (regs != 96) {
    note_cuda_error_code("fp8 kernel register allocation (expected 96)", regs);
    return GQ_ERR_CUDA;
  }
  const bool f32 = (prec & GQ_OUT_F32) != 0;
  fp8_block_gemm_kernel<<<grid, kF8Threads, smem, s>>>(
      mw, ma, reinterpret_cast<const float *>(a_scales), reinterpret_cast<const float *>(w_scales),
      f32 ? nullptr : reinterpret_cast<__nv_bfloat16 *>(out),
      f32 ? reinterpret_cast<float *>(out) : nullptr, M, K, N, f32 ? 1 : 0, f8_next_token());
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    note_cuda_error("launch(fp8)", e);
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

int fp8_set_wait_limit(long long cycles) {
  return cudaMemcpyToSymbol(g_f8_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? 0 : -1;
}

int fp8_read_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fp8_error, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(g_fp8_error, &z, sizeof(int));
  }
  return v;
}

}  // namespace gq

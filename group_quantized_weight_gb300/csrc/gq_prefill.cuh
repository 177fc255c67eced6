// Large-M ("prefill") kernel of the group-quantized weight-only GEMM: TMA + tcgen05 + TMEM.
//
// Where the path is a dense contraction ("GPU Kernel 工程（09）：量化与融合 kernel", section 3.2:
// at prefill both BF16 and INT4 GEMMs are compute-bound), the dequantized weights feed the
// 5th-generation tensor cores.  Roles inside one persistent CTA per SM (16 warps):
//   warps 0, 2, 3 TMA producers, taking the stages in turn: per 64-k stage, the packed codes
//                 of a 128-column tile (one 3-D box of 8 x 512 bytes) and the BM x 64 bf16
//                 activation tile (BM = 64, 128 or 256 rows, 128-byte swizzle) into a ring
//                 of up to 12 stages.
//   warp 1        TMEM allocator and MMA issuer: tcgen05.mma.cta_group::1.kind::f16,
//                 M = 128 (weight columns n) x N = BM (activation rows m) x K = 16, BF16 x
//                 BF16 -> FP32, into one of two TMEM accumulators (one per group parity).
//   warpgroup 1   dequantization of stage i's codes into operand buffer i mod 4 (K-major,
//                 exact bf16 integers q - z): by warp i mod 4 (up to four stages at once),
//                 or with 256-row tiles by a pair of warps (two stages at once, each faster).
//   warpgroups 2-3  promotion: tcgen05.ld of a finished group, times its scale (one per
//                 thread: a TMEM lane is one column n), into FP32 running sums; epilogue.
// The operand tiles hold the exact integers q - z (bf16 represents |q - z| <= 15 exactly);
// each group's FP32 result is multiplied by its scale after the whole group, as the
// group-wise GEMM of "04 · 分组量化 GEMM 内核", section 2 requires.  Rounding s * (q - z) to
// bf16 inside the operand would change the result by far more than the output's rounding.
//
// Every mbarrier wait is bounded; a wait that gives up records GQ_ERR_TIMEOUT in a device
// error word, every role then leaves its loop, and TMEM is released before the CTA exits.
//
// Two translation units instantiate the kernel: gq_prefill.cu with the tile height, ring depth
// and K split read at run time, gq_prefill_fixed.cu with them fixed at compile time for the
// large-M shape (256-row tiles, a four-deep ring, no split), where the constants make the
// role loops several percent faster.  Each keeps its own error word and wait limit.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gq_device.cuh"

namespace gq {

constexpr int kPfMaxStages = 12;             // TMA ring depth (64-k stages), at most
static_assert(kPfMaxStages <= 32, "one initialising thread per stage in a warp");
constexpr int kPfDqBufs = 4;                 // dequantized-operand buffers
constexpr int kPfDqWarps = 4;                // warpgroup 1
static_assert(kPfDqWarps == kPfDqBufs, "one warp per stage: warp d fills operand buffer d");
constexpr int kPfProducers = 3;              // TMA-issuing warps (0, 2 and 3)
// ring depth at least: the producers' and the dequant warps' waits rely on it (see the roles)
constexpr int kPfMinStages = kPfDqBufs > kPfProducers ? kPfDqBufs : kPfProducers;
constexpr int kPfTileN = 128;                // weight columns per tile (TMEM lanes)
constexpr int kPfMaxTileM = 256;             // activation rows per tile (TMEM columns), at most
static_assert(2 * kPfMaxTileM <= 512, "two accumulators of the tallest tile fill TMEM");
constexpr int kPfThreads = 512;              // 16 warps = 4 warpgroups
constexpr int kPfSumWarps = 8;               // warpgroups 2 and 3
constexpr uint32_t kPfPackedBytes = 8 * 512;                  // packed codes per stage
constexpr uint32_t kPfDqBytes = kPfTileN * 64 * 2;            // dequantized weights per stage
// one TMA stage: the BM x 64 bf16 activation box, then the 128 x 64 packed codes
__host__ __device__ constexpr uint32_t pf_stage_bytes(int BM) { return (uint32_t)BM * 128 + kPfPackedBytes; }
// bounded waits: SM clock cycles before a wait gives up (about two seconds by default;
// gq_set_wait_limit changes it)
// (one copy per translation unit, like the error word below)
static __device__ long long g_pf_wait_limit = 4000000000ll;

static __device__ int g_prefill_error;        // sticky status (GQ_ERR_TIMEOUT), read by the host
static __device__ unsigned g_prefill_abort;     // token of the launch that gave up

// the compile-time shape of the FIXED = 1 instances
constexpr int kPfFixedTileM = 256;
constexpr int kPfFixedStages = 4;

// ------------------------------------------------------------------ PTX wrappers

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

// Wait for the phase of parity `parity` to complete.  Bounded: gives up (false) once another
// role of the same launch gave up, or after g_pf_wait_limit SM clock cycles (about two
// seconds), recording GQ_ERR_TIMEOUT (sticky) and this launch's token.
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
      if (*(volatile unsigned *)&g_prefill_abort == token) return false;   // this launch gave up
      if (clock64() - t0 > g_pf_wait_limit) {
        atomicExch(&g_prefill_abort, token);
        atomicExch(&g_prefill_error, GQ_ERR_TIMEOUT);
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

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// UMMA shared-memory descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B
// apart (stride byte offset), leading byte offset unused for swizzled K-major (1).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
  d |= (uint64_t)1 << 16;                          // leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset
  d |= (uint64_t)1 << 46;                          // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}

// UMMA shared-memory descriptor: K-major operand without swizzle, made of 8-row x 16-byte
// core matrices; `lbo` = bytes between core matrices adjacent in K, `sbo` = bytes between
// 8-row groups.
__device__ __forceinline__ uint64_t umma_desc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;                          // descriptor version; swizzle field 0 = none
  return d;
}

// Instruction descriptor, kind::f16: FP32 accumulator, BF16 A and B, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// 32 consecutive TMEM columns of this thread's lane
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

// 16 consecutive TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// (a & 0x000F000F) | c in one LOP3: the mask is an immediate of the instruction and c a
// register (with both constants taken from memory operands the compiler emits two)
__device__ __forceinline__ uint32_t lo_nibbles(uint32_t a, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(r) : "r"(a), "r"(c));
  return r;
}

// two FP32 FMAs in one instruction: (x0, x1) * (y, y) + (z0, z1)
__device__ __forceinline__ void ffma2_bcast(float &z0, float &z1, float x0, float x1, float y) {
  asm("{\n\t.reg .b64 a, b, c;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %4};\n\tmov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 c, a, b, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "+f"(z0), "+f"(z1)
      : "f"(x0), "f"(x1), "f"(y));
}

__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

struct PrefillConsts {
  uint32_t magic;     // 0x43004300: bf16 128 in both halves
  uint32_t sym;       // 0x43084308: bf16 (128 + 8)
};

// Tile height, ring depth and K split of a launch.
struct PrefillShape {
  int BM;             // activation rows per tile: 64, 128 or 256 (the MMA's N, TMEM columns)
  int S;              // TMA ring stages
  int KS;             // K slices of whole groups (1 = no split)
  float *part;        // [KS][M][N] FP32 slice partial sums (KS > 1)
  unsigned *counters; // [tiles][8] arrival counters, one per promotion warp's part of a tile
};

// The groups of a work unit (g0 .. g1 - 1) are visited starting at a rotation that depends
// on the tile's column index: the CTAs working on one row block of activations then read
// different 64-k boxes of it at any moment, instead of all of them the same box (an L2 hot
// spot that held every CTA to one stage per half microsecond).  The i-th group visited:
__device__ __forceinline__ int pf_group(int g0, int g1, int tn, int i) {
  const int n = g1 - g0;
  int g = g0 + i + (tn * 5) % n;
  return g >= g1 ? g - n : g;
}

// ------------------------------------------------------------------ the kernel

template <int SPG, int SC, bool ZP, int FIXED>
__global__ void __launch_bounds__(kPfThreads, 1)
w4_prefill_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_a,
                  const void *__restrict__ scales, const uint32_t *__restrict__ zeros,
                  __nv_bfloat16 *__restrict__ out_bf16, float *__restrict__ out_f32,
                  int M, int K, int N, int out_f32_flag, const PrefillConsts pc,
                  const PrefillShape sh, unsigned token) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kPfMaxStages], bar_empty[kPfMaxStages],
      bar_dq[kPfDqBufs], bar_acc_full[2], bar_acc_empty[2];
  __shared__ uint32_t s_tmem;
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // TMA stage s: [activations BM x 128 bytes][packed codes 4 KB] (a multiple of 1 KB, as the
  // 128-byte swizzle wants); then kPfDqBufs dequantized operand buffers of 16 KB
  // FIXED = 1: 256-row tiles, a four-deep ring, no K split, as constants
  constexpr bool kFixed = FIXED != 0;
  const int BM = kFixed ? kPfFixedTileM : sh.BM;
  const int S = kFixed ? kPfFixedStages : sh.S;
  const int KS = kFixed ? 1 : sh.KS;
  // dequant warps per stage: a pair with 256-row tiles (whose four-deep ring needs the shorter
  // latency), one otherwise (64- and 128-row tiles have deep rings and fewer waits win)
  constexpr int kDqPerStage = kFixed ? 2 : 1;
  const uint32_t stage_bytes = pf_stage_bytes(BM), act_bytes = (uint32_t)BM * 128;
  auto act_at = [&](int s) { return smem + (size_t)s * stage_bytes; };
  auto pk_at = [&](int s) { return smem + (size_t)s * stage_bytes + act_bytes; };
  auto dq_at = [&](int d) { return smem + (size_t)S * stage_bytes + (size_t)d * kPfDqBytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wg = warp >> 2;                        // warpgroup: role and register budget
  const int ng = K / (SPG * 64);                   // groups (K / G)
  const int tiles_n = (N + kPfTileN - 1) / kPfTileN;
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles = tiles_n * tiles_m;
  // work units: (tile, K slice) pairs, tile fastest; slice z covers groups zsplit(ng, KS, z)
  const int units = tiles * KS;

  // barrier initialisation spread over the dequant warpgroup's threads (one thread doing all
  // of them delays every role's start), each fencing its own
  {
    const int t = (int)threadIdx.x - 128;          // warpgroup 1
    bool did = false;
    if (t >= 0 && t < S) {
      mbar_init(smem_u32(&bar_full[t]), 1);
      // a stage is free once the MMA read its activations and the dequantized operand made
      // from it (commit) and its dequant warps read its codes
      mbar_init(smem_u32(&bar_empty[t]), 1 + kDqPerStage);
      did = true;
    } else if (t >= 32 && t < 32 + kPfDqBufs) {
      mbar_init(smem_u32(&bar_dq[t - 32]), kDqPerStage);  // the stage's dequant warps
      did = true;
    } else if (t >= 64 && t < 66) {
      mbar_init(smem_u32(&bar_acc_full[t - 64]), 1);
      mbar_init(smem_u32(&bar_acc_empty[t - 64]), kPfSumWarps);  // one per promotion warp
      did = true;
    }
    if (did) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {   // TMEM: two accumulators of 256 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // Register budgets per warpgroup (launched with kPfThreads x 128 = 65,536): roles 56,
  // dequantization 88, promotion 176 each for two warpgroups; 7,168 + 11,264 + 2 x 22,528 =
  // 63,488 registers in total, within the launch's 65,536.
  if (wg == 0) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
   if (warp != 1) {
    // ---------------------------------------------------------------- TMA producers
    // Warps 0, 2 and 3 take the stages in turn (stage i: warp i mod 3).  One issuing thread
    // gets about one stage per memory round trip on this GPU whatever the ring depth, so the
    // stages of one ring are spread over three.  A producer's successive stages are three
    // apart and the ring is at least three deep, so the empty barrier it waits on is never
    // more than one phase behind the phase it waits for.
    if (lane == 0) {
      const int pid = warp == 0 ? 0 : warp - 1;
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_w) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_a) : "memory");
      uint32_t i = 0;                                // stage number within this CTA
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int tile = u % tiles, z = u / tiles;
        const int tn = tile % tiles_n, tm = tile / tiles_n;
        int g0, g1;
        zsplit_dev(ng, KS, z, g0, g1);
        const int nk = (g1 - g0) * SPG;
        for (int kk = 0; kk < nk && ok; ++kk, ++i) {
          if (i % kPfProducers != (uint32_t)pid) continue;
          const int s = (int)(i % (uint32_t)S);
          ok = mbar_wait(smem_u32(&bar_empty[s]), ((i / (uint32_t)S) & 1u) ^ 1u, token);
          if (!ok) break;
          const int kc = pf_group(g0, g1, tn, kk / SPG) * SPG + kk % SPG;
          const uint32_t fb = smem_u32(&bar_full[s]);
          mbar_expect_tx(fb, stage_bytes);
          tma_load_3d(smem_u32(pk_at(s)), &map_w, fb, 0, kc, tn * 8);
          tma_load_2d(smem_u32(act_at(s)), &map_a, fb, kc * 64, tm * BM);
        }
      }
    }
    __syncwarp();
   } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // Per stage one wait (the dequantized operand; its warp saw the stage's copies land, so
    // the activations are there too), four MMAs and one commit, which frees both the stage
    // and the operand buffer: each of these costs the single issuing thread 60 to 150 cycles,
    // as much as a 64-row stage's MMAs take.
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kPfTileN, BM);
      uint32_t i = 0, gg = 0;
      int s = 0;                                     // ring stage
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        int g0, g1;
        zsplit_dev(ng, KS, u / tiles, g0, g1);
        for (int g = g0; g < g1 && ok; ++g, ++gg) {
          const int b = gg & 1;
          ok = mbar_wait(smem_u32(&bar_acc_empty[b]), ((gg >> 1) & 1) ^ 1, token);
          if (!ok) break;
          tc_fence_after();
          for (int st = 0; st < SPG; ++st, ++i, s = s + 1 == S ? 0 : s + 1) {
            const int dbuf = i % kPfDqBufs;
            ok = mbar_wait(smem_u32(&bar_dq[dbuf]), (i / kPfDqBufs) & 1, token);
            if (!ok) break;
            tc_fence_after();

            // weights: core matrices, 16 k = two of them = 256 bytes = 16 descriptor units;
            // activations: 128-byte swizzle, 16 k = 32 bytes = 2 descriptor units
            const uint64_t da = umma_desc_plain(smem_u32(dq_at(dbuf)), 128, 1024);
            const uint64_t db = umma_desc_sw128(smem_u32(act_at(s)));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_bf16(tmem + (uint32_t)b * BM, da + 16 * k, db + 2 * k, idesc,
                        (st | k) != 0 ? 1u : 0u);
            umma_commit(smem_u32(&bar_empty[s]));        // stage and operand buffer consumed
          }
          if (!ok) break;
          umma_commit(smem_u32(&bar_acc_full[b]));       // group finished
        }
      }
    }
    __syncwarp();
   }
  } else if (wg == 1) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    // ---------------------------------------------------------------- dequantization
    // Warp d of the warpgroup owns 16-column sub-tiles 2d and 2d + 1 of every stage; lane
    // `lane` holds the 16-byte fragment of each: rows r0 = lane / 4 and r0 + 8 of the
    // sub-tile, k = 16j + 2(lane % 4) + 8h + {0,1}.  The dequantized operand is K-major core
    // matrices (8 rows x 16 bytes), core matrix (8-row group rg, 8-k group kg) at
    // rg * 1024 + kg * 128; pair p of word j of a fragment is core matrix
    // (2 sub + (p & 1), 2j + (p >> 1)), byte 16 r0 + 4 (lane % 4) = 4 lane inside it.
    // Stage i goes to operand buffer i mod 4, last read by the MMA of stage i - 4, whose
    // commit completed that stage's empty barrier (the ring is at least four deep, so that
    // barrier is never more than one phase away from the phase waited for).
    // Stage i goes to operand buffer i mod 4.  With 64- and 128-row tiles warp i mod 4
    // dequantizes it whole, so that each warp's two waits per stage cover a whole stage of
    // work (four warps sharing every stage measured slower: their waits, not the conversion,
    // set the pace); with 256-row tiles, whose ring is only four stages deep, the pair of
    // warps 2 (i mod 2) and 2 (i mod 2) + 1 takes half of it each, halving the stage's
    // latency (M=4096: 401 -> 355 us; with 64-row tiles the pair was slower, 31 -> 38 us).
    // Either way the buffer-reuse wait below (the MMA of stage i - 4) implies that stage
    // i - S was consumed, so the stage's full barrier is at most one phase behind.  Lane `lane` of
    // sub-tile u (columns 16u .. 16u + 15 of the tile) holds the 16-byte fragment: rows
    // r0 = lane / 4 and r0 + 8 of the sub-tile, k = 16j + 2(lane % 4) + 8h + {0,1}.  The
    // dequantized operand is K-major core matrices (8 rows x 16 bytes), core matrix (8-row
    // group rg, 8-k group kg) at rg * 1024 + kg * 128; pair p of word j of a fragment is core
    // matrix (2u + (p & 1), 2j + (p >> 1)), byte 16 r0 + 4 (lane % 4) = 4 lane inside it.
    const int d = warp & 3;
    const int r0 = lane >> 2;
    const int NW = N >> 3;
    uint32_t i = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int tn = (u % tiles) % tiles_n;
      int g0, g1;
      zsplit_dev(ng, KS, u / tiles, g0, g1);
      for (int gi = 0; gi < g1 - g0 && ok; ++gi) {
        const int g = pf_group(g0, g1, tn, gi);
        for (int st = 0; st < SPG; ++st, ++i) {
          // one warp per stage: stage i is warp i mod 4's; a pair: warps 2 (i mod 2) and
          // 2 (i mod 2) + 1, each with half of the stage's sub-tiles
          if ((int)(i % (kPfDqWarps / kDqPerStage)) != d / kDqPerStage) continue;
          const int s = (int)(i % (uint32_t)S);
          // the buffer was last read by the MMA of stage i - 4, whose commit completed that
          // stage's empty barrier; the ring is at least four deep, so that barrier is never
          // more than one phase away from the phase waited for
          const uint32_t pi = i - kPfDqBufs;
          ok = (i < (uint32_t)kPfDqBufs ||
                mbar_wait(smem_u32(&bar_empty[pi % (uint32_t)S]), (pi / (uint32_t)S) & 1, token)) &&
               mbar_wait(smem_u32(&bar_full[s]), (i / (uint32_t)S) & 1, token);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          const int dbuf = (int)(i % kPfDqBufs);
          uint8_t *dqb = dq_at(dbuf);
          // (with zero points the loop is kept rolled: fully unrolled, their loads are all
          // hoisted and spill)
          constexpr int kSubs = 8 / kDqPerStage;       // 16-column sub-tiles per warp
          const int sub0 = (d % kDqPerStage) * kSubs;
#pragma unroll (ZP ? 1 : kSubs)
          for (int su = 0; su < kSubs; ++su) {
            const int sub = sub0 + su;
            uint32_t zl = pc.sym, zh = pc.sym;
            if (ZP) {
              const int n = tn * kPfTileN + sub * 16 + r0;
              const uint32_t wa = __ldg(zeros + (size_t)g * NW + min(n >> 3, NW - 1));
              const uint32_t wb = __ldg(zeros + (size_t)g * NW + min((n + 8) >> 3, NW - 1));
              zl = (0x4300u | ((wa >> (4 * (n & 7))) & 0xFu)) * 0x00010001u;
              zh = (0x4300u | ((wb >> (4 * ((n + 8) & 7))) & 0xFu)) * 0x00010001u;
            }
            const uint4 f = *reinterpret_cast<const uint4 *>(pk_at(s) + sub * 512 + lane * 16);
            const uint32_t words[4] = {f.x, f.y, f.z, f.w};
            uint8_t *dq = dqb + sub * 2048 + lane * 4;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
              for (int p = 0; p < 4; ++p) {        // pair p: bits 4p and 4p + 16
                const uint32_t v = bsub2(lo_nibbles(words[j] >> (4 * p), pc.magic),
                                         (p & 1) ? zh : zl);
                *reinterpret_cast<uint32_t *>(dq + (p & 1) * 1024 + (2 * j + (p >> 1)) * 128) = v;
              }
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic -> tensor core
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&bar_dq[dbuf]));
            mbar_arrive(smem_u32(&bar_empty[s]));          // this warp is done with the codes
          }
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 176;" ::: "memory");
    // ---------------------------------------------------------------- promotion, epilogue
    const int wq = warp - 8;                       // 0..7
    const int lq = warp & 3;                       // TMEM lane quarter this warp may access
    const int half = wq >> 2;                      // activation-row half of the tile
    const int row = lq * 32 + lane;                // TMEM lane = weight column within the tile
    const bool odd = (lane & 1) != 0;
    auto load_scale = [&](int ncol, int g) -> float {
      if (SC == kScF32)
        return __ldg(reinterpret_cast<const float *>(scales) + (size_t)g * N + ncol);
      if (SC == kScBF16)
        return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(scales) +
                                               (size_t)g * N + ncol)
                               << 16);
      return __half2float(__ushort_as_half(
          __ldg(reinterpret_cast<const unsigned short *>(scales) + (size_t)g * N + ncol)));
    };
    float sum[128];
    uint32_t gg = 0;
    bool ok = true;
    const int hb = BM / 2;                         // activation rows of this warp's half
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int tile = u % tiles, z = u / tiles;
      const int tn = tile % tiles_n, tm = tile / tiles_n;
      int g0, g1;
      zsplit_dev(ng, KS, z, g0, g1);
      const int ncol = min(tn * kPfTileN + row, N - 1);
#pragma unroll
      for (int c = 0; c < 128; ++c) sum[c] = 0.f;
      // the group scales, four groups ahead of their use: a group's MMAs take only a few
      // hundred cycles with 64- and 128-row tiles, less than a load's latency
      const int ngu = g1 - g0;
      float sc1 = load_scale(ncol, pf_group(g0, g1, tn, 0));
      float sc2 = 1 < ngu ? load_scale(ncol, pf_group(g0, g1, tn, 1)) : 0.f;
      float sc3 = 2 < ngu ? load_scale(ncol, pf_group(g0, g1, tn, 2)) : 0.f;
      float sc4 = 3 < ngu ? load_scale(ncol, pf_group(g0, g1, tn, 3)) : 0.f;
      for (int gi = 0; gi < ngu; ++gi, ++gg) {
        const float sc = sc1;
        sc1 = sc2;
        sc2 = sc3;
        sc3 = sc4;
        if (gi + 4 < ngu) sc4 = load_scale(ncol, pf_group(g0, g1, tn, gi + 4));
        const int b = gg & 1;
        ok = mbar_wait(smem_u32(&bar_acc_full[b]), (gg >> 1) & 1, token);
        ok = __all_sync(0xffffffffu, ok);         // tcgen05.ld below is warp-collective
        if (!ok) break;
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)b * BM +
                               (uint32_t)half * hb;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          if (c4 * 32 < hb) {                       // BM / 64 loads of 32 columns
            float v[32];
            tmem_ld32(taddr + c4 * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; c += 2)
              ffma2_bcast(sum[c4 * 32 + c], sum[c4 * 32 + c + 1], v[c], v[c + 1], sc);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_acc_empty[b]));
      }
      if (!ok) break;
      const int n = tn * kPfTileN + row;
      const int mb = tm * BM + half * hb;
      if (KS > 1) {
        // K split: publish this slice's partial sums of the warp's part of the tile (32
        // columns x BM / 2 rows); the warp that adds the last of the KS slices to the part's
        // counter sums them in slice order 0, 1, ... (the same order whichever arrives last)
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int m = mb + c;
          if (c < hb && m < M && n < N) __stcg(sh.part + ((size_t)z * M + m) * N + n, sum[c]);
        }
        __threadfence();
        __syncwarp();
        unsigned last = 0u;
        if (lane == 0) {
          unsigned *ctr = sh.counters + (size_t)tile * kPfSumWarps + wq;
          last = atomicAdd(ctr, 1u) == (unsigned)(KS - 1) ? 1u : 0u;
          if (last) *ctr = 0u;                      // every slice has arrived: reset
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) continue;
        __threadfence();
        // every slice's partial, this warp's own included, read back in slice order
#pragma unroll
        for (int c = 0; c < 128; ++c) sum[c] = 0.f;
        for (int z2 = 0; z2 < KS; ++z2) {
          const float *pz = sh.part + (size_t)z2 * M * N + n;
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int m = mb + c;
            if (c < hb && m < M && n < N) sum[c] += __ldcg(pz + (size_t)m * N);
          }
        }
      }
      // the tile's output: column n = tn * 128 + row, rows m = tm * BM + half * BM / 2 + c.
      // Lanes pair up (lane, lane ^ 1) to write two adjacent columns per store: for rows
      // (m, m + 1) the even lane writes row m, columns (n, n + 1), the odd lane row m + 1,
      // columns (n - 1, n).  N is even, so both columns of a pair are in or out of range.
      const int ncol0 = n - (odd ? 1 : 0);
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        if (c < hb) {
          const float mine_keep = odd ? sum[c + 1] : sum[c];
          const float mine_send = odd ? sum[c] : sum[c + 1];
          const float other = __shfl_xor_sync(0xffffffffu, mine_send, 1);
          const float lo = odd ? other : mine_keep, hi = odd ? mine_keep : other;
          const int m = mb + c + (odd ? 1 : 0);
          if (m < M && ncol0 < N) {
            if (out_f32_flag) {
              *reinterpret_cast<float2 *>(out_f32 + (size_t)m * N + ncol0) = make_float2(lo, hi);
            } else {
              *reinterpret_cast<__nv_bfloat162 *>(out_bf16 + (size_t)m * N + ncol0) =
                  __floats2bfloat162_rn(lo, hi);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

template <int SPG, int SC, bool ZP, int FIXED>
static cudaError_t launch_pf(const Plan &p, int M, int K, int N, int prec, const CUtensorMap &mw,
                             const CUtensorMap &ma, const void *scales, const void *zeros,
                             void *out, float *part, unsigned *counters, unsigned token,
                             cudaStream_t s) {
  auto kern = w4_prefill_kernel<SPG, SC, ZP, FIXED>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       p.smem_bytes);
  if (e != cudaSuccess) {
    note_cuda_error("cudaFuncSetAttribute(prefill)", e);
    return e;
  }
  const bool f32 = (prec & GQ_OUT_F32) != 0;
  kern<<<p.grid_x, kPfThreads, p.smem_bytes, s>>>(
      mw, ma, scales, reinterpret_cast<const uint32_t *>(zeros),
      f32 ? nullptr : reinterpret_cast<__nv_bfloat16 *>(out), f32 ? reinterpret_cast<float *>(out) : nullptr,
      M, K, N, f32 ? 1 : 0, PrefillConsts{0x43004300u, 0x43084308u},
      PrefillShape{p.m_tile, p.slots, p.nsplit, part, counters}, token);
  return cudaGetLastError();
}

template <int SPG, int SC, int FIXED>
static cudaError_t launch_pf_z(const Plan &p, int M, int K, int N, int prec, const CUtensorMap &mw,
                               const CUtensorMap &ma, const void *scales, const void *zeros,
                               void *out, float *part, unsigned *counters, unsigned token,
                               cudaStream_t s) {
  if (prec & GQ_ZP)
    return launch_pf<SPG, SC, true, FIXED>(p, M, K, N, prec, mw, ma, scales, zeros, out, part,
                                           counters, token, s);
  return launch_pf<SPG, SC, false, FIXED>(p, M, K, N, prec, mw, ma, scales, zeros, out, part,
                                          counters, token, s);
}

template <int SPG, int FIXED>
static cudaError_t launch_pf_s(const Plan &p, int M, int K, int N, int prec, const CUtensorMap &mw,
                               const CUtensorMap &ma, const void *scales, const void *zeros,
                               void *out, float *part, unsigned *counters, unsigned token,
                               cudaStream_t s) {
  if (prec & GQ_SC_F32)
    return launch_pf_z<SPG, kScF32, FIXED>(p, M, K, N, prec, mw, ma, scales, zeros, out, part,
                                           counters, token, s);
  if (prec & GQ_SC_BF16)
    return launch_pf_z<SPG, kScBF16, FIXED>(p, M, K, N, prec, mw, ma, scales, zeros, out, part,
                                            counters, token, s);
  return launch_pf_z<SPG, kScF16, FIXED>(p, M, K, N, prec, mw, ma, scales, zeros, out, part,
                                         counters, token, s);
}

// every instance of one FIXED value, by group size
template <int FIXED>
static cudaError_t launch_pf_g(const Plan &p, int M, int K, int N, int G, int prec,
                               const CUtensorMap &mw, const CUtensorMap &ma, const void *scales,
                               const void *zeros, void *out, float *part, unsigned *counters,
                               unsigned token, cudaStream_t s) {
  switch (G) {
    case 64:
      return launch_pf_s<1, FIXED>(p, M, K, N, prec, mw, ma, scales, zeros, out, part, counters,
                                   token, s);
    case 128:
      return launch_pf_s<2, FIXED>(p, M, K, N, prec, mw, ma, scales, zeros, out, part, counters,
                                   token, s);
    case 256:
      return launch_pf_s<4, FIXED>(p, M, K, N, prec, mw, ma, scales, zeros, out, part, counters,
                                   token, s);
    default:
      return cudaErrorInvalidValue;
  }
}

// this translation unit's wait limit and error word
static int pf_tu_set_wait_limit(long long cycles) {
  return cudaMemcpyToSymbol(g_pf_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? 0 : -1;
}

static int pf_tu_read_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(g_prefill_error, &z, sizeof(int));
  }
  return v;
}

// gq_prefill_fixed.cu: the FIXED = 1 instances and that unit's wait limit and error word
cudaError_t launch_prefill_fixed(const Plan &p, int M, int K, int N, int G, int prec,
                                 const CUtensorMap &mw, const CUtensorMap &ma, const void *scales,
                                 const void *zeros, void *out, unsigned token, cudaStream_t s);
int prefill_fixed_set_wait_limit(long long cycles);
int prefill_fixed_read_error(int clear);

}  // namespace gq

// Internal declarations shared by the translation units of libgq (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gq.h"

namespace gq {

// Packed W4 layout: 16-column tiles x 64-k chunks; a chunk is 32 lanes x 16 bytes.
constexpr int kTileN = 16;
constexpr int kChunkK = 64;
// Packed W8 layout: 64-column blocks stored one after another, each holding its K/16 chunk
// rows contiguously; a chunk row of block b is w_b = min(64, N - 64b) columns x 16 bytes
// (16 consecutive k of one column).  K·N bytes in all.
constexpr int kChunkK8 = 16;
constexpr int kColBlock8 = 64;
// 16-byte index of chunk row c (k = 16c .. 16c+15) of column n
__host__ __device__ inline size_t w8_chunk_index(int K, int N, int n, int c) {
  const int b = n / kColBlock8, j = n - b * kColBlock8;
  const int wb = N - b * kColBlock8 < kColBlock8 ? N - b * kColBlock8 : kColBlock8;
  return (size_t)b * (kColBlock8 / kChunkK8) * K + (size_t)c * wb + j;
}

// Small-M tensor-core decode kernel: warps per CTA (each warp owns one 16-column tile).
constexpr int kDecWarps = 8;
constexpr int kDecMaxMT = 4;           // up to 4 x 8 = 32 rows of A per CTA
// Striped small-M decode kernel (M <= 8): warps per CTA, one CTA per SM.
constexpr int kStrWarps = 24;
// INT8 CUDA-core decode kernel: one column per thread.
constexpr int kQ8Threads = 128;
constexpr int kQ8MaxRows = 32;

// Scratch layout: a fixed region of arrival counters at offset 0 (every call leaves them
// at zero, and no problem's partial sums ever overlap them), then the partial sums.
constexpr size_t kCounterRegionBytes = 256u << 10;   // 65536 counters

enum Path { kPathMmaDecode = 0, kPathQ8Decode = 1, kPathPrefill = 2, kPathStripe = 3,
            kPathBatch = 4, kPathQ8Block = 5, kPathQ8Mma = 6, kPathQ8A8 = 7, kPathGemv = 8,
            kPathQ8Gemv = 9 };

struct Plan {
  int path;
  int nsplit;       // K slices (paths 0, 1) or warp stripes (path 3)
  int units;        // number of split units along K
  int unit_k;       // k per unit (a whole number of groups)
  int m_tile;       // rows per CTA
  int mt;           // n8 MMA blocks per CTA (path 0)
  int n_tile;       // columns per CTA
  int grid_x, grid_y, grid_z;
  int block_threads;
  size_t smem_bytes;
  size_t part_bytes;     // split-K partials
  size_t counter_bytes;  // arrival counters
  size_t workspace_bytes;
  int split_count, split_mult;   // paths 3, 8, 9: CTA c owns zsplit(split_count, grid, c) * split_mult
  int slots;                     // path 3: ring slots per warp; path 2: TMA ring stages
  int table_bytes;               // paths 8, 9: bytes of a consumer warp's scale table
};

// scale / output type codes used as template parameters
enum ScaleType { kScF16 = 0, kScBF16 = 1, kScF32 = 2 };

int validate(int M, int K, int N, int G, int prec);
// The K-slice count forced by gq_set_split_override (0 = the planner's own choice, -1 = the
// largest count the path supports, n > 0 = exactly n).  The slice choosers take it as
// `forced` and return 0 when the path cannot take that count.
int split_override();
int make_plan(int M, int K, int N, int G, int prec, int sm_count, Plan *p);
size_t plan_counter_bytes_used(const Plan &p, int M, int N);
// the body of gq_gemm (validation, plan, scratch, launch)
int gemm_impl(int M, int K, int N, int G, int prec, const void *A, const void *Wq,
              const void *scales, const void *zeros, void *out, void *stream);
size_t packed_bytes(int K, int N, int prec);
int device_sm_count(int *sms);
// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes) on the current device, issued
// only when this process has not yet raised that kernel's limit to at least `bytes` there
// (a per-call driver call costs host time on every launch of the decode path).
cudaError_t ensure_dynamic_smem(const void *func, size_t bytes);

// launchers (return cudaError_t of the launch)
cudaError_t launch_pack_w4(int K, int N, const uint32_t *codes, uint32_t *packed, bool gate_up,
                           cudaStream_t s);
cudaError_t launch_pack_w8(int K, int N, const int8_t *codes, uint8_t *packed, bool gate_up,
                           cudaStream_t s);
cudaError_t launch_mma_decode(const Plan &p, int M, int K, int N, int G, int prec,
                              const void *A, const void *Wq, const void *scales,
                              const void *zeros, void *out, float *part,
                              unsigned *counters, cudaStream_t s);
// warp-specialized small-M decode kernel (M <= 4): a producer warp and sixteen consumer
// warps per CTA
bool gemv_supported(int M, int K, int G, int prec);
int gemv_table_bytes(int G, int prec, int max_cta_slots);
size_t gemv_smem_bytes(int M, int K, int G, int prec, int max_cta_slots);
int gemv_threads();
cudaError_t launch_gemv(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                        const void *Wq, const void *scales, const void *zeros, void *out,
                        float *part, unsigned *counters, cudaStream_t s);
int gemv_read_error(int clear);
// per translation unit: the SM clock cycles after which a bounded device-side wait gives up
int gemv_set_wait_limit(long long cycles);
// GQ_FAULT_DEVICE_WAIT: the producer warps of later launches withhold one slot
int gemv_set_withhold(bool on);
// warp-specialized INT8 decode kernel (N a multiple of 64, M <= 4, W8A16 or W8A8): a producer
// warp and sixteen consumer warps per CTA over (64-column block, group) units
bool q8_gemv_supported(int M, int K, int N, int G, int prec);
int q8_gemv_table_bytes(int max_cta_units);
size_t q8_gemv_smem_bytes(int M, int K, int G, int prec, int max_cta_units);
size_t q8_gemv_part_bytes(int grid);
int q8_gemv_threads();
// A: fp32 activations, or INT8 ones with a_scales [M][K/G] (GQ_ACT_I8)
cudaError_t launch_q8_gemv(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                           const float *a_scales, const void *Wq, const void *scales,
                           void *out, float *part, unsigned *counters, cudaStream_t s);
int q8_gemv_read_error(int clear);
int q8_gemv_set_wait_limit(long long cycles);
// gq_set_fault_injection(GQ_FAULT_LAUNCH): true, with the error detail noted, when the next
// launch is to fail
bool launch_fault_injected();
int stripe_set_wait_limit(long long cycles);
int batch_set_wait_limit(long long cycles);
int prefill_set_wait_limit(long long cycles);
int fp8_set_wait_limit(long long cycles);
bool stripe_supported(int M, int K, int G, int prec);
size_t stripe_smem_bytes(int M, int K, int G, int prec, int slots);
int stripe_slots_for(int M, int K, int G, int prec, size_t smem_cap);
int stripe_slot_k();
cudaError_t launch_stripe_decode(const Plan &p, int M, int K, int N, int G, int prec,
                                const void *A, const void *Wq, const void *scales,
                                const void *zeros, void *out, float *part,
                                unsigned *counters, cudaStream_t s);
size_t prefill_smem_bytes(int BM, int stages);
int prefill_stages(int BM, size_t smem_cap);
bool prefill_supported(int M, int K, int N, int G, int prec);
cudaError_t launch_prefill(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                           const void *Wq, const void *scales, const void *zeros, void *out,
                           float *part, unsigned *counters, cudaStream_t s);
int prefill_read_error(int clear);
int stripe_read_error(int clear);
bool batch_supported(int M, int K, int G, int prec);
int batch_slice_k(int M, int K);
size_t batch_smem_bytes(int M, int K_slice, int G, int prec, int slots);
int batch_slots_for(int M, int K_slice, int G, int prec, size_t smem_cap);
int batch_threads(int M);
cudaError_t launch_batch(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                         const void *Wq, const void *scales, const void *zeros, void *out,
                         float *part, unsigned *counters, cudaStream_t s);
int batch_read_error(int clear);


// Records why a call is about to return GQ_ERR_CUDA (thread-local; read by gq_last_error_detail).
void note_cuda_error(const char *where, cudaError_t e);
void note_cuda_error_code(const char *where, int code);
// largest M of the small-batch kernel (it takes 33..64 rows only where the prefill kernel
// does not apply: G = 32)
constexpr int kBatchMaxM = 64;
// smallest M routed to the tensor-core prefill kernel: from 25 rows the small-batch kernel
// needs four 8-row MMA tiles per step and the prefill kernel's 64-row tile is faster
// (K=4096 N=14336 G=128: 33.0 against 31.3 us at M=28, 27.5 against 31.2 us at M=24);
// with INT4 zero points from 33 rows, where the small-batch kernel needs a second row block
constexpr int kPrefillMinM = 25;
constexpr int kPrefillMinMZp = 33;
constexpr int kPrefillThreads = 512;   // block size of the prefill kernel
cudaError_t launch_q8_decode(const Plan &p, int M, int K, int N, int G, int prec,
                             const void *A, const void *Wq, const void *scales,
                             void *out, float *part, unsigned *counters, cudaStream_t s);
// INT8 CUDA-core kernel for M <= kQ8BlockMaxM (64 columns x one K slice per CTA)
constexpr int kQ8BlockMaxM = 32;
bool q8_block_supported(int M, int K, int G, int prec);
size_t q8_block_smem_bytes(int M, int K, int G, int KS);
int q8_block_slices(int M, int K, int N, int G, int sms, size_t part_cap, int forced);
int q8_block_cols();
int q8_block_threads();
cudaError_t launch_q8_block(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                            const void *Wq, const void *scales, void *out, float *part,
                            unsigned *counters, cudaStream_t s);
// INT8 on BF16 tensor cores (codes exact, fp32 activations as three exact BF16 parts)
bool q8_mma_supported(int M, int K, int G, int prec);
size_t q8_mma_smem_bytes(int M, int K, int G, int KS);
int q8_mma_slices(int M, int K, int N, int G, int sms, size_t part_cap, int forced);
cudaError_t launch_q8_mma(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                          const void *Wq, const void *scales, void *out, float *part,
                          unsigned *counters, cudaStream_t s);
// INT8-activation variant (W8A8): the dynamic activation quantizer and the integer group GEMM
cudaError_t launch_quantize_act(int M, int K, int G, bool f32, const void *A, int8_t *Aq,
                                float *a_scales, cudaStream_t s);
int q8a8_slices(int M, int K, int N, int G, int sms, size_t part_cap, int forced);
size_t q8a8_smem_bytes(int M, int K, int G, int KS);
cudaError_t launch_q8a8(const Plan &p, int M, int K, int N, int G, int prec, const int8_t *Aq,
                        const float *As, const void *Wq, const void *scales, void *out,
                        float *part, unsigned *counters, cudaStream_t s);
// FP8 W8A8 block-scaled GEMM (tcgen05 kind::f8f6f4)
size_t fp8_smem_bytes();
int fp8_block_plan(int M, int N, int sms, int *grid);
int launch_fp8_block(int M, int K, int N, int prec, const void *A, const void *a_scales,
                     const void *W, const void *w_scales, void *out, int grid, cudaStream_t s);
int fp8_read_error(int clear);
int launch_quantize_fp8(int M, int K, bool f32, const void *A, void *Aq, void *scales,
                        cudaStream_t s);
// Launches the kernel of plan p (any path); part and counters may be NULL when the plan
// needs no workspace.
cudaError_t launch_plan(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                        const void *Wq, const void *scales, const void *zeros, void *out,
                        float *part, unsigned *counters, cudaStream_t s);

}  // namespace gq

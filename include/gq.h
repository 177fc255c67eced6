/*
 * gq.h — group-quantized weight-only GEMM on one NVIDIA GB300 (sm_103a).  C ABI.
 *
 * The operation (the group-wise GEMM of "04 · 分组量化 GEMM 内核", section 2, with the
 * activation scale fixed to 1; the affine relation x ≈ s·(q − z) of "GPU Kernel 工程（09）：
 * 量化与融合 kernel", section 2.1):
 *
 *     out[m][n] = Σ_g s[g][n] · Σ_{k ∈ group g} A[m][k] · (q[k][n] − z[g][n])
 *
 * for 0 ≤ m < M, 0 ≤ n < N, groups of G consecutive k.  Every group's dot product is
 * finished before its scale multiplies it; accumulation is FP32.
 *
 * Conventions for every call below:
 *   - Matrices are row-major and dense (no leading-dimension argument).
 *   - "device" pointers are CUDA device memory owned by the caller; the library never
 *     frees or retains them beyond the call (the workspace of gq_set_workspace excepted).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  gq_pack_weights and
 *     gq_gemm only enqueue work on it and return; they never synchronize the device.
 *   - Every call returns a gq_status.  Arguments are validated before anything is
 *     launched: an invalid call launches nothing and leaves every buffer untouched.
 *     Nothing is thrown across the ABI and nothing aborts the process.
 */
#ifndef GQ_H_
#define GQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gq_status {
  GQ_OK = 0,
  GQ_ERR_INVALID_ARG = 1,  /* shape, null pointer or flag combination outside the contract */
  GQ_ERR_UNSUPPORTED = 2,  /* legal in principle, not implemented (e.g. an unsupported G)   */
  GQ_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned                              */
  GQ_ERR_WORKSPACE = 4,    /* the registered workspace is smaller than gq_workspace_size    */
  GQ_ERR_CUDA = 5,         /* a CUDA runtime call or a launch failed                        */
  GQ_ERR_TIMEOUT = 6,      /* a bounded device-side wait gave up (sticky, see gq_device_error) */
  GQ_ERR_NO_DEVICE = 7     /* no CUDA device of compute capability 10.3 is current          */
} gq_status;

/* `prec`: a bit field describing the operand types. */
#define GQ_W4      0x01  /* INT4 codes in [0,15]; clear = INT8 codes in [-128,127], z = 0     */
#define GQ_ZP      0x02  /* W4 only: per-group INT4 zero points given; clear = z = 8 (W4)     */
#define GQ_ACT_F32 0x04  /* activations fp32; clear = bf16                                     */
#define GQ_SC_BF16 0x08  /* scales bf16                                                        */
#define GQ_SC_F32  0x10  /* scales fp32; neither SC flag = fp16                                */
#define GQ_OUT_F32 0x20  /* output fp32; clear = bf16 (round to nearest even)                  */
#define GQ_GATE_UP  0x80 /* fused gate+up projection: the N = 2F columns are F gate columns
                            then F up columns, and out is [M][F] = silu(gate) * up (silu(x) =
                            x / (1 + e^-x), in FP32 on the FP32 GEMM results, then rounded).
                            gq_pack_weights must get the flag too (it interleaves gate and up
                            columns: W4 tile by tile, W8 64-column block by block).  W4: N % 16
                            == 0 and, in gq_gemm, K % 256 == 0 and M <= 64 (the decode and
                            small-batch kernels); W8: N % 64 == 0 and M <= 32 (the INT8 CUDA-
                            core and tensor-core kernels); else GQ_ERR_UNSUPPORTED          */
#define GQ_ACT_I8  0x100  /* INT8-activation variant (gq_gemm_a8, and gq_plan / gq_workspace_size
                            for it): activations are int8 codes with one fp32 scale per (row,
                            group); W8 codes and GQ_SC_F32 only; gq_gemm refuses it         */
#define GQ_ZP_FLOAT 0x200 /* W4 float zero points ("GPU Kernel 工程（09）：量化与融合 kernel",
                            section 3.4, Machete's form out = (w_q * w_s - w_z) @ a): zeros is
                            [K/G][N] in the scales' format and W_hat = q * s - zf, the zero
                            subtracted after scaling.  Excludes GQ_ZP, GQ_GATE_UP, GQ_ACT_I8;
                            needs bf16 activations, K % 256 == 0 and M <= 64 (the small-batch
                            kernel), else GQ_ERR_UNSUPPORTED                                  */
#define GQ_STATIC_W 0x40 /* Wq, scales and zeros are not written by work still running on the
                            stream (weights loaded once, as in serving): the decode kernels
                            may start streaming them before the preceding kernel has ended;
                            activations and outputs still wait for it                         */

/*
 * Supported operand combinations (anything else returns GQ_ERR_UNSUPPORTED):
 *   W4 : activations bf16; scales fp16, bf16 or fp32; zero points optional (packed INT4 with
 *        GQ_ZP, or float in the scales' format with GQ_ZP_FLOAT); out bf16 or fp32.
 *   W8 : activations fp32; scales fp32; no zero points; out fp32 or bf16.
 * Shape contract: M ≥ 0, N ≥ 0 (either 0 is a valid empty call), N % 8 == 0, G in
 * {32, 64, 128, 256}, K ≥ G, K % G == 0, and K % 64 == 0 for W4 (K % 16 == 0 for W8).
 */

/* ---------------------------------------------------------------------------------------
 * Canonical input layouts (what callers hold):
 *   A       [M][K]      bf16 or fp32.
 *   codes   W4: uint32 [K/8][N]: word (r, n) holds k = 8r..8r+7 of column n, element j in
 *               bits 4j..4j+3 (the INT4 packing of "量化与融合 kernel" section 2.4 and its
 *               INT4 GEMV of section 9.4).
 *           W8: int8 [K][N] (the int8 code matrix of "分组量化 GEMM 内核" section 3.2).
 *   scales  [K/G][N]    fp16, bf16 or fp32 ("量化与融合 kernel" section 3.1).
 *   zeros   uint32 [K/G][N/8]: word (g, c) holds n = 8c..8c+7, element j in bits 4j
 *           (the [K/g, N/8] INT4 zero points of section 3.1).
 *   out     [M][N]      bf16 or fp32.
 * ------------------------------------------------------------------------------------- */

/* Size in bytes of the packed weight buffer for (K, N, G, prec).  Host only; touches no
 * device.  W4: ceil(N/16)·16 · K/2 bytes (N is padded to whole 16-column tiles);
 * W8: K·N bytes.  Errors: GQ_ERR_INVALID_ARG for a shape outside the contract or a NULL
 * `bytes`. */
int gq_packed_bytes(int K, int N, int G, int prec, size_t *bytes);

/* Repack canonical codes into the device layout that gq_gemm reads (the offline repack of
 * "量化与融合 kernel" section 3.3, item 1: the interleaved order lets one 16-byte load be
 * decoded in registers directly into tensor-core operand fragments).
 *   codes   device, canonical layout above (W4 uint32 [K/8][N]; W8 int8 [K][N]).
 *   packed  device, gq_packed_bytes(...) bytes, written entirely (padding included).
 * Deterministic; asynchronous on `stream`.  Errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT
 * (either pointer not 16-byte aligned), CUDA. */
int gq_pack_weights(int K, int N, int G, int prec, const void *codes, void *packed,
                    void *stream);

/* Scratch bytes gq_gemm needs for this problem on the current device (split-K partial
 * sums and per-tile arrival counters; 0 when the problem is not split).  Host only, but
 * reads the current device's SM count.  Errors: INVALID_ARG, UNSUPPORTED, NO_DEVICE. */
int gq_workspace_size(int M, int K, int N, int G, int prec, size_t *bytes);

/* Register caller-owned device scratch for the current device (NULL, 0 = drop it and go
 * back to the library-owned buffer).  The library zeroes it once here (synchronously) and
 * afterwards keeps its counters at zero between calls.  Calls that overlap in time on
 * different streams must not share one workspace.  Errors: ALIGNMENT (not 256-byte
 * aligned), CUDA. */
int gq_set_workspace(void *dev_ptr, size_t bytes);

/* out = the group-quantized GEMM above.
 *   A       device [M][K], bf16 (or fp32 with GQ_ACT_F32).
 *   Wq      device, packed by gq_pack_weights with the same (K, N, G, prec).
 *   scales  device [K/G][N].
 *   zeros   device [K/G][N/8] uint32 with GQ_ZP, [K/G][N] in the scales' format with
 *           GQ_ZP_FLOAT, else must be NULL.
 *   out     device [M][N], fully overwritten.
 * Path choice depends only on (M, K, N, G, prec) and the device's SM count, so a given
 * problem on a given device always produces the same bits.  Scratch comes from the
 * registered workspace, else from a library-owned per-device buffer allocated (once, and
 * grown when a larger problem needs it) on first use — that first use synchronizes the
 * device and must not happen during stream capture.  All pointers 16-byte aligned.
 * Errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA, NO_DEVICE. */
int gq_gemm(int M, int K, int N, int G, int prec, const void *A, const void *Wq,
            const void *scales, const void *zeros, void *out, void *stream);

/* gq_gemm on host-resident activations and output: the activations are copied to the
 * caller's device staging buffer, the GEMM runs, and the output is copied back, all three
 * asynchronous on `stream` in that order (the host buffers must stay valid, and `out_host`
 * must not be read, until the stream has passed the call; page-locked host memory keeps the
 * copies asynchronous).
 *   A_host    host [M][K], bf16 (or fp32 with GQ_ACT_F32).
 *   A_dev     device staging buffer of the same size, overwritten.
 *   Wq, scales, zeros  device, as for gq_gemm.
 *   out_dev   device [M][N] (gate+up: [M][N/2]), bf16 or fp32 with GQ_OUT_F32, overwritten.
 *   out_host  host buffer of the same size, receives the output.
 * The activations' and output's sizes follow from (M, K, N, prec).  Errors as gq_gemm, all
 * but CUDA reported before anything is issued; INVALID_ARG also for a NULL host pointer. */
int gq_gemm_host(int M, int K, int N, int G, int prec, const void *A_host, void *A_dev,
                 const void *Wq, const void *scales, const void *zeros, void *out_dev,
                 void *out_host, void *stream);

/* gq_gemm without any device allocation.  The pages have no counterpart: this call exists
 * for callers that cannot allocate device memory — serving runtimes that reserve all
 * device memory up front and forbid allocation once running, latency-critical loops where
 * an allocation and the device synchronization it may bring are not acceptable, and
 * embedders that route every device allocation through their own allocator.
 *   Arguments, layouts, results and errors are those of gq_gemm, computed by the same
 * kernels.  The split-K scratch comes from one array of GQ_STATIC_SCRATCH_BYTES compiled
 * into the library (every GPU that loads the library holds it until the process exits)
 * instead of the registered or library-owned workspace; a problem whose scratch
 * (gq_workspace_size) exceeds it returns GQ_ERR_WORKSPACE and launches nothing.
 *   The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call before any
 * stream capture.  Every call that splits K clears the arrival counters its plan indexes (an
 * asynchronous memset of 4 bytes per output tile on `stream`, a few KiB at most).  All calls on a device share the one array, which keeps the last call's
 * contents, so calls that overlap on the GPU — different streams, or host threads without
 * ordering between them — race on it and must be serialized by the caller. */
#define GQ_STATIC_SCRATCH_BYTES (4u << 20)
int gq_gemm_static_scratch(int M, int K, int N, int G, int prec, const void *A,
                           const void *Wq, const void *scales, const void *zeros, void *out,
                           void *stream);

/* Timing harness over caller buffers.  Runs `warmup` untimed and then `iters` timed gq_gemm calls back to back
 * on `stream`, call i reading weight copy i % n_copies (so that copies larger than L2 in
 * total make every call read from HBM), and reports the mean time per call from CUDA
 * events recorded on `stream`.  With use_graph != 0 the `iters` calls are captured once
 * into a CUDA graph and the graph is replayed (no host launch overhead); the workspace
 * must already exist then (call gq_gemm once first), and `stream` must not be the legacy
 * default stream (NULL), which cannot be captured.  Synchronizes `stream`. */
typedef struct gq_bench_args {
  int M, K, N, G, prec;
  const void *A;
  const void *const *Wq;       /* n_copies device pointers (host array) */
  const void *const *scales;   /* n_copies device pointers (host array) */
  const void *const *zeros;    /* n_copies device pointers, or NULL without GQ_ZP / GQ_ZP_FLOAT */
  int n_copies;
  void *out;
  int warmup, iters, use_graph;
  void *stream;
  const void *a_scales;        /* GQ_ACT_I8: device fp32 [M][K/G] activation scales (A holds the
                                  int8 codes) and each call is gq_gemm_a8; else NULL */
} gq_bench_args;

typedef struct gq_bench_result {
  double us_per_call;          /* mean device time per gq_gemm call */
  int launches_per_call;       /* kernels one gq_gemm call launches for this problem */
} gq_bench_result;

int gq_bench_calls(const gq_bench_args *args, gq_bench_result *result);

/* Self-contained benchmark of a named workload (the measured-data section, 四, of "04 · 分组量化
 * GEMM 内核" reports time per call per shape; its tables did not survive, so the workloads are
 * the library's five configurations):
 *   "tiny_gemv"     M=1    K=512  N=512   G=128  W4 sym, fp16 scales, bf16 act/out
 *   "decode_gateup" M=1    K=4096 N=28672 G=128  W4 sym, fp16 scales, 0.1% x50 activations
 *   "q8_m1"/"q8_m32" M=1/32 K=2048 N=12288 G=32  INT8 codes, fp32 scales/act/out
 *   "asym_m16"      M=16   K=8192 N=28672 G=128  W4 with INT4 zero points, bf16 scales
 *   "prefill"       M=4096 K=4096 N=14336 G=128  W4 sym, fp16 scales
 *   "all"           every one of the above, in that order (a JSON array).
 * It allocates the workload on the current device, fills it on the device from a
 * counter-based hash with the stated distributions (codes uniform, scales uniform in
 * [0.005, 0.02] or [1e-3, 1e-2], zero points uniform in [4, 11], activations N(0, 1) by
 * Box-Muller), packs the weights into enough rotated copies that one round of them exceeds
 * twice the L2 (decode shapes), and times gq_gemm with CUDA events: five repeats of a CUDA
 * graph of back-to-back calls (host-launched calls from M = 128), reporting the median, 10th
 * and 90th percentile microseconds per call, the median latency of single host-launched
 * calls, GB/s of the algorithmic bytes (codes, scales, zero points, activations once, output
 * once), TFLOPS (2·M·N·K), the roofline fraction — against the library's own 1 GiB copy kernel
 * (read + write bytes) for M < 128, against the nominal 2250 TFLOPS dense BF16 above — the
 * kernels launched per call, and whether two calls gave identical bits.  Synchronizes the
 * device and frees everything it allocated before returning.
 *   json_out  host buffer of `cap` bytes; receives one NUL-terminated JSON object (an array
 *             for "all").
 * Errors: GQ_ERR_INVALID_ARG (unknown name, NULL json_out, or cap too small for the result:
 * then json_out holds ""), GQ_ERR_NO_DEVICE, GQ_ERR_CUDA (an allocation or launch failed),
 * and any status of gq_gemm. */
int gq_bench(const char *config, char *json_out, size_t cap);

/* ---------------------------------------------------------------------------------------
 * INT8-activation variant: the group-wise GEMM with integer activations of "04 · 分组量化
 * GEMM 内核" section 2,
 *     out[m][n] = Σ_g a_scales[m][g] · scales[g][n] · ( Σ_{k ∈ g} Aq[m][k] · q[k][n] ),
 * the integer dot of a whole group finished exactly (INT32) before either scale.
 * ------------------------------------------------------------------------------------- */

/* Dynamic per-group INT8 quantization of activations (the absmax reduction and cast of
 * "量化与融合 kernel" section 四.5, with 127 and one scale per group of G):
 *   a_scales[m][g] = max_{k in g} |A[m][k]| / 127        (FP32 division)
 *   Aq[m][k]       = rint(A[m][k] / a_scales[m][g])      (FP32 division, ties to even),
 *                    clamped to [-127, 127]; a group of zeros gets scale 0 and codes 0.
 *   A        device [M][K] bf16, or fp32 with GQ_ACT_F32 (prec holds no other flag).
 *   Aq       device int8 [M][K];  a_scales  device fp32 [M][K/G].
 * Asynchronous on stream.  Errors: GQ_ERR_INVALID_ARG (M < 0, K % G != 0, G outside
 * {32, 64, 128, 256}, K % 16 != 0, NULL pointer, other flags), GQ_ERR_ALIGNMENT (a pointer
 * not 16-byte aligned), GQ_ERR_CUDA. */
int gq_quantize_act(int M, int K, int G, int prec, const void *A, void *Aq, void *a_scales,
                    void *stream);

/* The W8A8 group GEMM above.  prec = GQ_ACT_I8 | GQ_SC_F32 [| GQ_OUT_F32] [| GQ_STATIC_W].
 *   Aq        device int8 [M][K] (e.g. from gq_quantize_act);  a_scales  device fp32 [M][K/G].
 *   Wq        W8 codes packed by gq_pack_weights (prec without GQ_W4);
 *   scales    device fp32 [K/G][N];  out  device [M][N] bf16, or fp32 with GQ_OUT_F32.
 * Shape contract and workspace as gq_gemm (gq_workspace_size with the same prec).
 * Errors as gq_gemm; GQ_ERR_UNSUPPORTED for GQ_W4, GQ_ZP, GQ_ACT_F32 or GQ_GATE_UP. */
int gq_gemm_a8(int M, int K, int N, int G, int prec, const void *Aq, const void *a_scales,
               const void *Wq, const void *scales, void *out, void *stream);

/* ---------------------------------------------------------------------------------------
 * FP8 W8A8 GEMM with block scales ("GPU Kernel 工程（09）：量化与融合 kernel", section 四.3):
 *     out[m][n] = Σ_b a_scales[b][m] · w_scales[n/128][b] · Σ_{k in block b} A[m][k]·W[n][k]
 * over 128-k blocks b; each block's tensor-core sum is scaled and added into FP32 inside the
 * K loop (the scales depend on k, so they cannot wait for the epilogue).
 *   A         device FP8 E4M3 bytes [M][K];  a_scales  device fp32 [K/128][M] (one per row and
 *             block, M contiguous);
 *   W         device FP8 E4M3 bytes [N][K] (k contiguous: row n is output column n);
 *   w_scales  device fp32 [ceil(N/128)][K/128] (one per 128 x 128 block);
 *   out       device [M][N] bf16, or fp32 with GQ_OUT_F32 (prec holds no other flag).
 * Contract: M >= 0, N >= 0 (either 0: nothing launched), K >= 128, K % 128 == 0, N % 16 == 0;
 * pointers 16-byte aligned.  Needs no workspace.  Asynchronous on stream.  Errors:
 * GQ_ERR_INVALID_ARG, GQ_ERR_ALIGNMENT, GQ_ERR_CUDA; a bounded device wait that gives up
 * sets GQ_ERR_TIMEOUT in gq_device_error. */
int gq_gemm_fp8_block(int M, int K, int N, int prec, const void *A, const void *a_scales,
                      const void *W, const void *w_scales, void *out, void *stream);

/* Dynamic FP8 quantization of activations for gq_gemm_fp8_block (the absmax reduction and cast
 * of "量化与融合 kernel" section 四.5, one scale per row and 128-k block):
 *   a_scales[b][m] = max_{k in block b} |A[m][k]| / 448         (binary32 division)
 *   Aq[m][k]       = E4M3(A[m][k] / a_scales[b][m])              (binary32 division, round to
 *                    nearest even, saturated to ±448); a block of zeros: scale 0, codes 0.
 *   A         device [M][K] bf16, or fp32 with GQ_ACT_F32 (prec holds no other flag);
 *   Aq        device E4M3 bytes [M][K];  a_scales  device fp32 [K/128][M].
 * Contract: M >= 0, K >= 128, K % 128 == 0; pointers 16-byte aligned.  Asynchronous.
 * Errors: GQ_ERR_INVALID_ARG, GQ_ERR_ALIGNMENT, GQ_ERR_CUDA. */
int gq_quantize_act_fp8(int M, int K, int prec, const void *A, void *Aq, void *a_scales,
                        void *stream);

/* Testing and diagnostics: force the number of K slices (split-K over whole groups, summed in
 * slice order) that the planner gives the kernels that split K — paths 0, 1, 4, 5, 6 and 7 of
 * gq_plan_t below.  n >= 1 asks for exactly n slices, n = -1 for the largest count the path
 * supports, n = 0 restores the planner's own choice (the default).  Process-wide; it changes
 * what gq_plan, gq_workspace_size, gq_gemm, gq_gemm_a8 and gq_gemm_static_scratch do until it
 * is reset, and a count that the chosen path cannot take makes them return
 * GQ_ERR_UNSUPPORTED.  The path itself and paths that do not split K are unaffected.  Every
 * count gives results within the tolerance of the group GEMM; the bits may differ between
 * counts (another summation order) but never between runs at one count ("分组量化 GEMM 内核"
 * section 3.3: the z-split and its fixed-order reduction).  Host only; returns the previous
 * setting, or -2 (and changes nothing) for n < -1. */
int gq_set_split_override(int n);

/* Testing and diagnostics: the SM clock cycles after which every bounded device-side wait in
 * the library's kernels gives up (it records GQ_ERR_TIMEOUT, which gq_device_error reports,
 * and the kernel leaves early; nothing traps or hangs).  cycles = 0 restores the default,
 * 4e9 cycles (about two seconds at 2 GHz); otherwise 1e4 <= cycles <= 1e11.  Applies to the
 * current device from the next launch on; synchronous.  Errors: GQ_ERR_INVALID_ARG,
 * GQ_ERR_NO_DEVICE, GQ_ERR_CUDA. */
int gq_set_wait_limit(long long cycles);

/* Testing: injected failures, to check that each one surfaces as the documented status.
 *   GQ_FAULT_NONE         no injection (the default).
 *   GQ_FAULT_WORKSPACE    the library-owned scratch cannot be had: a gq_gemm or gq_gemm_a8
 *                         that needs it returns GQ_ERR_CUDA ("workspace allocation
 *                         (injected)" in gq_last_error_detail) and launches nothing.
 *   GQ_FAULT_LAUNCH       the kernel launch fails: gq_gemm, gq_gemm_a8 and
 *                         gq_gemm_static_scratch return GQ_ERR_CUDA ("launch (injected)") and
 *                         launch nothing.
 *   GQ_FAULT_DEVICE_WAIT  on the device: in the warp-specialized decode kernel (gq_plan path 8)
 *                         the producer warp of every CTA withholds its first consumer's first
 *                         slot, so that consumer's bounded wait runs out (gq_set_wait_limit
 *                         shortens it); the call ends early with an output that is not valid
 *                         and gq_device_error reports GQ_ERR_TIMEOUT.  Other paths ignore it.
 * Process-wide; the device-side form is set on the current device (synchronous).  Returns the
 * previous setting, or -1 (and changes nothing) for an unknown value. */
#define GQ_FAULT_NONE 0
#define GQ_FAULT_WORKSPACE 1
#define GQ_FAULT_LAUNCH 2
#define GQ_FAULT_DEVICE_WAIT 3
int gq_set_fault_injection(int fault);

/* Host-only description of the launch gq_gemm would make (for tests and reports).
 * sm_count > 0 overrides the device query, so it works without a GPU. */
typedef struct gq_plan_t {
  int path;          /* 0 = small-M tensor-core decode (mma.sync, K split across CTAs),
                        1 = INT8 CUDA-core decode (M > 32), 2 = tcgen05 prefill (W4, M >= 25; 33 with GQ_ZP),
                        3 = striped decode (M <= 8, warps stream contiguous slot ranges),
                        4 = small-batch tensor-core kernel (M <= 32, up to 64 with G = 32;
                            persistent CTAs over (K slice, tile range) pairs),
                        5 = INT8 CUDA-core kernel for M <= 4 where path 9 does not take the
                            shape (64 columns x one K slice per CTA, paired FP32 FMAs),
                        6 = INT8 on BF16 tensor cores for 5 <= M <= 32 (codes exact in
                            BF16, fp32 activations as three exact BF16 parts),
                        7 = W8A8 integer group GEMM (GQ_ACT_I8, dp4a),
                        8 = warp-specialized W4 decode (M <= 4: a producer warp streaming
                            2 KB slots of codes with cp.async.bulk, sixteen consumer warps
                            on mma.sync),
                        9 = warp-specialized INT8 decode (M <= 4, N a multiple of 64, G of
                            32, 64 or 128: the same roles, FP32 products on CUDA cores, or
                            dp4a group dots with GQ_ACT_I8) */
  int nsplit;        /* K-slices of whole groups (1 = no split) */
  int m_tile;        /* rows of A one CTA covers */
  int n_tile;        /* output columns one CTA covers */
  int grid_x, grid_y, grid_z;
  int block_threads;
  size_t smem_bytes; /* dynamic shared memory per CTA */
  size_t workspace_bytes;
} gq_plan_t;

int gq_plan(int M, int K, int N, int G, int prec, int sm_count, gq_plan_t *plan);

/* Slice z of the split of `units` equal work units into nsplit contiguous slices, as
 * "分组量化 GEMM 内核" section 3.3 defines it: base = units / nsplit, rem = units % nsplit,
 * begin = z·base + min(z, rem), end = begin + base + (z < rem).  Host only. */
int gq_zsplit(int units, int nsplit, int z, int *begin, int *end);

/* Sticky device-side error word of the current device (0 = none; GQ_ERR_TIMEOUT after a
 * bounded wait gave up).  Reading it synchronizes the device; `clear` resets it. */
int gq_device_error(int clear);

const char *gq_status_string(int status);

/* Text describing the last GQ_ERR_CUDA returned on the calling host thread: which CUDA call
 * failed and its error name (for example "launch: cudaErrorInvalidValue").  Empty if none.
 * The string is owned by the library and valid until the thread's next failing call. */
const char *gq_last_error_detail(void);

#ifdef __cplusplus
}
#endif
#endif /* GQ_H_ */

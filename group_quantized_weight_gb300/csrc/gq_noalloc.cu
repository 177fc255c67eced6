// gq_gemm_static_scratch: gq_gemm for callers that cannot allocate device memory.
//
// Some callers must not call cudaMalloc at all: serving runtimes that reserve every byte of
// device memory up front and forbid allocation once they are running, latency-critical
// loops where an allocation (and the device synchronization that may come with it) is not
// acceptable, and embedders that route all device memory through their own allocator.
// gq_gemm would allocate its split-K scratch on first use; this entry point instead takes
// its scratch from one fixed array compiled into the library, and never allocates.
//
// The array is GQ_STATIC_SCRATCH_BYTES bytes of file-scope __device__ memory: every GPU
// that loads the library holds it until the process exits.  All calls on a device share
// it and it keeps whatever the last call left there, so calls that overlap on the GPU
// (different streams, or different host threads without ordering) race on it.
#include <mutex>

#include "gq_internal.h"

namespace gq {

static __device__ __align__(256) unsigned char g_static_scratch[GQ_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch per device, looked up once (with that device current).
static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[64];
static bool g_noalloc_ready[64];

static int static_scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GQ_ERR_NO_DEVICE; }
  if (dev < 0 || dev >= 64) return GQ_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ready[dev]) {
    void *p = nullptr;
    // In host code the array's name is only a host-side stand-in; the device address comes
    // from the runtime.
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return GQ_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
    g_noalloc_ready[dev] = true;
  }
  *out = g_noalloc_ptr[dev];
  return GQ_OK;
}

}  // namespace gq

using namespace gq;

extern "C" int gq_gemm_static_scratch(int M, int K, int N, int G, int prec, const void *A,
                                      const void *Wq, const void *scales, const void *zeros,
                                      void *out, void *stream) {
  if (prec & GQ_ACT_I8) return GQ_ERR_INVALID_ARG;   // the W8A8 entry is gq_gemm_a8
  int st = validate(M, K, N, G, prec);
  if (st != GQ_OK) return st;
  if (M == 0 || N == 0) return GQ_OK;
  if (!A || !Wq || !scales || !out) return GQ_ERR_INVALID_ARG;
  if (((prec & (GQ_ZP | GQ_ZP_FLOAT)) != 0) != (zeros != nullptr)) return GQ_ERR_INVALID_ARG;
  const uintptr_t mis = (uintptr_t)A | (uintptr_t)Wq | (uintptr_t)scales | (uintptr_t)out |
                        (uintptr_t)zeros;
  if (mis & 15u) return GQ_ERR_ALIGNMENT;
  int sms = 0;
  st = device_sm_count(&sms);
  if (st != GQ_OK) return st;
  Plan p;
  st = make_plan(M, K, N, G, prec, sms, &p);
  if (st != GQ_OK) return st;
  if (p.workspace_bytes > (size_t)GQ_STATIC_SCRATCH_BYTES) return GQ_ERR_WORKSPACE;

  void *ws = nullptr;
  if (p.workspace_bytes > 0) {
    st = static_scratch_address(&ws);
    if (st != GQ_OK) return st;
  }
  cudaStream_t s = (cudaStream_t)stream;
  unsigned *counters = (unsigned *)ws;
  float *part = ws ? (float *)((char *)ws + p.counter_bytes) : nullptr;
  // the arrival counters this plan indexes must start at zero; the array keeps the previous
  // call's contents (the kernels leave their counters at zero, but a call cut short by a
  // device-side timeout may not)
  if (launch_fault_injected()) return GQ_ERR_CUDA;
  const size_t ctr = plan_counter_bytes_used(p, M, N);
  if (ctr && cudaMemsetAsync(counters, 0, ctr, s) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  const cudaError_t e = launch_plan(p, M, K, N, G, prec, A, Wq, scales, zeros, out, part,
                                    counters, s);
  if (e != cudaSuccess) {
    note_cuda_error("launch", e);
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

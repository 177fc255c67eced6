// gq_bench: a self-contained benchmark of the library's named workloads.
//
// Everything a run needs is created here on the current device: the inputs are drawn on the
// device from a counter-based hash (no host copies of the weights), the weights are packed
// into enough rotated copies that a round of them overflows L2, and gq_gemm is timed with
// CUDA events.  The result is a JSON text in a caller buffer.  The pages report time per call
// per shape ("04 · 分组量化 GEMM 内核", section 四); the roofline figures follow the bound of
// "GPU Kernel 工程（09）：量化与融合 kernel", section 3.2 (bytes over bandwidth below the ridge,
// FLOPs over tensor throughput above it).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gq_internal.h"

namespace gq {
namespace {

// ------------------------------------------------------------------ device-side generator

// 32-bit finaliser of a 64-bit counter (splitmix64's mixing function, truncated)
__device__ __forceinline__ uint32_t mix(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return (uint32_t)((x ^ (x >> 31)) >> 32);
}
// uniform in [0, 1) with 24 random bits
__device__ __forceinline__ float unif(uint64_t seed, uint64_t i) {
  return (float)(mix(seed * 0x100000001B3ull + i) >> 8) * (1.0f / 16777216.0f);
}

__global__ void fill_bits(uint32_t *p, size_t n, uint64_t seed) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = mix(seed * 0x100000001B3ull + i);
}

// INT8 codes uniform in [-127, 127] (floor(u * 255) - 127, 24-bit u: bias below 2^-16)
__global__ void fill_i8(int8_t *p, size_t n, uint64_t seed) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = (int8_t)((int)(unif(seed, i) * 255.0f) - 127);
}

// INT4 zero points uniform in [lo, hi], eight per word
__global__ void fill_zeros(uint32_t *p, size_t n, int lo, int hi, uint64_t seed) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    uint32_t w = 0;
    for (int j = 0; j < 8; ++j) {
      const int z = lo + (int)(unif(seed, i * 8 + j) * (float)(hi - lo + 1));
      w |= (uint32_t)min(z, hi) << (4 * j);
    }
    p[i] = w;
  }
}

// reals uniform in [lo, hi] stored as fp16 (t = 0), bf16 (1) or fp32 (2)
__global__ void fill_uniform(void *p, size_t n, int t, float lo, float hi, uint64_t seed) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = lo + (hi - lo) * unif(seed, i);
    if (t == 0) reinterpret_cast<__half *>(p)[i] = __float2half_rn(v);
    else if (t == 1) reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    else reinterpret_cast<float *>(p)[i] = v;
  }
}

// activations N(0, 1) (Box-Muller on two uniforms); a fraction `frac` of them multiplied by
// `mult`; stored as bf16 (t = 1) or fp32 (2)
__global__ void fill_normal(void *p, size_t n, int t, float frac, float mult, uint64_t seed) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float u1 = unif(seed, 3 * i) + 1.0f / 33554432.0f;   // (0, 1]
    const float u2 = unif(seed, 3 * i + 1);
    float v = sqrtf(-2.0f * logf(u1)) * cospif(2.0f * u2);
    if (frac > 0.f && unif(seed, 3 * i + 2) < frac) v *= mult;
    if (t == 1) reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    else reinterpret_cast<float *>(p)[i] = v;
  }
}

// the library's own HBM peak: a 16-byte-vector copy
__global__ void copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// ------------------------------------------------------------------ host side

struct Workload {
  const char *name;
  int M, K, N, G, prec;
  float s_lo, s_hi, out_frac;
};

const Workload kWorkloads[] = {
    {"tiny_gemv", 1, 512, 512, 128, GQ_W4, 0.005f, 0.02f, 0.f},
    {"decode_gateup", 1, 4096, 28672, 128, GQ_W4, 0.005f, 0.02f, 0.001f},
    {"q8_m1", 1, 2048, 12288, 32, GQ_ACT_F32 | GQ_SC_F32 | GQ_OUT_F32, 1e-3f, 1e-2f, 0.f},
    {"q8_m32", 32, 2048, 12288, 32, GQ_ACT_F32 | GQ_SC_F32 | GQ_OUT_F32, 1e-3f, 1e-2f, 0.f},
    {"asym_m16", 16, 8192, 28672, 128, GQ_W4 | GQ_ZP | GQ_SC_BF16, 0.005f, 0.02f, 0.f},
    {"prefill", 4096, 4096, 14336, 128, GQ_W4, 0.005f, 0.02f, 0.f},
};
constexpr double kNominalBf16Tflops = 2250.0;

// every device allocation of one run, freed on every exit path
struct Arena {
  std::vector<void *> ptrs;
  ~Arena() {
    for (void *p : ptrs) cudaFree(p);
  }
  void *get(size_t bytes) {
    void *p = nullptr;
    if (cudaMalloc(&p, bytes < 16 ? 16 : bytes) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    ptrs.push_back(p);
    return p;
  }
};

double pct(std::vector<double> v, double q) {
  std::sort(v.begin(), v.end());
  const double pos = (v.size() - 1) * q / 100.0;
  const size_t lo = (size_t)pos, hi = std::min(lo + 1, v.size() - 1);
  return v[lo] + (v[hi] - v[lo]) * (pos - lo);
}

#define BENCH_CUDA(call)                          \
  do {                                            \
    const cudaError_t e_ = (call);                \
    if (e_ != cudaSuccess) {                      \
      note_cuda_error("gq_bench: " #call, e_);    \
      cudaGetLastError();                         \
      return GQ_ERR_CUDA;                         \
    }                                             \
  } while (0)

// Copy bandwidth of this device (read + write bytes per second), measured once per process.
int hbm_copy_gbs(double *gbs) {
  static double cached = 0.0;
  if (cached > 0.0) {
    *gbs = cached;
    return GQ_OK;
  }
  const size_t bytes = (size_t)1 << 30;
  Arena ar;
  void *a = ar.get(bytes), *b = ar.get(bytes);
  if (!a || !b) return GQ_ERR_CUDA;
  int sms = 0;
  int st = device_sm_count(&sms);
  if (st != GQ_OK) return st;
  cudaEvent_t e0, e1;
  BENCH_CUDA(cudaEventCreate(&e0));
  BENCH_CUDA(cudaEventCreate(&e1));
  BENCH_CUDA(cudaMemset(a, 1, bytes));
  float best = 1e30f;
  for (int r = 0; r < 6; ++r) {
    cudaEventRecord(e0, 0);
    copy_kernel<<<sms * 4, 512>>>((const uint4 *)a, (uint4 *)b, bytes / 16);
    cudaEventRecord(e1, 0);
    BENCH_CUDA(cudaEventSynchronize(e1));
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    if (r > 0) best = std::min(best, ms);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  BENCH_CUDA(cudaGetLastError());
  cached = 2.0 * bytes / (best * 1e-3) / 1e9;
  *gbs = cached;
  return GQ_OK;
}

int run_one(const Workload &w, std::string &json) {
  const int M = w.M, K = w.K, N = w.N, G = w.G, prec = w.prec | GQ_STATIC_W;
  const bool w4 = (w.prec & GQ_W4) != 0, zp = (w.prec & GQ_ZP) != 0;
  const int sc_t = (w.prec & GQ_SC_F32) ? 2 : (w.prec & GQ_SC_BF16) ? 1 : 0;
  const size_t es_sc = sc_t == 2 ? 4 : 2, es_act = (w.prec & GQ_ACT_F32) ? 4 : 2;
  const size_t es_out = (w.prec & GQ_OUT_F32) ? 4 : 2;
  const int ng = K / G;
  const size_t codes_b = w4 ? (size_t)K / 8 * N * 4 : (size_t)K * N;
  const size_t sc_b = (size_t)ng * N * es_sc, z_b = zp ? (size_t)ng * (N / 8) * 4 : 0;
  size_t packed_b = 0;
  int st = gq_packed_bytes(K, N, G, prec, &packed_b);
  if (st != GQ_OK) return st;
  int dev = 0, l2 = 0, sms = 0;
  BENCH_CUDA(cudaGetDevice(&dev));
  BENCH_CUDA(cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev));
  st = device_sm_count(&sms);
  if (st != GQ_OK) return st;
  const bool big = M >= 128;
  const size_t wbytes = packed_b + sc_b + z_b;
  // one round of the copies overflows L2 twice over: ceil(2 L2 / bytes) + 1, at most 16
  const int copies = big ? 1 : (int)std::min<size_t>(16, (2 * (size_t)l2 + wbytes - 1) / wbytes + 1);

  Arena ar;
  void *A = ar.get((size_t)M * K * es_act), *codes = ar.get(codes_b);
  void *out0 = ar.get((size_t)M * N * es_out), *out1 = ar.get((size_t)M * N * es_out);
  if (!A || !codes || !out0 || !out1) return GQ_ERR_CUDA;
  std::vector<void *> Wc(copies), Sc(copies), Zc(copies, nullptr);
  for (int c = 0; c < copies; ++c) {
    Wc[c] = ar.get(packed_b);
    Sc[c] = ar.get(sc_b);
    if (zp) Zc[c] = ar.get(z_b);
    if (!Wc[c] || !Sc[c] || (zp && !Zc[c])) return GQ_ERR_CUDA;
  }
  cudaStream_t s = nullptr;
  BENCH_CUDA(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
  struct StreamGuard {
    cudaStream_t s;
    ~StreamGuard() { cudaStreamDestroy(s); }
  } sg{s};
  const int grid = sms * 4;
  const uint64_t seed = 0x6751u;
  if (w4) fill_bits<<<grid, 256, 0, s>>>((uint32_t *)codes, codes_b / 4, seed + 1);
  else fill_i8<<<grid, 256, 0, s>>>((int8_t *)codes, codes_b, seed + 1);
  fill_uniform<<<grid, 256, 0, s>>>(Sc[0], (size_t)ng * N, sc_t, w.s_lo, w.s_hi, seed + 2);
  if (zp) fill_zeros<<<grid, 256, 0, s>>>((uint32_t *)Zc[0], z_b / 4, 4, 11, seed + 3);
  fill_normal<<<grid, 256, 0, s>>>(A, (size_t)M * K, es_act == 4 ? 2 : 1, w.out_frac, 50.f, seed + 4);
  BENCH_CUDA(cudaGetLastError());
  for (int c = 0; c < copies; ++c) {
    st = gq_pack_weights(K, N, G, prec, codes, Wc[c], s);
    if (st != GQ_OK) return st;
    if (c > 0) {
      BENCH_CUDA(cudaMemcpyAsync(Sc[c], Sc[0], sc_b, cudaMemcpyDeviceToDevice, s));
      if (zp) BENCH_CUDA(cudaMemcpyAsync(Zc[c], Zc[0], z_b, cudaMemcpyDeviceToDevice, s));
    }
  }
  auto call = [&](int i, void *out) {
    const int c = i % copies;
    return gemm_impl(M, K, N, G, prec, A, Wc[c], Sc[c], Zc[c], out, s);
  };
  // warm-up (creates the library's scratch outside any capture), then two calls whose bits
  // must agree
  for (int i = 0; i < 3; ++i)
    if ((st = call(i, out0)) != GQ_OK) return st;
  if ((st = call(0, out0)) != GQ_OK || (st = call(0, out1)) != GQ_OK) return st;
  BENCH_CUDA(cudaStreamSynchronize(s));
  std::vector<unsigned char> h0((size_t)M * N * es_out), h1(h0.size());
  BENCH_CUDA(cudaMemcpy(h0.data(), out0, h0.size(), cudaMemcpyDeviceToHost));
  BENCH_CUDA(cudaMemcpy(h1.data(), out1, h1.size(), cudaMemcpyDeviceToHost));
  const bool deterministic = memcmp(h0.data(), h1.data(), h0.size()) == 0;

  cudaEvent_t e0, e1;
  BENCH_CUDA(cudaEventCreate(&e0));
  BENCH_CUDA(cudaEventCreate(&e1));
  struct EventGuard {
    cudaEvent_t a, b;
    ~EventGuard() {
      cudaEventDestroy(a);
      cudaEventDestroy(b);
    }
  } eg{e0, e1};
  const int iters = big ? 10 : 200;
  std::vector<double> rep_us;
  if (!big) {
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ge = nullptr;
    BENCH_CUDA(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
    int cst = GQ_OK;
    for (int i = 0; i < iters && cst == GQ_OK; ++i) cst = call(i, out0);
    const cudaError_t ec = cudaStreamEndCapture(s, &g);
    if (cst != GQ_OK) {
      if (g) cudaGraphDestroy(g);
      return cst;
    }
    BENCH_CUDA(ec);
    struct GraphGuard {
      cudaGraph_t g;
      cudaGraphExec_t *ge;
      ~GraphGuard() {
        if (*ge) cudaGraphExecDestroy(*ge);
        cudaGraphDestroy(g);
      }
    } gg{g, &ge};
    BENCH_CUDA(cudaGraphInstantiate(&ge, g, 0));
    BENCH_CUDA(cudaGraphLaunch(ge, s));
    for (int r = 0; r < 5; ++r) {
      BENCH_CUDA(cudaEventRecord(e0, s));
      BENCH_CUDA(cudaGraphLaunch(ge, s));
      BENCH_CUDA(cudaEventRecord(e1, s));
      BENCH_CUDA(cudaEventSynchronize(e1));
      float ms = 0.f;
      BENCH_CUDA(cudaEventElapsedTime(&ms, e0, e1));
      rep_us.push_back(1e3 * ms / iters);
    }
  } else {
    for (int r = 0; r < 5; ++r) {
      BENCH_CUDA(cudaEventRecord(e0, s));
      for (int i = 0; i < iters; ++i)
        if ((st = call(i, out0)) != GQ_OK) return st;
      BENCH_CUDA(cudaEventRecord(e1, s));
      BENCH_CUDA(cudaEventSynchronize(e1));
      float ms = 0.f;
      BENCH_CUDA(cudaEventElapsedTime(&ms, e0, e1));
      rep_us.push_back(1e3 * ms / iters);
    }
  }
  // single host-launched calls, each alone on an idle device
  std::vector<double> single;
  for (int i = 0; i < 12; ++i) {
    BENCH_CUDA(cudaStreamSynchronize(s));
    BENCH_CUDA(cudaEventRecord(e0, s));
    if ((st = call(i, out0)) != GQ_OK) return st;
    BENCH_CUDA(cudaEventRecord(e1, s));
    BENCH_CUDA(cudaEventSynchronize(e1));
    float ms = 0.f;
    BENCH_CUDA(cudaEventElapsedTime(&ms, e0, e1));
    if (i >= 2) single.push_back(1e3 * ms);
  }
  BENCH_CUDA(cudaStreamSynchronize(s));

  const double us = pct(rep_us, 50.0);
  const double bytes = (double)(w4 ? (size_t)K * N / 2 : (size_t)K * N) + (double)sc_b +
                       (double)z_b + (double)M * K * es_act + (double)M * N * es_out;
  const double gbs = bytes / (us * 1e-6) / 1e9;
  const double tflops = 2.0 * M * (double)N * K / (us * 1e-6) / 1e12;
  double peak = 0.0;
  const char *bound = big ? "tensor" : "hbm";
  const char *peak_src = big ? "nominal dense BF16 (2250 TFLOPS)" : "own 1 GiB copy kernel";
  if (big) {
    peak = kNominalBf16Tflops;
  } else if ((st = hbm_copy_gbs(&peak)) != GQ_OK) {
    return st;
  }
  Plan pl;
  st = make_plan(M, K, N, G, prec, sms, &pl);
  if (st != GQ_OK) return st;
  char buf[1024];
  snprintf(buf, sizeof(buf),
           "{\"config\": \"%s\", \"M\": %d, \"K\": %d, \"N\": %d, \"G\": %d, \"prec\": %d, "
           "\"path\": %d, \"nsplit\": %d, \"us_median\": %.4f, \"us_p10\": %.4f, "
           "\"us_p90\": %.4f, \"us_single_call\": %.4f, \"repeats\": %d, "
           "\"calls_per_repeat\": %d, \"graph\": %s, \"algorithmic_bytes\": %.0f, "
           "\"GB/s\": %.2f, \"TFLOPS\": %.3f, \"bound\": \"%s\", \"peak\": %.1f, "
           "\"peak_unit\": \"%s\", \"peak_source\": \"%s\", \"frac\": %.4f, "
           "\"launches_per_call\": 1, \"weight_copies\": %d, \"deterministic\": %s}",
           w.name, M, K, N, G, prec, pl.path, pl.nsplit, us, pct(rep_us, 10.0),
           pct(rep_us, 90.0), pct(single, 50.0), (int)rep_us.size(), iters,
           big ? "false" : "true", bytes, gbs, tflops, bound, peak, big ? "TFLOP/s" : "GB/s",
           peak_src, big ? tflops / peak : gbs / peak, copies,
           deterministic ? "true" : "false");
  json = buf;
  return GQ_OK;
}

}  // namespace
}  // namespace gq

using namespace gq;

extern "C" int gq_bench(const char *config, char *json_out, size_t cap) {
  if (!config || !json_out || cap == 0) return GQ_ERR_INVALID_ARG;
  json_out[0] = '\0';
  std::vector<const Workload *> todo;
  for (const Workload &w : kWorkloads)
    if (strcmp(config, "all") == 0 || strcmp(config, w.name) == 0) todo.push_back(&w);
  if (todo.empty()) return GQ_ERR_INVALID_ARG;
  int sms = 0;
  int st = device_sm_count(&sms);
  if (st != GQ_OK) return st;
  std::string all = todo.size() > 1 ? "[" : "";
  for (size_t i = 0; i < todo.size(); ++i) {
    std::string one;
    st = run_one(*todo[i], one);
    if (st != GQ_OK) return st;
    if (i) all += ", ";
    all += one;
  }
  if (todo.size() > 1) all += "]";
  if (all.size() + 1 > cap) return GQ_ERR_INVALID_ARG;
  memcpy(json_out, all.c_str(), all.size() + 1);
  return GQ_OK;
}

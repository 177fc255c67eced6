// Host access to cuTensorMapEncodeTiled (internal).  It is a driver-API call, fetched through
// the runtime so that the library does not link libcuda directly (it then still loads on a
// machine without a driver).
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>

namespace gq {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The encoder, or nullptr when the driver does not provide it.
inline EncodeTiledFn tensor_map_encoder() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load();
  if (f) return f;
  void *p = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !p) {
    cudaGetLastError();
    return nullptr;
  }
  f = reinterpret_cast<EncodeTiledFn>(p);
  fn.store(f);
  return f;
}

}  // namespace gq

// mla_tmap.cuh -- host side: the driver's tensor-map encoder (cuTensorMapEncodeTiled),
// looked up once through the runtime's driver entry-point query, so that the library links
// against the CUDA runtime only.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace mla {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// nullptr when the driver does not provide it (the static is initialised once, thread-safely)
inline EncodeTiledFn tmap_encode_fn() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(f);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

}  // namespace mla

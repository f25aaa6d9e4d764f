// Host-side TMA tensor-map encoding. The driver entry point is fetched
// through the runtime (no link against libcuda).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace nys {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tiled map over a row-major tensor of `rank` dims (dims[0] innermost,
// strides in bytes for dims 1..rank-1), box `box` elements per dim, zero
// fill out of bounds. Returns false if encoding fails.
inline bool make_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                            const uint64_t* dims, const uint64_t* strides_bytes,
                            const uint32_t* box, CUtensorMapSwizzle swizzle) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  uint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                   reinterpret_cast<const cuuint64_t*>(dims),
                   reinterpret_cast<const cuuint64_t*>(strides_bytes),
                   reinterpret_cast<const cuuint32_t*>(box),
                   reinterpret_cast<const cuuint32_t*>(elem_strides),
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace nys

// Host helper: TMA tensor maps (cuTensorMapEncodeTiled, reached through the runtime's driver
// entry-point query so the library needs no link against the driver library).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace moe {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A rank-r tiled map: dims[0] is the contiguous dimension (in elements), strides[i] the byte
// stride of dimension i + 1, box the tile copied per instruction.  False when the encoder is
// missing or refuses the description.
inline bool make_tensor_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr,
                            const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                            CUtensorMapSwizzle sw) {
  auto fn = tensor_map_encoder();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides[i];
  }
  return fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
            sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe

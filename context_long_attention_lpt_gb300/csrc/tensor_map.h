// Host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled through the
// runtime's driver entry point, so the library needs no link against libcuda).
#pragma once

#include <cstdint>

#include <cuda.h>

namespace splitkv {

// Encodes a 3-D tiled map of bf16 elements.  dims[0] is innermost;
// strides_bytes[i] is the byte stride of dims[i+1].  Returns 0 on success or
// a negative SPLITKV_ERR_* status (message recorded for splitkv_last_error).
int encode_bf16_3d(CUtensorMap* map, const void* base, const uint64_t dims[3],
                   const uint64_t strides_bytes[2], const uint32_t box[3],
                   CUtensorMapSwizzle swizzle);

}  // namespace splitkv

// Device helpers shared by the split-KV kernels.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "work_layout.h"

namespace splitkv {

// Read-only view of the work descriptor in device memory.
struct WorkView {
  const int32_t* w;
  __device__ __forceinline__ explicit WorkView(const int32_t* p) : w(p) {}
  __device__ __forceinline__ int32_t hdr(int i) const { return __ldg(w + i); }
  __device__ __forceinline__ const int32_t* item(int32_t i) const {
    return w + hdr(kOffItems) + kItemWords * static_cast<int64_t>(i);
  }
  __device__ __forceinline__ const int32_t* seq(int32_t b) const {
    return w + hdr(kOffSeq) + kSeqWords * static_cast<int64_t>(b);
  }
  __device__ __forceinline__ const int32_t* blocks() const { return w + hdr(kOffBlocks); }
  __device__ __forceinline__ const int32_t* seq_items() const { return w + hdr(kOffSeqItems); }
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Keys of a sequence that query token t sees: [0, visible).
__device__ __forceinline__ int32_t visible_keys(int32_t q_len, int32_t kv_len, int32_t t,
                                                int32_t causal) {
  return causal ? kv_len - q_len + t + 1 : kv_len;
}

}  // namespace splitkv

// Device helpers shared by the split-KV kernels.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "work_layout.h"

namespace splitkv {

// Read-only view of the work descriptor in device memory.  The sequence rows, item
// rows and block lists sit at offsets fixed by B and n_items (work_layout.h), so
// finding an item's row takes no load; only the per-sequence item lists, placed
// after the block lists, are found through the header.
struct WorkView {
  const int32_t* w;
  const int32_t* items_;
  const int32_t* blocks_;
  __device__ __forceinline__ WorkView(const int32_t* p, int32_t B, int32_t n_items)
      : w(p), items_(p + work_off_items(B)), blocks_(p + work_off_blocks(B, n_items)) {}
  // for the merges, which read sequence and item rows but no block list
  __device__ __forceinline__ WorkView(const int32_t* p, int32_t B)
      : w(p), items_(p + work_off_items(B)), blocks_(nullptr) {}
  __device__ __forceinline__ int32_t hdr(int i) const { return __ldg(w + i); }
  __device__ __forceinline__ const int32_t* item(int32_t i) const {
    return items_ + kItemWords * static_cast<int64_t>(i);
  }
  __device__ __forceinline__ const int32_t* seq(int32_t b) const {
    return w + work_off_seq() + kSeqWords * static_cast<int64_t>(b);
  }
  __device__ __forceinline__ const int32_t* blocks() const { return blocks_; }
  __device__ __forceinline__ const int32_t* seq_items() const { return w + hdr(kOffSeqItems); }
};

// Status bit: the work descriptor was not built for the launch's B and n_items (its
// magic word, B or n_items differ); the launch's CTAs did nothing.
constexpr unsigned int kStatusBadWork = 8u;

// Whether a descriptor header (magic word, B, n_items, loaded by the caller alongside
// the item row, not before it) belongs to a launch over B sequences and n_items items.
__device__ __forceinline__ bool work_matches(int32_t magic, int32_t b, int32_t n, int32_t B, int32_t n_items) {
  return magic == kWorkMagic && b == B && n == n_items;
}

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

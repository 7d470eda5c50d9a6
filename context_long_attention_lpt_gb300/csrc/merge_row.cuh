// One (query row, query head) of the exact merge, computed by one warp.  Used by
// the merge kernel and by the tensor-core kernel's in-launch merge, so both
// give the same bits.
//
// The Split-KV card ("All Facts") states the sharded result equals the
// unsharded one.  With L = ln sum_i exp(L_i) over the shards i holding keys of
// the row's sequence and w_i = exp(L_i - L), the unsharded output is
// O = sum_i w_i O_i, because each O_i is the softmax mean over shard i's keys and
// exp(L_i) is that shard's share of the full denominator.
//
// Lanes first load the shards' L_i (one per lane, strided), reduce max and sum
// with warp shuffles, then stream the O_i rows with each lane owning D/32
// contiguous floats, so a warp reads each partial row as one coalesced 512 B
// (D = 128) transaction, eight partial rows in flight.
#pragma once

#include <cmath>

#include "device_common.cuh"

namespace splitkv {

template <int N>
struct Vec {
  float v[N];
};

// kCoherent: the partials were written by other CTAs of the same launch, so they
// are read through L2 only; otherwise through the read-only path.
template <bool kCoherent>
__device__ __forceinline__ float load_f32(const float* src) {
  if constexpr (kCoherent) return __ldcg(src);
  return __ldg(src);
}

template <int N, bool kCoherent>
__device__ __forceinline__ Vec<N> load_vec(const float* src) {
  Vec<N> r;
  if constexpr (N == 4) {
    const float4 x = kCoherent ? __ldcg(reinterpret_cast<const float4*>(src))
                               : __ldg(reinterpret_cast<const float4*>(src));
    r.v[0] = x.x; r.v[1] = x.y; r.v[2] = x.z; r.v[3] = x.w;
  } else if constexpr (N == 2) {
    const float2 x = kCoherent ? __ldcg(reinterpret_cast<const float2*>(src))
                               : __ldg(reinterpret_cast<const float2*>(src));
    r.v[0] = x.x; r.v[1] = x.y;
  } else {
#pragma unroll
    for (int k = 0; k < N; ++k) r.v[k] = load_f32<kCoherent>(src + k);
  }
  return r;
}

// A zero weight (a shard with no visible key for this row) contributes nothing,
// whatever its partial row holds.
template <int N>
__device__ __forceinline__ void accumulate(float (&acc)[N], float w, const Vec<N>& x) {
#pragma unroll
  for (int k = 0; k < N; ++k) acc[k] = w != 0.f ? fmaf(w, x.v[k], acc[k]) : acc[k];
}

// Merges token t of a sequence whose items are seq_items[p0 .. p1) for query
// head h into out[gw] (D values) and lse_out[gw].  Whole warp, converged.
template <typename OutT, int D, bool kCoherent>
__device__ __forceinline__ void merge_row(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                                          const WorkView& wv, int32_t p0, int32_t p1, int32_t t, int32_t h,
                                          int32_t Hq, int64_t gw, OutT* __restrict__ out,
                                          float* __restrict__ lse_out) {
  constexpr int kPer = D / 32;
  constexpr int kUnroll = 8;
  const int lane = threadIdx.x & 31;
  const int32_t* seq_items = wv.seq_items();
  // pass 1: max of the shards' LSE values
  float m = -INFINITY;
  for (int32_t i = p0 + lane; i < p1; i += 32) {
    const int32_t pr = __ldg(wv.item(__ldg(seq_items + i)) + kItPartRow);
    m = fmaxf(m, load_f32<kCoherent>(lse_part + static_cast<int64_t>(pr + t) * Hq + h));
  }
  m = warp_max(m);
  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  float denom = 0.f;
  if (m != -INFINITY) {
    for (int32_t base = p0; base < p1; base += 32) {
      const int32_t i = base + lane;
      int64_t my_row = 0;
      float my_w = 0.f;
      if (i < p1) {
        const int32_t pr = __ldg(wv.item(__ldg(seq_items + i)) + kItPartRow);
        my_row = static_cast<int64_t>(pr + t) * Hq + h;
        my_w = expf(load_f32<kCoherent>(lse_part + my_row) - m);  // 0 for an empty shard
      }
      denom += my_w;
      const int n = min(32, p1 - base);
      // Eight partial rows per round: all eight loads are issued before the
      // first FMA, so a warp has eight independent 512 B reads in flight.
      int k2 = 0;
      for (; k2 + kUnroll <= n; k2 += kUnroll) {
        Vec<kPer> x[kUnroll];
        float w[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          w[u] = __shfl_sync(0xffffffffu, my_w, k2 + u);
          const int64_t r = __shfl_sync(0xffffffffu, my_row, k2 + u);
          x[u] = load_vec<kPer, kCoherent>(o_part + r * D + lane * kPer);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) accumulate(acc, w[u], x[u]);
      }
      for (; k2 < n; ++k2) {
        const float w = __shfl_sync(0xffffffffu, my_w, k2);
        const int64_t r = __shfl_sync(0xffffffffu, my_row, k2);
        accumulate(acc, w, load_vec<kPer, kCoherent>(o_part + r * D + lane * kPer));
      }
    }
    denom = warp_sum(denom);
  }
  const float inv = denom > 0.f ? 1.f / denom : 0.f;
  OutT* dst = out + gw * D + lane * kPer;
#pragma unroll
  for (int k = 0; k < kPer; ++k) dst[k] = from_f32<OutT>(acc[k] * inv);
  if (lane == 0) lse_out[gw] = denom > 0.f ? m + logf(denom) : -INFINITY;
}

}  // namespace splitkv

// Exact merge of per-shard partials, one warp per (query row, query head).
//
// The Split-KV card ("All Facts") states the sharded result equals the
// unsharded one.  With L = ln sum_i exp(L_i) over the shards i holding keys of
// the row's sequence and w_i = exp(L_i - L), the unsharded output is
// O = sum_i w_i O_i, because each O_i is the softmax mean over shard i's keys and
// exp(L_i) is that shard's share of the full denominator.  Only query-sized
// tensors are read (card intro: communication decoupled from context length).
//
// Lanes first load the shards' L_i (one per lane, strided), reduce max and sum
// with warp shuffles, then stream the O_i rows with each lane owning D/32
// contiguous floats, so a warp reads each partial row as one coalesced 512 B
// (D = 128) transaction.

#include <cmath>

#include "device_common.cuh"
#include "launch.h"

namespace splitkv {
namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 8;

template <int N>
struct Vec {
  float v[N];
};

template <int N>
__device__ __forceinline__ Vec<N> load_vec(const float* src) {
  Vec<N> r;
  if constexpr (N == 4) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(src));
    r.v[0] = x.x; r.v[1] = x.y; r.v[2] = x.z; r.v[3] = x.w;
  } else if constexpr (N == 2) {
    const float2 x = __ldg(reinterpret_cast<const float2*>(src));
    r.v[0] = x.x; r.v[1] = x.y;
  } else {
#pragma unroll
    for (int k = 0; k < N; ++k) r.v[k] = __ldg(src + k);
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

template <typename OutT, int D>
__global__ void __launch_bounds__(kWarps * 32, 1)
    merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                 int64_t part_rows, const int32_t* __restrict__ work, int32_t B, int32_t total_q,
                 int32_t Hq, OutT* __restrict__ out, float* __restrict__ lse_out,
                 unsigned int* status) {
  constexpr int kPer = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (gw >= static_cast<int64_t>(total_q) * Hq) return;
  const int32_t row = static_cast<int32_t>(gw / Hq);
  const int32_t h = static_cast<int32_t>(gw % Hq);

  const WorkView wv(work);
  // sequence of this row: last b with cu_q[b] <= row
  int32_t lo = 0, hi = B - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (__ldg(wv.seq(mid) + kSqCuQ) <= row) lo = mid; else hi = mid - 1;
  }
  const int32_t b = lo;
  const int32_t t = row - __ldg(wv.seq(b) + kSqCuQ);
  const int32_t p0 = __ldg(wv.seq(b) + kSqItemPtr), p1 = __ldg(wv.seq(b + 1) + kSqItemPtr);
  const int32_t* seq_items = wv.seq_items();
  // every partial row this warp reads must lie inside the buffers
  bool bad = false;
  for (int32_t i = p0 + lane; i < p1; i += 32) {
    const int32_t pr = __ldg(wv.item(__ldg(seq_items + i)) + kItPartRow);
    bad |= pr < 0 || static_cast<int64_t>(pr) + t >= part_rows;
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) atomicOr(status, 2u);
    return;
  }

  // pass 1: max and sum of the shards' LSE values
  float m = -INFINITY;
  for (int32_t i = p0 + lane; i < p1; i += 32) {
    const int32_t pr = __ldg(wv.item(__ldg(seq_items + i)) + kItPartRow);
    m = fmaxf(m, __ldg(lse_part + static_cast<int64_t>(pr + t) * Hq + h));
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
        my_w = expf(__ldg(lse_part + my_row) - m);  // 0 for an empty shard
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
          x[u] = load_vec<kPer>(o_part + r * D + lane * kPer);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) accumulate(acc, w[u], x[u]);
      }
      for (; k2 < n; ++k2) {
        const float w = __shfl_sync(0xffffffffu, my_w, k2);
        const int64_t r = __shfl_sync(0xffffffffu, my_row, k2);
        accumulate(acc, w, load_vec<kPer>(o_part + r * D + lane * kPer));
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

template <typename OutT, int D>
cudaError_t launch_typed(const float* o_part, const float* lse_part, int64_t part_rows,
                         const int32_t* work, int32_t B, int32_t total_q, int32_t Hq, void* out,
                         float* lse_out, unsigned int* status, cudaStream_t stream) {
  const int64_t warps = static_cast<int64_t>(total_q) * Hq;
  if (warps == 0) return cudaSuccess;
  const int64_t grid = (warps + kWarps - 1) / kWarps;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  merge_kernel<OutT, D><<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(
      o_part, lse_part, part_rows, work, B, total_q, Hq, static_cast<OutT*>(out), lse_out, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const float* o_part, const float* lse_part, int64_t part_rows,
                         const int32_t* work, int32_t B, int32_t total_q, int32_t Hq, int32_t d,
                         int32_t dtype, void* out, float* lse_out, unsigned int* status,
                         cudaStream_t stream) {
#define SPLITKV_MERGE_ARGS o_part, lse_part, part_rows, work, B, total_q, Hq, out, lse_out, status, stream
  if (dtype == SPLITKV_F32)
    return d == 64 ? launch_typed<float, 64>(SPLITKV_MERGE_ARGS) : launch_typed<float, 128>(SPLITKV_MERGE_ARGS);
  return d == 64 ? launch_typed<__nv_bfloat16, 64>(SPLITKV_MERGE_ARGS)
                 : launch_typed<__nv_bfloat16, 128>(SPLITKV_MERGE_ARGS);
#undef SPLITKV_MERGE_ARGS
}

}  // namespace splitkv

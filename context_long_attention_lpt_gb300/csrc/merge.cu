// Exact merge of per-shard partials, one warp per (query row, query head).
//
// The per-row arithmetic (Split-KV card, "All Facts": the sharded result equals
// the unsharded one) is merge_row in merge_row.cuh, shared with the
// tensor-core kernel's in-launch merge.  Only query-sized tensors are read
// (card intro: communication decoupled from context length).

#include <cmath>

#include "device_common.cuh"
#include "launch.h"
#include "merge_row.cuh"

namespace splitkv {
namespace {

constexpr int kWarps = 8;

template <typename OutT, int D>
__global__ void __launch_bounds__(kWarps * 32, 1)
    merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                 int64_t part_rows, const int32_t* __restrict__ work, int32_t B, int32_t total_q,
                 int32_t Hq, OutT* __restrict__ out, float* __restrict__ lse_out,
                 unsigned int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (gw >= static_cast<int64_t>(total_q) * Hq) return;
  const int32_t row = static_cast<int32_t>(gw / Hq);
  const int32_t h = static_cast<int32_t>(gw % Hq);

  const WorkView wv(work, B);
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

  merge_row<OutT, D, false>(o_part, lse_part, wv, p0, p1, t, h, Hq, gw, out, lse_out);
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

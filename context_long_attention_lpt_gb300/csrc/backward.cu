// Split-KV backward pass on CUDA cores: D = rowsum(dO * O), per-shard dK / dV
// and partial dQ, and the dQ reduction over shards.
//
// The Split-KV card presents the method for training ("asymmetric training
// scenarios with very short queries and very long contexts", card intro) and
// as exact ("All Facts").  With the merged forward's O and L, a shard needs
// only query-sized tensors (Q, dO, L, D) to produce the exact gradients of its
// own keys and a query-sized partial dQ; the partials of all shards holding a
// sequence's keys sum to its dQ - the backward counterpart of the forward merge.
//
// Chain rule through s = scale*q.k, P = exp(s - L), O = P V, for every query
// row r (each query head of the K/V head's group) and visible key j:
//   dV_j += P_rj dO_r,  dP_rj = dO_r . V_j,  dS_rj = P_rj (dP_rj - D_r),
//   dQ_r += scale dS_rj K_j,  dK_j += scale dS_rj Q_r.
//
// One CTA owns one (work item, K/V head, 16-key tile): it keeps the tile's K,
// V and its dK, dV accumulators while it walks every query row of the
// sequence in 16-row tiles, so dK / dV need no atomics; the dQ contributions of
// different key tiles of the same item meet in fp32 atomic adds on the item's
// partial dQ rows.

#include <cmath>

#include "device_common.cuh"
#include "launch.h"
#include "status.h"

namespace splitkv {
namespace {

constexpr int kRows = 16;      // query rows per inner tile
constexpr int kKeys = 16;      // keys per CTA tile (keeps the shared tiles under 48 KB)
constexpr int kThreads = 128;
constexpr int kTilesY = 16;    // CTAs per (item, K/V head); each strides over the item's key tiles

template <typename T>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                      int64_t n_rows, int32_t d, float* __restrict__ delta) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (r >= n_rows) return;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) s = fmaf(to_f32(o[r * d + c]), to_f32(dout[r * d + c]), s);
  s = warp_sum(s);
  if (lane == 0) delta[r] = s;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    bwd_partial_kernel(PartialArgs a, const T* __restrict__ dout, const float* __restrict__ lse,
                       const float* __restrict__ delta, float* __restrict__ dq_part, float* __restrict__ dk_pool,
                       float* __restrict__ dv_pool) {
  constexpr int kOwnKV = kKeys * D / kThreads;  // dK / dV elements per thread
  constexpr int kOwnQ = kRows * D / kThreads;   // dQ elements per thread per row tile
  __shared__ float k_s[kKeys][D + 1];
  __shared__ float v_s[kKeys][D + 1];
  __shared__ float q_s[kRows][D + 1];
  __shared__ float do_s[kRows][D + 1];
  __shared__ float p_s[kRows][kKeys + 1];
  __shared__ float ds_s[kRows][kKeys + 1];
  __shared__ float l_s[kRows], dl_s[kRows];
  __shared__ int32_t vis_s[kRows];

  const int tid = threadIdx.x;
  const int32_t item = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv;
  const WorkView wv(a.work, a.B, a.n_items);
  const int32_t* it = wv.item(item);
  const int32_t h_magic = wv.hdr(kMagic), h_b = wv.hdr(kB), h_n = wv.hdr(kNItems);
  const int32_t seq = __ldg(it + kItSeq);
  const int32_t blk_off = __ldg(it + kItBlockOff), blk_cnt = __ldg(it + kItBlockCnt);
  const int32_t part_row = __ldg(it + kItPartRow);
  const int32_t cu_q = __ldg(it + kItCuQ), q_len = __ldg(it + kItQLen), kv_len = __ldg(it + kItKvLen);
  if (!work_matches(h_magic, h_b, h_n, a.B, a.n_items)) {
    if (tid == 0) atomicOr(a.status, kStatusBadWork);
    return;
  }
  const int32_t G = a.Hq / a.Hkv;
  const int32_t rows = q_len * G;
  if (rows == 0) return;
  if (part_row < 0 || static_cast<int64_t>(part_row) + q_len > a.part_rows) {
    if (tid == 0) atomicOr(a.status, 2u);
    return;
  }
  const T* q = static_cast<const T*>(a.q);
  const T* kp = static_cast<const T*>(a.k_pool);
  const T* vp = static_cast<const T*>(a.v_pool);
  const int32_t bl = a.block_len;
  const int32_t tiles_per_block = (bl + kKeys - 1) / kKeys;
  const int32_t n_tiles = blk_cnt * tiles_per_block;

  for (int32_t tile = blockIdx.y; tile < n_tiles; tile += gridDim.y) {
    const int32_t j = __ldg(wv.blocks() + blk_off + tile / tiles_per_block);
    const int32_t key0 = j * bl + (tile % tiles_per_block) * kKeys;          // position of the tile's first key
    const int32_t nk = min(kKeys, min(kv_len, (j + 1) * bl) - key0);         // keys of the tile in the sequence
    if (nk <= 0) continue;
    if (j >= a.max_blocks_per_seq) {
      if (tid == 0) atomicOr(a.status, 1u);
      continue;
    }
    const int32_t phys = __ldg(a.block_table + static_cast<int64_t>(seq) * a.max_blocks_per_seq + j);
    if (phys < 0 || phys >= a.n_pool_blocks) {
      if (tid == 0) atomicOr(a.status, 1u);
      continue;
    }
    const int64_t tok0 = static_cast<int64_t>(phys) * bl + (key0 - j * bl);
    __syncthreads();  // the previous tile's shared data is no longer read
    for (int i = tid; i < kKeys * D; i += kThreads) {
      const int kk = i / D, c = i % D;
      float kx = 0.f, vx = 0.f;
      if (kk < nk) {
        const int64_t gi = ((tok0 + kk) * a.Hkv + kvh) * D + c;
        kx = to_f32(kp[gi]);
        vx = to_f32(vp[gi]);
      }
      k_s[kk][c] = kx;
      v_s[kk][c] = vx;
    }
    float dk[kOwnKV], dv[kOwnKV];
#pragma unroll
    for (int m = 0; m < kOwnKV; ++m) dk[m] = dv[m] = 0.f;

    // rows whose token sees the tile's first key: token >= key0 - (kv_len - q_len) when causal
    const int32_t first_tok = a.causal ? max(0, key0 - (kv_len - q_len)) : 0;
    for (int32_t r0 = first_tok * G; r0 < rows; r0 += kRows) {
      const int32_t n_r = min(kRows, rows - r0);
      __syncthreads();
      for (int i = tid; i < kRows * D; i += kThreads) {
        const int r = i / D, c = i % D;
        float qx = 0.f, dx = 0.f;
        if (r < n_r) {
          const int32_t row = r0 + r;
          const int64_t qi = (static_cast<int64_t>(cu_q + row / G) * a.Hq + kvh * G + row % G) * D + c;
          qx = to_f32(q[qi]);
          dx = to_f32(dout[qi]);
        }
        q_s[r][c] = qx;
        do_s[r][c] = dx;
      }
      if (tid < kRows) {
        float lv = -INFINITY, dlv = 0.f;
        int32_t vis = 0;
        if (tid < n_r) {
          const int32_t row = r0 + tid;
          const int64_t ri = static_cast<int64_t>(cu_q + row / G) * a.Hq + kvh * G + row % G;
          lv = lse[ri];
          dlv = delta[ri];
          vis = visible_keys(q_len, kv_len, row / G, a.causal);
        }
        l_s[tid] = lv;
        dl_s[tid] = dlv;
        vis_s[tid] = vis;
      }
      __syncthreads();
      // P and dS for the 16 x 16 block
      for (int i = tid; i < kRows * kKeys; i += kThreads) {
        const int r = i / kKeys, kk = i % kKeys;
        float p = 0.f, ds = 0.f;
        if (r < n_r && kk < nk && key0 + kk < vis_s[r] && l_s[r] != -INFINITY) {
          float s = 0.f, dp = 0.f;
#pragma unroll 8
          for (int c = 0; c < D; ++c) {
            s = fmaf(q_s[r][c], k_s[kk][c], s);
            dp = fmaf(do_s[r][c], v_s[kk][c], dp);
          }
          p = expf(s * a.scale - l_s[r]);
          ds = p * (dp - dl_s[r]);
        }
        p_s[r][kk] = p;
        ds_s[r][kk] = ds;
      }
      __syncthreads();
      // dV += P^T dO, dK += scale dS^T Q  (thread owns fixed (key, column) pairs)
#pragma unroll
      for (int m = 0; m < kOwnKV; ++m) {
        const int i = tid + m * kThreads;
        const int kk = i / D, c = i % D;
        float av = dv[m], ak = dk[m];
        for (int r = 0; r < n_r; ++r) {
          av = fmaf(p_s[r][kk], do_s[r][c], av);
          ak = fmaf(ds_s[r][kk], q_s[r][c], ak);
        }
        dv[m] = av;
        dk[m] = ak;
      }
      // partial dQ rows of this item: scale dS K, summed over the tiles' CTAs by atomics
#pragma unroll
      for (int m = 0; m < kOwnQ; ++m) {
        const int i = tid + m * kThreads;
        const int r = i / D, c = i % D;
        if (r >= n_r) continue;
        float acc = 0.f;
        for (int kk = 0; kk < nk; ++kk) acc = fmaf(ds_s[r][kk], k_s[kk][c], acc);
        if (acc != 0.f) {
          const int32_t row = r0 + r;
          const int64_t qrow = static_cast<int64_t>(part_row + row / G) * a.Hq + kvh * G + row % G;
          atomicAdd(dq_part + qrow * D + c, acc * a.scale);
        }
      }
    }
    // the tile's keys are owned by this CTA alone: plain stores
#pragma unroll
    for (int m = 0; m < kOwnKV; ++m) {
      const int i = tid + m * kThreads;
      const int kk = i / D, c = i % D;
      if (kk >= nk) continue;
      const int64_t gi = ((tok0 + kk) * a.Hkv + kvh) * D + c;
      dk_pool[gi] = dk[m] * a.scale;
      dv_pool[gi] = dv[m];
    }
  }
}

// dQ = sum over the sequence's items of their partial dQ rows; one warp per (row, head).
template <int D>
__global__ void __launch_bounds__(256)
    dq_reduce_kernel(const float* __restrict__ dq_part, int64_t part_rows, const int32_t* __restrict__ work, int32_t B,
                     int32_t total_q, int32_t Hq, float* __restrict__ dq, unsigned int* status) {
  constexpr int kPer = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (gw >= static_cast<int64_t>(total_q) * Hq) return;
  const int32_t row = static_cast<int32_t>(gw / Hq), h = static_cast<int32_t>(gw % Hq);
  const WorkView wv(work, B);
  int32_t lo = 0, hi = B - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (__ldg(wv.seq(mid) + kSqCuQ) <= row) lo = mid; else hi = mid - 1;
  }
  const int32_t t = row - __ldg(wv.seq(lo) + kSqCuQ);
  const int32_t p0 = __ldg(wv.seq(lo) + kSqItemPtr), p1 = __ldg(wv.seq(lo + 1) + kSqItemPtr);
  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  for (int32_t p = p0; p < p1; ++p) {
    const int32_t pr = __ldg(wv.item(__ldg(wv.seq_items() + p)) + kItPartRow);
    if (pr < 0 || static_cast<int64_t>(pr) + t >= part_rows) {
      if (lane == 0) atomicOr(status, 2u);
      continue;
    }
    const float* src = dq_part + (static_cast<int64_t>(pr + t) * Hq + h) * D + lane * kPer;
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] += src[k];
  }
  float* dst = dq + gw * D + lane * kPer;
#pragma unroll
  for (int k = 0; k < kPer; ++k) dst[k] = acc[k];
}

template <typename T, int D>
cudaError_t launch_partial(const PartialArgs& a, const void* dout, const float* lse, const float* delta, float* dq_part,
                           float* dk_pool, float* dv_pool, cudaStream_t stream) {
  const int64_t gx = static_cast<int64_t>(a.n_items) * a.Hkv;
  if (gx == 0) return cudaSuccess;
  if (gx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  bwd_partial_kernel<T, D><<<dim3(static_cast<unsigned>(gx), kTilesY), kThreads, 0, stream>>>(
      a, static_cast<const T*>(dout), lse, delta, dq_part, dk_pool, dv_pool);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_delta(const void* o, const void* dout, int64_t n_rows, int32_t d, int32_t dtype, float* delta,
                             cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t grid = (n_rows + 7) / 8;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (dtype == SPLITKV_F32)
    bwd_delta_kernel<float><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
        static_cast<const float*>(o), static_cast<const float*>(dout), n_rows, d, delta);
  else
    bwd_delta_kernel<__nv_bfloat16><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), n_rows, d, delta);
  return cudaGetLastError();
}

cudaError_t launch_bwd_partial(const PartialArgs& a, const void* dout, const float* lse, const float* delta,
                               float* dq_part, float* dk_pool, float* dv_pool, cudaStream_t stream) {
  if (a.dtype == SPLITKV_F32)
    return a.d == 64 ? launch_partial<float, 64>(a, dout, lse, delta, dq_part, dk_pool, dv_pool, stream)
                     : launch_partial<float, 128>(a, dout, lse, delta, dq_part, dk_pool, dv_pool, stream);
  return a.d == 64 ? launch_partial<__nv_bfloat16, 64>(a, dout, lse, delta, dq_part, dk_pool, dv_pool, stream)
                   : launch_partial<__nv_bfloat16, 128>(a, dout, lse, delta, dq_part, dk_pool, dv_pool, stream);
}

cudaError_t launch_dq_reduce(const float* dq_part, int64_t part_rows, const int32_t* work, int32_t B, int32_t total_q,
                             int32_t Hq, int32_t d, float* dq, unsigned int* status, cudaStream_t stream) {
  const int64_t warps = static_cast<int64_t>(total_q) * Hq;
  if (warps == 0) return cudaSuccess;
  const int64_t grid = (warps + 7) / 8;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (d == 64)
    dq_reduce_kernel<64><<<static_cast<unsigned>(grid), 256, 0, stream>>>(dq_part, part_rows, work, B, total_q, Hq,
                                                                          dq, status);
  else
    dq_reduce_kernel<128><<<static_cast<unsigned>(grid), 256, 0, stream>>>(dq_part, part_rows, work, B, total_q, Hq,
                                                                           dq, status);
  return cudaGetLastError();
}

}  // namespace splitkv

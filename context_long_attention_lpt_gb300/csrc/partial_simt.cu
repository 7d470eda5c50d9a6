// Generic CUDA-core partial attention: any q_len, fp32 or bf16, d in {64, 128}.
//
// One CTA computes one (work item, K/V head, tile of kRows query rows).  The
// rows of a (sequence, K/V head) pair are its q_len tokens x G query heads,
// row r = token r / G, head h*G + r % G.  K/V are streamed in tiles of kKeys
// keys through shared memory; every row keeps an online softmax (running max
// m, running sum l, rescaled output accumulator), which over the item's keys
// gives the shard's partial (O_i, L_i) of the Split-KV card's local attention
// step ("Timeline": K/V stay local, only query-sized results leave).
//
// This kernel is the reference implementation on the GPU side: the fp32 path
// (fp32 FFMA throughout, as the 1e-4 tolerance needs) and the fallback for
// shapes the specialised kernels do not take.

#include <cmath>

#include "device_common.cuh"
#include "launch.h"

namespace splitkv {
namespace {

constexpr int kRows = 16;      // query rows per CTA
constexpr int kKeys = 32;      // keys per shared-memory tile (one per lane)
constexpr int kThreads = 128;  // 4 warps

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    partial_simt_kernel(PartialArgs a, int32_t tiles_per_item) {
  constexpr int kOwn = kRows * D / kThreads;  // output elements owned per thread
  __shared__ float q_s[kRows][D];
  __shared__ float k_s[kKeys][D + 1];
  __shared__ float v_s[kKeys][D];
  __shared__ float p_s[kRows][kKeys];
  __shared__ float m_s[kRows], l_s[kRows], alpha_s[kRows];
  __shared__ int32_t vis_s[kRows];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = blockIdx.x;
  const int32_t tile = static_cast<int32_t>(u % tiles_per_item);
  const int32_t kvh = static_cast<int32_t>((u / tiles_per_item) % a.Hkv);
  const int32_t item = static_cast<int32_t>(u / (static_cast<int64_t>(tiles_per_item) * a.Hkv));

  const WorkView wv(a.work, a.B, a.n_items);
  const int32_t* it = wv.item(item);
  const int32_t h_magic = wv.hdr(kMagic), h_b = wv.hdr(kB), h_n = wv.hdr(kNItems);
  const int32_t seq = __ldg(it + kItSeq);
  const int32_t blk_off = __ldg(it + kItBlockOff), blk_cnt = __ldg(it + kItBlockCnt);
  const int32_t part_row = __ldg(it + kItPartRow);
  const int32_t cu_q = __ldg(it + kItCuQ), q_len = __ldg(it + kItQLen), kv_len = __ldg(it + kItKvLen);
  if (!work_matches(h_magic, h_b, h_n, a.B, a.n_items)) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBadWork);
    return;
  }
  const int32_t G = a.Hq / a.Hkv;
  const int32_t rows = q_len * G;
  const int32_t r0 = tile * kRows;
  if (r0 >= rows) return;
  if (part_row < 0 || static_cast<int64_t>(part_row) + q_len > a.part_rows) {
    if (threadIdx.x == 0) atomicOr(a.status, 2u);  // descriptor does not fit the partial buffers
    return;
  }
  const int32_t n_rows = min(kRows, rows - r0);

  const T* q = static_cast<const T*>(a.q);
  const T* kp = static_cast<const T*>(a.k_pool);
  const T* vp = static_cast<const T*>(a.v_pool);

  // Query rows, pre-multiplied by the softmax scale.
  for (int i = tid; i < kRows * D; i += kThreads) {
    const int r = i / D, c = i % D;
    float x = 0.f;
    if (r < n_rows) {
      const int32_t row = r0 + r;
      const int64_t qi = (static_cast<int64_t>(cu_q + row / G) * a.Hq + kvh * G + row % G) * D + c;
      x = to_f32(q[qi]) * a.scale;
    }
    q_s[r][c] = x;
  }
  if (tid < kRows) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
    vis_s[tid] = tid < n_rows ? visible_keys(q_len, kv_len, (r0 + tid) / G, a.causal) : 0;
  }
  float o[kOwn];
#pragma unroll
  for (int k = 0; k < kOwn; ++k) o[k] = 0.f;
  __syncthreads();
  const int32_t vis_max = vis_s[n_rows - 1];  // rows are ordered by token: the last sees most

  const int32_t bl = a.block_len;
  const int32_t* blocks = wv.blocks() + blk_off;
  for (int32_t bi = 0; bi < blk_cnt; ++bi) {
    const int32_t j = __ldg(blocks + bi);
    const int32_t key_lo = j * bl;
    const int32_t key_hi = min(min(kv_len, key_lo + bl), vis_max);
    if (key_lo >= key_hi) continue;
    if (j >= a.max_blocks_per_seq) {
      if (tid == 0) atomicOr(a.status, 1u);
      continue;
    }
    const int32_t phys = __ldg(a.block_table + static_cast<int64_t>(seq) * a.max_blocks_per_seq + j);
    if (phys < 0 || phys >= a.n_pool_blocks) {
      if (tid == 0) atomicOr(a.status, 1u);
      continue;
    }
    const int64_t blk_base = static_cast<int64_t>(phys) * bl;
    for (int32_t k0 = key_lo; k0 < key_hi; k0 += kKeys) {
      const int32_t nk = min(kKeys, key_hi - k0);
      for (int i = tid; i < kKeys * D; i += kThreads) {
        const int kk = i / D, c = i % D;
        float kx = 0.f, vx = 0.f;
        if (kk < nk) {
          const int64_t gi = ((blk_base + (k0 - key_lo) + kk) * a.Hkv + kvh) * D + c;
          kx = to_f32(kp[gi]);
          vx = to_f32(vp[gi]);
        }
        k_s[kk][c] = kx;
        v_s[kk][c] = vx;
      }
      __syncthreads();
      // scores of this tile, masked
      for (int i = tid; i < kRows * kKeys; i += kThreads) {
        const int r = i / kKeys, kk = i % kKeys;
        float s = -INFINITY;
        if (r < n_rows && kk < nk && k0 + kk < vis_s[r]) {
          float acc = 0.f;
#pragma unroll 8
          for (int c = 0; c < D; ++c) acc = fmaf(q_s[r][c], k_s[kk][c], acc);
          s = acc;
        }
        p_s[r][kk] = s;
      }
      __syncthreads();
      // online softmax, one warp per row, one key per lane
      for (int r = warp; r < kRows; r += kThreads / 32) {
        const float s = p_s[r][lane];
        const float m_old = m_s[r];
        const float m_new = fmaxf(m_old, warp_max(s));
        float p = 0.f, alpha = 1.f;
        if (m_new != -INFINITY) {
          p = expf(s - m_new);
          alpha = expf(m_old - m_new);
        }
        const float tile_sum = warp_sum(p);
        p_s[r][lane] = p;
        if (lane == 0) {
          alpha_s[r] = alpha;
          m_s[r] = m_new;
          l_s[r] = l_s[r] * alpha + tile_sum;
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kOwn; ++k) {
        const int i = tid + k * kThreads;
        const int r = i / D, c = i % D;
        float acc = o[k] * alpha_s[r];
        for (int kk = 0; kk < nk; ++kk) acc = fmaf(p_s[r][kk], v_s[kk][c], acc);
        o[k] = acc;
      }
      __syncthreads();
    }
  }

#pragma unroll
  for (int k = 0; k < kOwn; ++k) {
    const int i = tid + k * kThreads;
    const int r = i / D, c = i % D;
    if (r >= n_rows) continue;
    const int32_t row = r0 + r;
    const int64_t orow = static_cast<int64_t>(part_row + row / G) * a.Hq + kvh * G + row % G;
    const float l = l_s[r];
    a.o_part[orow * D + c] = l > 0.f ? o[k] / l : 0.f;
    if (c == 0) a.lse_part[orow] = l > 0.f ? m_s[r] + logf(l) : -INFINITY;
  }
}

template <typename T, int D>
cudaError_t launch_typed(const PartialArgs& a, cudaStream_t stream) {
  const int32_t G = a.Hq / a.Hkv;
  const int32_t tiles = (a.max_q_len * G + kRows - 1) / kRows;
  const int64_t grid = static_cast<int64_t>(tiles) * a.Hkv * a.n_items;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  partial_simt_kernel<T, D><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a, tiles);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_partial_simt(const PartialArgs& a, cudaStream_t stream) {
  if (a.dtype == SPLITKV_F32) {
    return a.d == 64 ? launch_typed<float, 64>(a, stream) : launch_typed<float, 128>(a, stream);
  }
  return a.d == 64 ? launch_typed<__nv_bfloat16, 64>(a, stream)
                   : launch_typed<__nv_bfloat16, 128>(a, stream);
}

}  // namespace splitkv

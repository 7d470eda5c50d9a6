// CUDA-core partial attention for decode-shaped work: bf16, d = 128,
// q_len * G <= 8 query rows per (sequence, K/V head), block_len % 64 == 0.
//
// The Split-KV card's local step ("Timeline": each shard attends over its own
// KV blocks) is, for a single query token, one read of every K/V row of the
// shard's blocks: the kernel is bound by HBM bandwidth.  The design keeps many
// bytes in flight with few instructions per byte:
//
// * One CTA takes one (work item, K/V head) unit.  A producer warp streams the
//   unit's K and V rows with TMA (3-D tiled bulk copies of 64 keys x 256 B out
//   of the paged pool viewed as [tokens, Hkv, d]) into a ring of kStages
//   shared-memory stages, each guarded by a full and an empty mbarrier.
// * Four consumer warps read the stages.  A half-warp works on one key row at
//   a time: lane i holds d-elements [8i, 8i+8) (one 16-byte shared load), and
//   per batch a half-warp takes KPB keys, so a lane computes KPB keys x R rows
//   = 16 partial dot products with packed fp32x2 FMAs.
// * A four-step butterfly over the half-warp (xor 8, 4, 2, 1) sums them.  Each
//   lane reads its keys and query rows in an order permuted by its own lane
//   index (slot i holds logical value i XOR lane), so every step is one shuffle
//   and one add with no selects; afterwards lane i holds the full score of
//   logical value i = key * R + row.
// * Online softmax in base 2 (queries pre-scaled by scale*log2 e): per row a
//   running max m and sum l over lanes sharing the row; P.V accumulates in
//   per-lane fp32x2 registers acc[row][8].  At the end the two half-warps and
//   the four warps are combined exactly through shared memory and the unit's
//   partial (O_i, L_i) is written.
//
// Keys past the sequence end or a row's causal limit get score -inf and their
// V rows are replaced by zeros, so whatever the pool holds there (NaN
// included) never reaches the result.

#include <cmath>

#include "device_common.cuh"
#include "launch.h"
#include "ptx.cuh"
#include "status.h"
#include "tensor_map.h"

namespace splitkv {
namespace {

constexpr int kD = 128;
constexpr int kKT = 64;                       // keys per TMA tile
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kTileBytes = kKT * kD * 2;  // one K (or V) tile
constexpr size_t kSmemBytes = kStages * 2 * kTileBytes + 2 * kStages * sizeof(uint64_t) + 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxFusedItems = 2048;  // items of one sequence the in-kernel merge can hold in shared memory

// Tiles of a work item: for each of its blocks the keys [lo, lo + n) that some
// row of the unit can see, cut into kKT-key tiles.  Producer and consumers
// walk the same sequence.
struct TileWalk {
  const int32_t* blocks;
  const int32_t* table;
  int32_t blk_cnt, bl, max_blocks, kv_len, vis_max;
  int64_t n_pool;

  // Returns the physical block of block bi and its visible key count (0: skip it).
  __device__ __forceinline__ int32_t block(int32_t bi, int32_t* lo, int32_t* n, bool* bad) const {
    const int32_t j = __ldg(blocks + bi);
    *lo = j * bl;
    *n = min(min(bl, kv_len - *lo), vis_max - *lo);
    *bad = false;
    if (*n <= 0) return -1;
    const int32_t phys = j < max_blocks ? __ldg(table + j) : -1;
    if (phys < 0 || phys >= n_pool) {
      *bad = true;
      return -1;
    }
    return phys;
  }
};

template <int R>
__global__ void __launch_bounds__(kThreads, 2)
    partial_decode_kernel(PartialArgs a, const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v) {
  constexpr int KPB = 16 / R;               // keys per half-warp per batch
  constexpr int KPW = 2 * KPB;              // keys per warp per batch
  constexpr int BPW = kKT / (kConsumerWarps * KPW);  // batches per warp per tile
  static_assert(BPW * kConsumerWarps * KPW == kKT, "tile split");

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stage_k = smem;
  uint8_t* stage_v = smem + kStages * kTileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 2 * kStages * kTileBytes);
  uint64_t* empty = full + kStages;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t item = blockIdx.x / a.Hkv;
  const int32_t kvh = blockIdx.x % a.Hkv;

  const WorkView wv(a.work, a.B, a.n_items);
  const int32_t* it = wv.item(item);
  // the header words and the item row are independent loads: one round trip
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
  if (rows == 0) return;
  if (part_row < 0 || static_cast<int64_t>(part_row) + q_len > a.part_rows) {
    if (threadIdx.x == 0) atomicOr(a.status, 2u);
    return;
  }
  const TileWalk walk{wv.blocks() + blk_off,
                      a.block_table + static_cast<int64_t>(seq) * a.max_blocks_per_seq,
                      blk_cnt, a.block_len, a.max_blocks_per_seq, kv_len,
                      visible_keys(q_len, kv_len, (rows - 1) / G, a.causal), a.n_pool_blocks};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], kConsumerWarps);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmap_k);
      ptx::prefetch_tmap(&tmap_v);
      int32_t t = 0;
      bool ok = true;
      for (int32_t bi = 0; bi < blk_cnt && ok; ++bi) {
        int32_t lo, n;
        bool bad;
        const int32_t phys = walk.block(bi, &lo, &n, &bad);
        if (bad) atomicOr(a.status, 1u);
        if (phys < 0) continue;
        for (int32_t off = 0; off < n; off += kKT, ++t) {
          const int s = t % kStages;
          if (t >= kStages && !ptx::mbar_wait(&empty[s], ((t / kStages) & 1) ^ 1)) {
            atomicOr(a.status, ptx::kStatusTimeout);
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[s], 2 * kTileBytes);
          const int32_t row = phys * a.block_len + off;
          ptx::tma_load_3d(stage_k + s * kTileBytes, &tmap_k, 0, kvh, row, &full[s]);
          ptx::tma_load_3d(stage_v + s * kTileBytes, &tmap_v, 0, kvh, row, &full[s]);
        }
      }
      // Copies still in flight land before this CTA's shared memory goes away.
      for (int32_t u = max(0, t - kStages); u < t; ++u)
        if (!ptx::mbar_wait(&full[u % kStages], (u / kStages) & 1)) atomicOr(a.status, ptx::kStatusTimeout);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------------ consumers
  const int hw = lane >> 4, li = lane & 15;
  const int rot_k = li / R, rot_r = li % R;  // this lane's slot permutation
  float2 qf[R][4];
  float m_run = -INFINITY, l_run = 0.f;
  float2 acc[R][4];
  int32_t my_vis = 0;
  if (warp < kConsumerWarps) {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
    const float qscale = a.scale * kLog2e;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = r ^ rot_r;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (row < rows) {
        const int64_t qi = (static_cast<int64_t>(cu_q + row / G) * a.Hq + kvh * G + row % G) * kD + 8 * li;
        u = __ldg(reinterpret_cast<const uint4*>(q + qi));
      }
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = ptx::bf16x2_to_f32x2(w4[e]);
        qf[r][e] = make_float2(f.x * qscale, f.y * qscale);
        acc[r][e] = make_float2(0.f, 0.f);
      }
    }
    my_vis = rot_r < rows ? visible_keys(q_len, kv_len, rot_r / G, a.causal) : 0;

    int32_t t = 0;
    bool ok = true;
    for (int32_t bi = 0; bi < blk_cnt && ok; ++bi) {
      int32_t lo, n;
      bool bad;
      const int32_t phys = walk.block(bi, &lo, &n, &bad);
      if (phys < 0) continue;
      for (int32_t off = 0; off < n; off += kKT, ++t) {
        const int s = t % kStages;
        if (!ptx::mbar_wait(&full[s], (t / kStages) & 1)) {
          if (lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
          ok = false;
          break;
        }
        const int32_t nvalid = min(kKT, n - off);
        const int32_t pos0 = lo + off;
        const __nv_bfloat16* ks = reinterpret_cast<const __nv_bfloat16*>(stage_k + s * kTileBytes);
        const __nv_bfloat16* vs = reinterpret_cast<const __nv_bfloat16*>(stage_v + s * kTileBytes);
#pragma unroll
        for (int bb = 0; bb < BPW; ++bb) {
          const int32_t half_base = (warp * BPW + bb) * KPW + hw * KPB;
          // partial dot products in permuted slots
          float v[16];
#pragma unroll
          for (int k = 0; k < KPB; ++k) {
            const int key = half_base + (k ^ rot_k);
            const uint4 u = *reinterpret_cast<const uint4*>(ks + key * kD + 8 * li);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
            float2 kf[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) kf[e] = ptx::bf16x2_to_f32x2(w4[e]);
#pragma unroll
            for (int r = 0; r < R; ++r) {
              float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < 4; ++e) d2 = ptx::ffma2(qf[r][e], kf[e], d2);
              v[k * R + r] = d2.x + d2.y;
            }
          }
#pragma unroll
          for (int m = 8, nv = 16; m >= 1; m >>= 1, nv >>= 1)
#pragma unroll
            for (int j = 0; j < nv / 2; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j + nv / 2], m);
          // lane holds the score of key half_base + li / R for row li % R
          const int32_t key = half_base + li / R;
          float sc = v[0];
          if (key >= nvalid || pos0 + key >= my_vis) sc = -INFINITY;
          float bmax = sc;
#pragma unroll
          for (int m = R; m < 32; m <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, m));
          const float m_new = fmaxf(m_run, bmax);
          float p = 0.f, alpha = 1.f;
          if (m_new != -INFINITY) {
            p = exp2f(sc - m_new);
            alpha = exp2f(m_run - m_new);
          }
          float psum = p;
#pragma unroll
          for (int m = R; m < 32; m <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, m);
          l_run = l_run * alpha + psum;
          m_run = m_new;
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const float ar = __shfl_sync(0xffffffffu, alpha, (lane & 16) | r);
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[r][e] = make_float2(acc[r][e].x * ar, acc[r][e].y * ar);
            }
          }
          const bool tail = nvalid < kKT;
#pragma unroll
          for (int k = 0; k < KPB; ++k) {
            const int key_k = half_base + k;
            uint4 u = *reinterpret_cast<const uint4*>(vs + key_k * kD + 8 * li);
            if (tail && key_k >= nvalid) u = make_uint4(0, 0, 0, 0);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
            float2 vf[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) vf[e] = ptx::bf16x2_to_f32x2(w4[e]);
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const float pk = __shfl_sync(0xffffffffu, p, (lane & 16) | (k * R + r));
              const float2 pp = make_float2(pk, pk);
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[r][e] = ptx::ffma2(pp, vf[e], acc[r][e]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[s]);
      }
    }
    // The two half-warps saw different keys under the same running max.
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[r][e].x += __shfl_xor_sync(0xffffffffu, acc[r][e].x, 16);
        acc[r][e].y += __shfl_xor_sync(0xffffffffu, acc[r][e].y, 16);
      }
  }
  __syncthreads();  // pipeline drained: the stage memory is free for the combine

  float* sm_acc = reinterpret_cast<float*>(smem);            // [warps][R][kD]
  float* sm_m = sm_acc + kConsumerWarps * R * kD;            // [warps][R]
  float* sm_l = sm_m + kConsumerWarps * R;
  if (warp < kConsumerWarps && hw == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        reinterpret_cast<float2*>(sm_acc + (warp * R + r) * kD + 8 * li)[e] = acc[r][e];
    if (li < R) {
      sm_m[warp * R + li] = m_run;
      sm_l[warp * R + li] = l_run;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < R * kD; i += kThreads) {
    const int r = i / kD, c = i % kD;
    if (r >= rows) continue;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, sm_m[w * R + r]);
    float l = 0.f, o = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float f = exp2f(sm_m[w * R + r] - mx);
        l += sm_l[w * R + r] * f;
        o += sm_acc[(w * R + r) * kD + c] * f;
      }
    }
    const int64_t orow = static_cast<int64_t>(part_row + r / G) * a.Hq + kvh * G + r % G;
    a.o_part[orow * kD + c] = l > 0.f ? o / l : 0.f;
    if (c == 0) a.lse_part[orow] = l > 0.f ? (mx + log2f(l)) * kLn2 : -INFINITY;
  }
  if (!a.fused) return;

  // ---- fused merge: the last CTA of this (sequence, K/V head) group merges ----
  // The CTA's partial rows are published before the group's ticket is taken:
  // the barrier orders every thread's writes before thread 0's fence, whose
  // release covers them (fence-then-count); no CTA ever waits for another.
  __shared__ int s_last;
  __syncthreads();
  uint32_t* ticket = a.tickets + static_cast<int64_t>(seq) * a.Hkv + kvh;
  const WorkView mv(a.work, a.B, a.n_items);  // rebuilt from the arguments: nothing kept live across the loop
  const int32_t p0 = __ldg(mv.seq(seq) + kSqItemPtr), p1 = __ldg(mv.seq(seq + 1) + kSqItemPtr);
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t taken = atomicAdd(ticket, 1u);
    s_last = taken == static_cast<uint32_t>(p1 - p0 - 1);
    __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  // Merge: all LSEs of the group at once, weights per row, then the weighted sum
  // of the partial rows with independent loads (they sit in L2, just written).
  const int32_t* seq_items = mv.seq_items();
  const int32_t n_it = p1 - p0;
  float* sm_w = reinterpret_cast<float*>(smem);            // [n_it][R] weights
  int32_t* sm_pr = reinterpret_cast<int32_t*>(sm_w + kMaxFusedItems * R);  // [n_it] partial rows
  for (int i = threadIdx.x; i < n_it; i += kThreads) sm_pr[i] = __ldg(mv.item(__ldg(seq_items + p0 + i)) + kItPartRow);
  __syncthreads();
  for (int i = threadIdx.x; i < n_it * rows; i += kThreads) {
    const int it = i / rows, r = i % rows;
    sm_w[it * R + r] = __ldcg(a.lse_part + static_cast<int64_t>(sm_pr[it] + r / G) * a.Hq + kvh * G + r % G);
  }
  __syncthreads();
  if (threadIdx.x < rows) {
    const int r = threadIdx.x;
    float mx = -INFINITY;
    for (int it = 0; it < n_it; ++it) mx = fmaxf(mx, sm_w[it * R + r]);
    float sum = 0.f;
    for (int it = 0; it < n_it; ++it) {
      const float e = mx == -INFINITY ? 0.f : exp2f((sm_w[it * R + r] - mx) * kLog2e);
      sm_w[it * R + r] = e;
      sum += e;
    }
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int it = 0; it < n_it; ++it) sm_w[it * R + r] *= inv;
    const int64_t orow = static_cast<int64_t>(cu_q + r / G) * a.Hq + kvh * G + r % G;
    a.lse_out[orow] = sum > 0.f ? mx + logf(sum) : -INFINITY;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < rows * (kD / 4); i += kThreads) {
    const int r = i / (kD / 4), c4 = i % (kD / 4);
    const int32_t tok = r / G, h = kvh * G + r % G;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int it = 0; it < n_it; ++it) {
      const float w = sm_w[it * R + r];
      const float4 x = __ldcg(reinterpret_cast<const float4*>(a.o_part + (static_cast<int64_t>(sm_pr[it] + tok) * a.Hq + h) * kD) + c4);
      o.x = fmaf(w, x.x, o.x);
      o.y = fmaf(w, x.y, o.y);
      o.z = fmaf(w, x.z, o.z);
      o.w = fmaf(w, x.w, o.w);
    }
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(a.out) +
                                                            (static_cast<int64_t>(cu_q + tok) * a.Hq + h) * kD) + 2 * c4;
    dst[0] = __floats2bfloat162_rn(o.x, o.y);
    dst[1] = __floats2bfloat162_rn(o.z, o.w);
  }
  if (threadIdx.x == 0) *ticket = 0u;  // ready for the next launch
}

template <int R>
int launch_r(const PartialArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  auto kern = partial_decode_kernel<R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "decode smem attribute: %s", cudaGetErrorString(e));
  const int64_t grid = static_cast<int64_t>(a.n_items) * a.Hkv;
  kern<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(a, tk, tv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return SPLITKV_OK;
}

}  // namespace

// The in-kernel merge keeps one weight per (item, row) of a sequence in the
// freed stage memory: at most kMaxFusedItems items, i.e. a sequence spread over
// no more than that many shards (weights + rows take 2048 x (8 + 1) x 4 = 73 KB).
bool decode_fuses(const PartialArgs& a) { return decode_supports(a) && a.n_items <= kMaxFusedItems; }

bool decode_supports(const PartialArgs& a) {
  if (a.dtype != SPLITKV_BF16 || a.d != kD || a.Hkv <= 0 || a.Hq % a.Hkv != 0) return false;
  const int64_t rows = static_cast<int64_t>(a.max_q_len) * (a.Hq / a.Hkv);
  return rows >= 1 && rows <= 8 && a.block_len % kKT == 0 &&
         static_cast<int64_t>(a.n_pool_blocks) * a.block_len < (1ll << 31);
}

int decode_blocks_per_sm(const PartialArgs& a, int* blocks) {
  const int64_t rows = static_cast<int64_t>(a.max_q_len) * (a.Hq / a.Hkv);
  cudaError_t e;
  if (rows <= 4) {
    e = cudaFuncSetAttribute(partial_decode_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, partial_decode_kernel<4>, kThreads, kSmemBytes);
  } else {
    e = cudaFuncSetAttribute(partial_decode_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, partial_decode_kernel<8>, kThreads, kSmemBytes);
  }
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "decode occupancy: %s", cudaGetErrorString(e));
  return SPLITKV_OK;
}

int launch_partial_decode(const PartialArgs& a, cudaStream_t stream) {
  const int64_t grid = static_cast<int64_t>(a.n_items) * a.Hkv;
  if (grid == 0) return SPLITKV_OK;
  if (grid > 0x7fffffffLL) return fail(SPLITKV_ERR_UNSUPPORTED, "too many work units");
  // K/V pools as [tokens, Hkv, d] bf16; one box = 64 tokens of one head.
  const uint64_t dims[3] = {kD, static_cast<uint64_t>(a.Hkv),
                            static_cast<uint64_t>(a.n_pool_blocks) * a.block_len};
  const uint64_t strides[2] = {kD * 2ull, static_cast<uint64_t>(a.Hkv) * kD * 2ull};
  const uint32_t box[3] = {kD, 1, kKT};
  CUtensorMap tk, tv;
  int st = encode_bf16_3d(&tk, a.k_pool, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != SPLITKV_OK) return st;
  st = encode_bf16_3d(&tv, a.v_pool, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != SPLITKV_OK) return st;
  const int64_t rows = static_cast<int64_t>(a.max_q_len) * (a.Hq / a.Hkv);
  return rows <= 4 ? launch_r<4>(a, tk, tv, stream) : launch_r<8>(a, tk, tv, stream);
}

}  // namespace splitkv

// CUDA-core partial attention for decode-shaped work: bf16, d = 128,
// q_len * G <= 8 query rows per (sequence, K/V head).
//
// The Split-KV card's local step ("Timeline": each shard attends over its own
// KV blocks) is, for one query token, a read of every K/V row of the shard's
// blocks once: the kernel is bound by HBM bandwidth, so the design goal is
// coalesced 128-bit loads with many bytes in flight and few instructions per
// byte.
//
// One CTA (4 warps) takes one (work item, K/V head) unit.  A half-warp owns one
// 256-byte K (or V) row per load: lane i of the half-warp loads d-elements
// [8i, 8i+8) with one 16-byte load, so each row is two full 128-byte lines.
// A warp processes batches of 2*KPB keys (KPB per half-warp); the next batch
// is prefetched into registers while the current one is computed.
//
// Scores: every lane has partial dot products over its 8 elements for KPB keys
// x R rows = 16 values.  A four-step butterfly (xor 8, 4, 2, 1) halves the
// values per lane at each step while summing across the half-warp, leaving lane
// i with the full score of value i = key * R + row: 15 shuffles for 16 scores.
// The online softmax (running max m, running sum l, in base 2 with the query
// pre-scaled by scale*log2(e)) then runs per row over lanes sharing the row,
// and P.V accumulates into per-lane registers acc[row][8].  At the end the two
// half-warps and the 4 warps are combined exactly (max / rescaled sums)
// through shared memory and the unit's partial (O_i, L_i) is written.

#include <cmath>

#include "device_common.cuh"
#include "launch.h"

namespace splitkv {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// One butterfly step over N values: lanes whose `mask` bit is set keep the
// upper half, the others the lower half; each kept value adds the partner's.
template <int N>
__device__ __forceinline__ void butterfly(float (&v)[16], bool upper, int mask) {
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    const float send = upper ? v[j] : v[j + N / 2];
    const float keep = upper ? v[j + N / 2] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
  }
}

template <int R>
__global__ void __launch_bounds__(kWarps * 32, R == 4 ? 3 : 2) partial_decode_kernel(PartialArgs a) {
  constexpr int KPB = 16 / R;   // keys per half-warp per batch
  constexpr int KPW = 2 * KPB;  // keys per warp per batch
  __shared__ float sm_acc[kWarps][R][kD];
  __shared__ float sm_m[kWarps][R];
  __shared__ float sm_l[kWarps][R];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hw = lane >> 4, li = lane & 15;
  const int32_t item = blockIdx.x / a.Hkv;
  const int32_t kvh = blockIdx.x % a.Hkv;

  const WorkView wv(a.work);
  const int32_t* it = wv.item(item);
  const int32_t seq = __ldg(it + kItSeq);
  const int32_t blk_off = __ldg(it + kItBlockOff), blk_cnt = __ldg(it + kItBlockCnt);
  const int32_t part_row = __ldg(it + kItPartRow);
  const int32_t* sq = wv.seq(seq);
  const int32_t cu_q = __ldg(sq + kSqCuQ), q_len = __ldg(sq + kSqQLen), kv_len = __ldg(sq + kSqKvLen);
  const int32_t G = a.Hq / a.Hkv;
  const int32_t rows = q_len * G;
  if (rows == 0) return;
  if (part_row < 0 || static_cast<int64_t>(part_row) + q_len > a.part_rows) {
    if (threadIdx.x == 0) atomicOr(a.status, 2u);
    return;
  }

  // Query rows (token r / G, head kvh*G + r % G), this lane's 8 elements, scaled to base 2.
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const float qscale = a.scale * kLog2e;
  float qf[R][8];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r < rows) {
      const int64_t qi = (static_cast<int64_t>(cu_q + r / G) * a.Hq + kvh * G + r % G) * kD + 8 * li;
      float f[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(q + qi)), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[r][e] = f[e] * qscale;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[r][e] = 0.f;
    }
  }
  // This lane's score after the butterfly belongs to row li % R.
  const int my_row = li % R;
  const int32_t my_vis = my_row < rows ? visible_keys(q_len, kv_len, my_row / G, a.causal) : 0;

  const uint4* kp = static_cast<const uint4*>(a.k_pool);
  const uint4* vp = static_cast<const uint4*>(a.v_pool);
  const int32_t bl = a.block_len;
  const int32_t* blocks = wv.blocks() + blk_off;
  const int32_t* table = a.block_table + static_cast<int64_t>(seq) * a.max_blocks_per_seq;
  const int64_t n_batches = static_cast<int64_t>(blk_cnt) * (bl / KPW);
  const int64_t row_stride = static_cast<int64_t>(a.Hkv) * (kD / 8);  // uint4 per token

  // Loads the K/V rows of batch `b` for this half-warp; returns the position of
  // its first key (or -1 if the batch's block is unusable).  Keys past the
  // sequence end are not read (zeros), so their slots never carry NaN.
  auto load = [&](int64_t b, uint4 (&kb)[KPB], uint4 (&vb)[KPB]) -> int32_t {
    const int32_t bi = static_cast<int32_t>(b / (bl / KPW));
    const int32_t off = static_cast<int32_t>(b % (bl / KPW)) * KPW + hw * KPB;
    const int32_t j = __ldg(blocks + bi);
    int32_t phys = j < a.max_blocks_per_seq ? __ldg(table + j) : -1;
    if (phys < 0 || phys >= a.n_pool_blocks) {
      if (lane == 0) atomicOr(a.status, 1u);
      phys = -1;
    }
    const int32_t pos0 = j * bl + off;
    const int64_t base = ((static_cast<int64_t>(phys) * bl + off) * a.Hkv + kvh) * (kD / 8) + li;
#pragma unroll
    for (int k = 0; k < KPB; ++k) {
      if (phys >= 0 && pos0 + k < kv_len) {
        kb[k] = __ldg(kp + base + k * row_stride);
        vb[k] = __ldg(vp + base + k * row_stride);
      } else {
        kb[k] = make_uint4(0, 0, 0, 0);
        vb[k] = make_uint4(0, 0, 0, 0);
      }
    }
    return phys >= 0 ? pos0 : -1;
  };

  float m_run = -INFINITY, l_run = 0.f;
  float acc[R][8];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[r][e] = 0.f;

  uint4 kc[KPB], vc[KPB], kn[KPB], vn[KPB];
  int64_t b = warp;
  int32_t pos_c = b < n_batches ? load(b, kc, vc) : -1;
  for (; b < n_batches; b += kWarps) {
    const int64_t bn = b + kWarps;
    int32_t pos_n = -1;
    if (bn < n_batches) pos_n = load(bn, kn, vn);

    // partial dot products: v[k*R + r] over this lane's 8 elements
    float v[16];
#pragma unroll
    for (int k = 0; k < KPB; ++k) {
      float kf[8];
      bf16x8_to_f32(kc[k], kf);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) s = fmaf(qf[r][e], kf[e], s);
        v[k * R + r] = s;
      }
    }
    butterfly<16>(v, li & 8, 8);
    butterfly<8>(v, li & 4, 4);
    butterfly<4>(v, li & 2, 2);
    butterfly<2>(v, li & 1, 1);
    // lane holds the score of key (hw*KPB + li / R) for row li % R
    const int32_t pos = pos_c + li / R;
    float s = v[0];
    if (pos_c < 0 || pos >= kv_len || pos >= my_vis) s = -INFINITY;
    float bmax = s;
#pragma unroll
    for (int m = R; m < 32; m <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, m));
    const float m_new = fmaxf(m_run, bmax);
    float p = 0.f, alpha = 1.f;
    if (m_new != -INFINITY) {
      p = exp2f(s - m_new);
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
        for (int e = 0; e < 8; ++e) acc[r][e] *= ar;
      }
    }
#pragma unroll
    for (int k = 0; k < KPB; ++k) {
      float vf[8];
      bf16x8_to_f32(vc[k], vf);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float pk = __shfl_sync(0xffffffffu, p, (lane & 16) | (k * R + r));
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[r][e] = fmaf(pk, vf[e], acc[r][e]);
      }
    }
#pragma unroll
    for (int k = 0; k < KPB; ++k) {
      kc[k] = kn[k];
      vc[k] = vn[k];
    }
    pos_c = pos_n;
  }

  // The two half-warps saw different keys under the same running max: add them.
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[r][e] += __shfl_xor_sync(0xffffffffu, acc[r][e], 16);
  if (hw == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int e = 0; e < 8; ++e) sm_acc[warp][r][8 * li + e] = acc[r][e];
    if (li < R) {
      sm_m[warp][li] = m_run;
      sm_l[warp][li] = l_run;
    }
  }
  __syncthreads();

  // Exact combination of the warps' running (m, l, acc), then the unit's partial.
  for (int i = threadIdx.x; i < R * kD; i += kWarps * 32) {
    const int r = i / kD, c = i % kD;
    if (r >= rows) continue;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, sm_m[w][r]);
    float l = 0.f, o = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(sm_m[w][r] - mx);
        l += sm_l[w][r] * f;
        o += sm_acc[w][r][c] * f;
      }
    }
    const int64_t orow = static_cast<int64_t>(part_row + r / G) * a.Hq + kvh * G + r % G;
    a.o_part[orow * kD + c] = l > 0.f ? o / l : 0.f;
    if (c == 0) a.lse_part[orow] = l > 0.f ? (mx + log2f(l)) * kLn2 : -INFINITY;
  }
}

}  // namespace

bool decode_supports(const PartialArgs& a) {
  if (a.dtype != SPLITKV_BF16 || a.d != kD || a.Hkv <= 0 || a.Hq % a.Hkv != 0) return false;
  const int64_t rows = static_cast<int64_t>(a.max_q_len) * (a.Hq / a.Hkv);
  return rows >= 1 && rows <= 8 && a.block_len % 8 == 0;
}

cudaError_t launch_partial_decode(const PartialArgs& a, cudaStream_t stream) {
  const int64_t grid = static_cast<int64_t>(a.n_items) * a.Hkv;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int64_t rows = static_cast<int64_t>(a.max_q_len) * (a.Hq / a.Hkv);
  if (rows <= 4)
    partial_decode_kernel<4><<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(a);
  else
    partial_decode_kernel<8><<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace splitkv

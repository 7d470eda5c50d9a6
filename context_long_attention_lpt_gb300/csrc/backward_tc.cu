// Tensor-core backward of the split-KV attention for sm_103a: TMA + tcgen05 +
// TMEM.  Same results as the CUDA-core backward in backward.cu (per-shard dK,
// dV and partial dQ over the work items), for bf16, d = 128, block_len % 128 == 0
// and G | 64 (a 64-row tile of the dK/dV kernel holds whole query tokens).
//
// The Split-KV card places the method in training (card intro) and states it
// is exact ("All Facts").  With the merged forward's L and D = rowsum(dO * O),
// a shard's keys need only query-sized tensors:
//   P = exp(s - L), dP = dO V^T, dS = P (dP - D),
//   dQ_i = scale dS K   (partial, summed over the shards by splitkv_dq_reduce),
//   dK = scale dS^T Q,  dV = P^T dO.
//
// Two kernels:
//  * bwd_dq_tc_kernel: one CTA per (work item, K/V head, 128 query rows).  It
//    walks the item's key tiles like the forward: S = Q K^T and dP = dO V^T in
//    TMEM, the row threads form dS (bf16) over S, then dQ += dS K.  S is double
//    buffered, so the next tile's S MMAs run during the row threads' pass.
//  * bwd_dkdv_tc_kernel: one CTA per (work item, K/V head, a stride of the
//    item's 128-key tiles).  Keys sit in the TMEM lanes: S^T = K Q^T and
//    dP^T = V dO^T, the key threads form P^T and dS^T (bf16) in place, then
//    dV += P^T dO and dK += dS^T Q accumulate over all query rows of the
//    sequence, 64 at a time (two row tiles' S^T | dP^T pairs fit in TMEM, so
//    the next tile's MMAs run during the key threads' pass).
// The MMA warps wait only on named barriers, which the other warps hand over;
// every mbarrier wait has a time limit.  On expiry the status word gets bit 2,
// the warp stops waiting and touching TMEM but keeps taking part in every
// named-barrier hand-off, and the CTA unwinds (all MMAs drained, TMEM freed).

#include <algorithm>
#include <cmath>

#include "device_common.cuh"
#include "launch.h"
#include "ptx.cuh"
#include "status.h"
#include "tc_ptx.cuh"
#include "tensor_map.h"

namespace splitkv {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;  // query rows per tile
constexpr int kN = 128;     // keys per tile
constexpr uint32_t kHalfBytes = 128 * 64 * 2;    // 128 rows x 64 bf16: one swizzled half
constexpr uint32_t kTileBytes = 2 * kHalfBytes;  // one 128 x 128 bf16 operand tile
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
// dQ kernel: warps 0-7 elementwise, two per TMEM lane quarter (warp w: rows of
// quarter w % 4, key columns w / 4 * 64 .. + 63 of each key tile); 8: TMA; 9: MMA
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kRowWarps = 8;
// Named barriers of the dQ kernel (0 is __syncthreads), between the row warps
// (bar.arrive) and the MMA warp (bar.sync): kBarDpFree, dP(t) read; kBarDsQ +
// (t & 1), dS(t) written.  A row warp reaches dP(t+1) only after dP(t+1) was
// issued, which follows the MMA warp's pass of kBarDpFree for tile t, and
// dS(t+2) only after S(t+2), which follows its pass of kBarDsQ for tile t: no
// generation mixes arrivals of two tiles.
constexpr int kBarDpFree = 1, kBarDsQ = 2, kBarDqThreads = (kRowWarps + 1) * 32;
// dS (bf16 pairs) of keys 16 kk .. 16 kk + 15, relative to the S columns of the
// tile: keys 0-63 over columns 0-31, keys 64-127 over columns 64-95 (each row
// warp writes over the columns it has read; the other half stays intact).
__device__ __forceinline__ uint32_t ds_col(int kk) { return 8u * kk + (kk >= 4 ? 32u : 0u); }

// TMEM columns of the dK/dV kernel's two fp32 accumulators.
constexpr uint32_t kColAcc0 = 256, kColAcc1 = 384;

// Byte offset (>> 4) of 16-wide K step kk inside a K-major SW128 tile made of two
// 64-column halves: steps 0-3 in the first half, 4-7 in the second.
__device__ __forceinline__ uint32_t kstep_off(int kk) { return ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4; }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// One item's key blocks: keys [lo, lo + n) of block bi that some row of the
// unit can see, or -1 (nothing to read; *bad if the block-table entry is out
// of the pool).
struct ItemBlocks {
  const int32_t* blocks;
  const int32_t* table;
  int32_t blk_cnt, bl, max_blocks, kv_len, vis_max;
  int64_t n_pool;
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

// Tiles of the item in order, for the roles that only need their key counts.
struct TileSeq {
  ItemBlocks ib;
  int32_t bi = 0, off = 0, n = 0, lo = 0, phys = -1;
  bool have = false;
  bool bad_seen = false;  // a block-table entry outside the pool was skipped
  __device__ __forceinline__ bool next(int32_t* pos0, int32_t* nvalid, int32_t* tok) {
    while (true) {
      if (have && off + kN < n) {
        off += kN;
        break;
      }
      have = false;
      while (bi < ib.blk_cnt && !have) {
        bool bad;
        phys = ib.block(bi++, &lo, &n, &bad);
        bad_seen |= bad;
        if (phys >= 0) {
          have = true;
          off = 0;
        }
      }
      if (!have) return false;
      break;
    }
    *pos0 = lo + off;
    *nvalid = min(kN, n - off);
    *tok = phys * ib.bl + off;
    return true;
  }
};

// ============================================================== dQ kernel

constexpr int kKStages = 3;  // K(t) is read by S(t) and, after the row threads' pass, by dQ(t)
constexpr int kVStages = 2;  // V(t) only by dP(t)
// TMEM: S of tile parity b at 128 b (dS is written over it), dP, then dQ
constexpr uint32_t kColS0 = 0, kColDPq = 256, kColDQ = 384;

struct DqBarriers {
  uint64_t qd_full;                               // Q and dO tiles of the unit
  uint64_t k_full[kKStages], k_free[kKStages];    // K(t); its dQ MMA has read it
  uint64_t v_full[kVStages], v_free[kVStages];    // V(t); its dP MMA has read it
  uint64_t s_full[2];                             // S of tile parity b ready
  uint64_t dp_full;                               // dP(t) ready
  uint64_t o_done, drain;
  uint32_t tmem_base;
  // Tile t's key count | (tile t+1 exists) << 16 | (tile t+2 exists) << 17, at [t & 1]:
  // written by row warp 0 before its dP(t)-read arrival, read by the MMA warp after it
  uint32_t tinfo[2];
};
constexpr size_t kDqSmem = 1024 + kTileBytes * (2 + kKStages + kVStages) + sizeof(DqBarriers);

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(PartialArgs a, const float* __restrict__ lse, const float* __restrict__ delta,
                     float* __restrict__ dq_part, int32_t units_per_item, const __grid_constant__ CUtensorMap tmap_q,
                     const __grid_constant__ CUtensorMap tmap_do, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem;                        // Q tile
  uint8_t* sdo = smem + kTileBytes;          // dO tile
  uint8_t* sk = smem + 2 * kTileBytes;       // K ring
  uint8_t* sv = sk + kKStages * kTileBytes;  // V ring
  DqBarriers* bar = reinterpret_cast<DqBarriers*>(sv + kVStages * kTileBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t u = blockIdx.x;
  const int32_t utile = static_cast<int32_t>(u % units_per_item);
  const int32_t kvh = static_cast<int32_t>((u / units_per_item) % a.Hkv);
  const int32_t item = static_cast<int32_t>(u / (static_cast<int64_t>(units_per_item) * a.Hkv));

  const WorkView wv(a.work, a.B, a.n_items);
  const int32_t* it = wv.item(item);
  // the header words and the item row are independent loads: one round trip
  const int32_t h_magic = wv.hdr(kMagic), h_b = wv.hdr(kB), h_n = wv.hdr(kNItems);
  const int32_t seq = __ldg(it + kItSeq);
  const int32_t part_row = __ldg(it + kItPartRow);
  const int32_t cu_q = __ldg(it + kItCuQ), q_len = __ldg(it + kItQLen), kv_len = __ldg(it + kItKvLen);
  if (!work_matches(h_magic, h_b, h_n, a.B, a.n_items)) {  // uniform over the CTA
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBadWork);
    return;
  }
  const int32_t G = a.Hq / a.Hkv;
  const int32_t rows = q_len * G;
  const int32_t r0 = utile * kRows;
  if (r0 >= rows) return;  // uniform over the CTA
  if (part_row < 0 || static_cast<int64_t>(part_row) + q_len > a.part_rows) {
    if (threadIdx.x == 0) atomicOr(a.status, 2u);
    return;
  }
  const int32_t n_rows = min(kRows, rows - r0);
  const int32_t vis_last = visible_keys(q_len, kv_len, (r0 + n_rows - 1) / G, a.causal);
  TileSeq tiles;
  tiles.ib = ItemBlocks{wv.blocks() + __ldg(it + kItBlockOff),
                        a.block_table + static_cast<int64_t>(seq) * a.max_blocks_per_seq, __ldg(it + kItBlockCnt),
                        a.block_len, a.max_blocks_per_seq, kv_len, vis_last, a.n_pool_blocks};

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar->qd_full, 1);
    for (int s = 0; s < kKStages; ++s) {
      ptx::mbar_init(&bar->k_full[s], 1);
      ptx::mbar_init(&bar->k_free[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      ptx::mbar_init(&bar->v_full[s], 1);
      ptx::mbar_init(&bar->v_free[s], 1);
    }
    for (int b = 0; b < 2; ++b) ptx::mbar_init(&bar->s_full[b], 1);
    ptx::mbar_init(&bar->dp_full, 1);
    ptx::mbar_init(&bar->o_done, 1);
    ptx::mbar_init(&bar->drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&bar->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bar->tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmap_q);
      ptx::prefetch_tmap(&tmap_do);
      ptx::prefetch_tmap(&tmap_k);
      ptx::prefetch_tmap(&tmap_v);
      const int32_t tok0 = cu_q + r0 / G;
      ptx::mbar_arrive_expect_tx(&bar->qd_full, 2 * kTileBytes);
      ptx::tma_load_3d(sq, &tmap_q, 0, kvh * G, tok0, &bar->qd_full);
      ptx::tma_load_3d(sq + kHalfBytes, &tmap_q, 64, kvh * G, tok0, &bar->qd_full);
      ptx::tma_load_3d(sdo, &tmap_do, 0, kvh * G, tok0, &bar->qd_full);
      ptx::tma_load_3d(sdo + kHalfBytes, &tmap_do, 64, kvh * G, tok0, &bar->qd_full);
      int32_t t = 0, pos0, nv, tok;
      bool ok = true;
      while (ok && tiles.next(&pos0, &nv, &tok)) {
        const int ks = t % kKStages, vs = t % kVStages;
        if (t >= kKStages && !ptx::mbar_wait(&bar->k_free[ks], ((t - kKStages) / kKStages) & 1)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(&bar->k_full[ks], kTileBytes);
        ptx::tma_load_3d(sk + ks * kTileBytes, &tmap_k, 0, kvh, tok, &bar->k_full[ks]);
        ptx::tma_load_3d(sk + ks * kTileBytes + kHalfBytes, &tmap_k, 64, kvh, tok, &bar->k_full[ks]);
        if (t >= kVStages && !ptx::mbar_wait(&bar->v_free[vs], ((t - kVStages) / kVStages) & 1)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(&bar->v_full[vs], kTileBytes);
        ptx::tma_load_3d(sv + vs * kTileBytes, &tmap_v, 0, kvh, tok, &bar->v_full[vs]);
        ptx::tma_load_3d(sv + vs * kTileBytes + kHalfBytes, &tmap_v, 64, kvh, tok, &bar->v_full[vs]);
        ++t;
      }
      if (!ok) atomicOr(a.status, ptx::kStatusTimeout);
      // every copy issued has landed before shared memory is released
      if (!ptx::mbar_wait(&bar->qd_full, 0)) atomicOr(a.status, ptx::kStatusTimeout);
      for (int32_t v = max(0, t - kKStages); v < t; ++v)
        if (!ptx::mbar_wait(&bar->k_full[v % kKStages], (v / kKStages) & 1)) atomicOr(a.status, ptx::kStatusTimeout);
      for (int32_t v = max(0, t - kVStages); v < t; ++v)
        if (!ptx::mbar_wait(&bar->v_full[v % kVStages], (v / kVStages) & 1)) atomicOr(a.status, ptx::kStatusTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    // Tile t: S(t) = Q K(t)^T into the S buffer of parity t & 1, dP(t) = dO V(t)^T,
    // and, once the row threads have put dS(t) over S(t), dQ += dS(t) K(t).
    // dP(t+1) goes in as soon as the row threads have read dP(t) (halfway through
    // their pass), ahead of dQ(t); S(t+2) follows dQ(t) into tile t's buffer
    // (MMAs run in order, so dQ(t) has read dS(t) first).  The next tile's S and
    // dP are thus done or in the pipe when the row threads finish a tile.
    // This lane's issue waits for the pipe, so every other wait here leaves the
    // pipe idle: past the first two tiles the row threads, which have time to
    // spare, wait for the V and K copies (V(t+1) before their dP(t)-read arrival,
    // K(t+2) before their dS(t) arrival) and pass each tile's key count along.
    const uint32_t idesc_s = tc::idesc_bf16_f32(kRows, kN, false, false);
    const uint32_t idesc_dq = tc::idesc_bf16_f32(kRows, kD, false, true);
    const tc::Desc dq0 = tc::split(tc::smem_desc(ptx::smem_addr(sq), 16, 1024, tc::kSwizzle128B));
    const tc::Desc ddo = tc::split(tc::smem_desc(ptx::smem_addr(sdo), 16, 1024, tc::kSwizzle128B));
    const tc::Desc dk = tc::split(tc::smem_desc(ptx::smem_addr(sk), 16, 1024, tc::kSwizzle128B));
    const tc::Desc dv = tc::split(tc::smem_desc(ptx::smem_addr(sv), 16, 1024, tc::kSwizzle128B));
    const tc::Desc dk_mn = tc::split(tc::smem_desc(ptx::smem_addr(sk), kHalfBytes, 1024, tc::kSwizzle128B));
    constexpr uint32_t kTile16 = kTileBytes >> 4;
    auto issue_s = [&](int32_t t) {
      const uint32_t koff = (t % kKStages) * kTile16;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk)
        tc::mma_ss_fast(tmem + kColS0 + 128 * (t & 1), dq0, kstep_off(kk), dk, koff + kstep_off(kk), idesc_s, kk > 0);
      tc::commit(&bar->s_full[t & 1]);
    };
    auto issue_dp = [&](int32_t t) {
      const int vs = t % kVStages;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk)
        tc::mma_ss_fast(tmem + kColDPq, ddo, kstep_off(kk), dv, vs * kTile16 + kstep_off(kk), idesc_s, kk > 0);
      tc::commit(&bar->dp_full);
      tc::commit(&bar->v_free[vs]);
    };
    auto wait_all = [&](uint64_t* b, uint32_t parity) { return __all_sync(0xffffffffu, ptx::mbar_wait(b, parity)); };
    int32_t pos0, tok, nv0 = 0, nv1 = 0;
    TileSeq walk = tiles;
    // The tile walk does not depend on the waits: this warp takes part in one
    // kBarDpFree and one kBarDsQ hand-off per tile whatever happens (after a
    // timeout its MMAs may read stale operands; the status word reports it).
    bool ok = wait_all(&bar->qd_full, 0);
    bool has_cur = walk.next(&pos0, &nv0, &tok);
    const bool has_one = has_cur && walk.next(&pos0, &nv1, &tok);
    if (has_cur) {
      ok = wait_all(&bar->k_full[0], 0) && wait_all(&bar->v_full[0], 0) && ok;
      tc::fence_after_sync();
      if (tc::elect_one()) {
        issue_s(0);
        issue_dp(0);
      }
      __syncwarp();
      if (has_one) {
        ok = wait_all(&bar->k_full[1 % kKStages], 0) && ok;
        tc::fence_after_sync();
        if (tc::elect_one()) issue_s(1);
        __syncwarp();
      }
    }
    int32_t t = 0;
    while (has_cur) {
      ptx::bar_sync(kBarDpFree, kBarDqThreads);  // dP(t) read; V(t+1) landed; tinfo
      tc::fence_after_sync();
      const uint32_t info = bar->tinfo[t & 1];
      const int32_t nv_cur = static_cast<int32_t>(info & 0xffffu);
      const bool has_next = (info >> 16) & 1u, has_next2 = (info >> 17) & 1u;
      if (has_next && tc::elect_one()) issue_dp(t + 1);
      __syncwarp();
      ptx::bar_sync(kBarDsQ + (t & 1), kBarDqThreads);  // dS(t) written; K(t+2) landed
      tc::fence_after_sync();
      const int ks = t % kKStages;
      const int ksteps = (min(max(nv_cur, 0), kN) + 15) >> 4;
      if (nv_cur < ksteps * 16) {
        // K rows of keys past the end inside the last 16-key step: zero (their dS
        // is 0, but the pool slot may hold anything); S(t) has read them already
        uint8_t* ktile = sk + ks * kTileBytes;
        for (int r = nv_cur + (lane >> 4); r < ksteps * 16; r += 2) {
          const int cc = lane & 15;
          reinterpret_cast<uint4*>(ktile + (cc < 8 ? 0 : kHalfBytes) + r * 128)[cc & 7] = make_uint4(0, 0, 0, 0);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
      }
      if (tc::elect_one()) {
        for (int kk = 0; kk < ksteps; ++kk)
          tc::mma_ts_fast(tmem + kColDQ, tmem + kColS0 + 128 * (t & 1) + ds_col(kk), dk_mn,
                          ks * kTile16 + kk * (2048 >> 4), idesc_dq, (t > 0 || kk > 0) ? 1u : 0u);
        tc::commit(&bar->k_free[ks]);
        if (!has_next) tc::commit(&bar->o_done);
        if (has_next2) issue_s(t + 2);
      }
      __syncwarp();
      ++t;
      has_cur = has_next;
    }
    if (!ok && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
    if (tc::elect_one()) tc::commit(&bar->drain);
    __syncwarp();
    if (!ptx::mbar_wait(&bar->drain, 0) && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
  } else {
    // ----------------------------------------------------- row threads (dS)
    const int rq = warp & 3, hh = warp >> 2;  // TMEM lane quarter; 64-key half of each key tile
    const int32_t row = rq * 32 + lane;       // TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(rq * 32) << 16);
    const bool row_valid = row < n_rows;
    const int32_t token = (r0 + row) / G, h = kvh * G + (r0 + row) % G;
    const int64_t grow = static_cast<int64_t>(cu_q + token) * a.Hq + h;
    const float L = row_valid ? __ldg(lse + grow) : -INFINITY;
    const float Dr = row_valid ? __ldg(delta + grow) : 0.f;
    const bool live = L != -INFINITY;  // a row with no visible key has no gradient
    const float c = a.scale * kLog2e, lc = live ? L * kLog2e : 0.f;
    const int32_t my_vis = row_valid ? visible_keys(q_len, kv_len, token, a.causal) : 0;
    TileSeq walk = tiles, ahead = tiles;  // ahead runs two tiles in front
    int32_t pos0, nvalid, tok, apos, anv, atok, t = 0;
    bool has1 = ahead.next(&apos, &anv, &atok);
    bool has2 = has1 && ahead.next(&apos, &anv, &atok);  // tile 1 exists
    bool has3 = has2 && ahead.next(&apos, &anv, &atok);  // tile 2 exists
    bool ok = true;
    const float2 c2 = make_float2(c, c), nlc2 = make_float2(-lc, -lc), nd2 = make_float2(-Dr, -Dr);
    while (walk.next(&pos0, &nvalid, &tok)) {
      const bool has_next = has2, has_next2 = has3;
      // tile t's key count and whether tiles t+1, t+2 exist, for the MMA warp
      const uint32_t info = static_cast<uint32_t>(nvalid) | (has_next ? 1u << 16 : 0u) | (has_next2 ? 1u << 17 : 0u);
      if (ok)
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->s_full[t & 1], (t >> 1) & 1)) &&
             __all_sync(0xffffffffu, ptx::mbar_wait(&bar->dp_full, t & 1));
      if (!ok) {
        // a wait ran out: no more TMEM work, but both hand-offs of every tile
        // still take place (bar.sync keeps this warp in step with the MMA warp)
        if (warp == 0 && lane == 0) bar->tinfo[t & 1] = info;
        __syncwarp();
        ptx::bar_sync(kBarDpFree, kBarDqThreads);
        ptx::bar_sync(kBarDsQ + (t & 1), kBarDqThreads);
        has2 = has3;
        has3 = has3 && ahead.next(&apos, &anv, &atok);
        ++t;
        continue;
      }
      tc::fence_after_sync();
      // keys [0, lim) of this warp's 64 columns are seen
      const int32_t lim = (live ? min(nvalid, my_vis - pos0) : 0) - 64 * hh;
      const bool whole = __all_sync(0xffffffffu, lim >= 64);  // no masking in this warp
      const uint32_t s_col = kColS0 + 128 * (t & 1) + 64 * hh, dp_col = kColDPq + 64 * hh;
      // this warp's 64 columns, 32 at a time; dS (bf16) over the first 32 S
      // columns of its half, all already read when written
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {
        uint32_t sr[32], dp[32], pk[16];
        tc::tmem_ld32(lane_addr + s_col + 32 * q, sr);
        tc::tmem_ld32(lane_addr + dp_col + 32 * q, dp);
        tc::tmem_ld_wait();
        if (q == 1) {  // all of this warp's dP(t) is in registers: the next dP may be issued
          if (warp == 0) {
            if (lane == 0) bar->tinfo[t & 1] = info;
            if (has_next && !__all_sync(0xffffffffu, ptx::mbar_wait(&bar->v_full[(t + 1) % kVStages],
                                                                    ((t + 1) / kVStages) & 1)))
              ok = false;
          }
          tc::fence_before_sync();
          __syncwarp();
          ptx::bar_arrive(kBarDpFree, kBarDqThreads);
        }
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = ptx::ffma2(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), c2, nlc2);
          const float2 y = ptx::fadd2(make_float2(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1])), nd2);
          float2 ds = ptx::fmul2(make_float2(fast_exp2(x.x), fast_exp2(x.y)), y);
          if (!whole) {
            const int j = 32 * q + i;
            ds.x = j < lim ? ds.x : 0.f;
            ds.y = j + 1 < lim ? ds.y : 0.f;
          }
          pk[i / 2] = pack_bf16(ds.x, ds.y);
        }
        tc::tmem_st16(lane_addr + s_col + 16 * q, pk);
      }
      if (warp == 1 && has_next2 &&
          !__all_sync(0xffffffffu, ptx::mbar_wait(&bar->k_full[(t + 2) % kKStages], ((t + 2) / kKStages) & 1)))
        ok = false;
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      ptx::bar_arrive(kBarDsQ + (t & 1), kBarDqThreads);
      has2 = has3;
      has3 = has3 && ahead.next(&apos, &anv, &atok);
      ++t;
    }
    // epilogue: dQ = scale * sum dS K.  The destination rows are worked out
    // while the last MMAs run (G divides 64, a power of two: shifts).
    // (the row base goes through an opaque move, so the compiler cannot hoist this
    // work into the tile loop, where it would hold registers across every tile)
    int32_t row_base;
    asm volatile("mov.b32 %0, %1;" : "=r"(row_base) : "r"(part_row));
    const int lg = __ffs(G) - 1;
    float4* dst_k[8];  // the staged path's row pieces: row 4 i + lane / 8 of this warp's 32
    bool valid_k[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int32_t rk = rq * 32 + 4 * i + (lane >> 3);
      valid_k[i] = rk < n_rows;
      dst_k[i] = reinterpret_cast<float4*>(
          dq_part + (static_cast<int64_t>(row_base + ((r0 + rk) >> lg)) * a.Hq + kvh * G + ((r0 + rk) & (G - 1))) * kD);
    }
    if (ok && t > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait(&bar->o_done, 0))) ok = false;
    if (!ok && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
    tc::fence_after_sync();
    const int64_t orow = static_cast<int64_t>(part_row + token) * a.Hq + h;
    if (ok && t > 0) {
      // The Q tile is free once o_done is seen (every S MMA has completed): each
      // warp passes 32 rows x 32 columns at a time through its 4 KB of it (16-byte
      // slot y of row k at y ^ (k & 7)) and stores whole 128-byte row pieces.
      float4* wst = reinterpret_cast<float4*>(sq + (hh * 4 + rq) * 4096);
#pragma unroll 1
      for (int q4 = 2 * hh; q4 < 2 * hh + 2; ++q4) {
        uint32_t acc[32];
        tc::tmem_ld32(lane_addr + kColDQ + 32 * q4, acc);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          wst[lane * 8 + (i ^ (lane & 7))] =
              make_float4(__uint_as_float(acc[4 * i]) * a.scale, __uint_as_float(acc[4 * i + 1]) * a.scale,
                          __uint_as_float(acc[4 * i + 2]) * a.scale, __uint_as_float(acc[4 * i + 3]) * a.scale);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int kr = 4 * i + (lane >> 3), y = lane & 7;
          if (valid_k[i]) dst_k[i][8 * q4 + y] = wst[kr * 8 + (y ^ (kr & 7))];
        }
        __syncwarp();
      }
    } else {  // no key tile (the Q copy was never waited for) or the waits ran out: direct stores
#pragma unroll 1
      for (int q4 = 2 * hh; q4 < 2 * hh + 2; ++q4) {
        uint32_t acc[32];
        if (t > 0) {
          tc::tmem_ld32(lane_addr + kColDQ + 32 * q4, acc);
          tc::tmem_ld_wait();
        }
        if (row_valid) {
          float4* dst = reinterpret_cast<float4*>(dq_part + orow * kD + 32 * q4);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t > 0)
              v = make_float4(__uint_as_float(acc[4 * i]) * a.scale, __uint_as_float(acc[4 * i + 1]) * a.scale,
                              __uint_as_float(acc[4 * i + 2]) * a.scale, __uint_as_float(acc[4 * i + 3]) * a.scale);
            dst[i] = v;
          }
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ========================================================== dK / dV kernel

// Warps 0-7: key threads, two per TMEM lane quarter (warp w: keys of quarter w % 4,
// rows w / 4 * 32 .. + 31 of each 64-row tile); 8: TMA; 9: MMA; 10: sync warp,
// which takes the copy waits off the MMA warp.
constexpr int kKvThreads = 352;
constexpr int kKvProducerWarp = 8, kKvMmaWarp = 9, kKvSyncWarp = 10, kKeyWarps = 8;
// Named barriers (0 is __syncthreads).  kBarHand: the sync warp hands the MMA
// warp each row tile's operands, both sides with bar.sync, so neither runs a
// hand-off ahead.  kBarDs + (g & 1): the key warps hand over P^T, dS^T of row
// tile g (bar.arrive; the MMA warp syncs).  A key warp reaches row tile g + 2
// only after S^T(g + 2) completed, which the MMA warp issues after passing the
// barrier of tile g, so the two parities never mix.
constexpr int kBarHand = 1, kBarHandThreads = 64;
constexpr int kBarDs = 2, kBarDsThreads = (kKeyWarps + 1) * 32;
// P^T / dS^T (bf16 pairs) of rows 16 kk .. 16 kk + 15, relative to the S^T / dP^T
// columns of the tile: rows 0-31 over columns 0-15, rows 32-63 over columns 32-47
// (each key warp writes over the columns it has read; the other half stays intact).
__device__ __forceinline__ uint32_t pt_col(int kk) { return 8u * kk + (kk >= 2 ? 16u : 0u); }
constexpr int kRowsB = 64;      // query rows per tile here: two tiles' S^T / dP^T fit in TMEM
constexpr int kQdStages = 4;    // Q / dO ring: the tile in the elementwise pass, the next one's
                                // S^T / dP^T in the pipe, and two loading
constexpr uint32_t kHalf64 = kRowsB * 128;         // 64 rows x 64 bf16 (one swizzled half)
constexpr uint32_t kTile64 = 2 * kHalf64;          // 64 x 128 bf16
// TMEM: S^T of row-tile parity b at 64 b, dP^T at 128 + 64 b; dV and dK as in the dQ kernel
constexpr uint32_t kColST = 0, kColDPT = 128;

__device__ __forceinline__ uint32_t kstep_off64(int kk) { return ((kk >> 2) * kHalf64 + (kk & 3) * 32) >> 4; }

struct KvBarriers {
  uint64_t kv_full;                 // K and V of the current key tile
  uint64_t qd_full[kQdStages];      // Q, dO (TMA) and L, D (producer lanes) of a row tile
  uint64_t qd_free[kQdStages];      // the row tile's dV / dK MMAs have read Q and dO
  uint64_t s_full[2];               // per row-tile parity: S^T, dP^T ready
  uint64_t kv_free;                 // the key tile's last S^T, dP^T completed: K, V no longer read
  uint64_t o_done;                  // the key tile's last dV / dK MMA completed
  uint64_t drain;
  uint32_t tmem_base;
  // -L log2(e) and -D of the row tile's rows; -inf and 0 for rows without a
  // gradient (past the sequence, or no visible key: L = -inf), whose P is then 0
  alignas(16) float ld[kQdStages][2][kRowsB];
};
// Epilogue staging: each key warp passes 32 keys x 32 columns of dV or dK through
// shared memory so that global stores go out as whole rows
constexpr uint32_t kStageBytes = 4 * 32 * 32 * 4;
constexpr size_t kKvSmem = 1024 + 2 * kTileBytes + 2 * kQdStages * kTile64 + kStageBytes + sizeof(KvBarriers);

// The key threads' pass over one row tile: P^T = exp2(S^T c - L log2 e) and
// dS^T = P^T (dP^T - D) for this thread's key and 32 rows, packed to bf16.
// nl / nd: -L log2(e) and -D of the 32 rows.  Rows i < jlo come before the
// key's position (causal) and get P = 0 (kMasked only).  A key past the end of
// the tile may hold anything; its P^T, dS^T only reach its own dV, dK rows,
// which are not stored.
template <bool kMasked>
__device__ __forceinline__ void key_pass(const uint32_t (&sr)[32], const uint32_t (&dp)[32], const float* nl,
                                         const float* nd, float c, int32_t jlo, uint32_t (&pk)[16],
                                         uint32_t (&dk2)[16]) {
  const float2 c2 = make_float2(c, c);
#pragma unroll
  for (int i4 = 0; i4 < 8; ++i4) {
    const float4 l = reinterpret_cast<const float4*>(nl)[i4];
    const float4 dd = reinterpret_cast<const float4*>(nd)[i4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = 4 * i4 + 2 * h;
      const float2 x = ptx::ffma2(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), c2,
                                  h ? make_float2(l.z, l.w) : make_float2(l.x, l.y));
      float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
      if (kMasked) {
        pp.x = i >= jlo ? pp.x : 0.f;
        pp.y = i + 1 >= jlo ? pp.y : 0.f;
      }
      const float2 y = ptx::fadd2(make_float2(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1])),
                                  h ? make_float2(dd.z, dd.w) : make_float2(dd.x, dd.y));
      const float2 dsv = ptx::fmul2(pp, y);
      pk[i / 2] = pack_bf16(pp.x, pp.y);
      dk2[i / 2] = pack_bf16(dsv.x, dsv.y);
    }
  }
}

__global__ void __launch_bounds__(kKvThreads, 1)
    bwd_dkdv_tc_kernel(PartialArgs a, int32_t key_split, const float* __restrict__ lse, const float* __restrict__ delta,
                       float* __restrict__ dk_pool, float* __restrict__ dv_pool,
                       const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_do,
                       const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sk = smem;                          // K tile
  uint8_t* sv = smem + kTileBytes;             // V tile
  uint8_t* sq = smem + 2 * kTileBytes;         // Q ring
  uint8_t* sdo = sq + kQdStages * kTile64;     // dO ring
  float* stage = reinterpret_cast<float*>(sdo + kQdStages * kTile64);  // epilogue staging
  KvBarriers* bar = reinterpret_cast<KvBarriers*>(sdo + kQdStages * kTile64 + kStageBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // key_split CTAs per (item, K/V head); CTA `split` takes key tiles split,
  // split + key_split, ... of the item
  const int32_t split = static_cast<int32_t>(blockIdx.x % key_split);
  const int32_t kvh = static_cast<int32_t>((blockIdx.x / key_split) % a.Hkv);
  const int32_t item = static_cast<int32_t>(blockIdx.x / (static_cast<int64_t>(key_split) * a.Hkv));

  const WorkView wv(a.work, a.B, a.n_items);
  const int32_t* it = wv.item(item);
  const int32_t h_magic = wv.hdr(kMagic), h_b = wv.hdr(kB), h_n = wv.hdr(kNItems);
  const int32_t seq = __ldg(it + kItSeq);
  const int32_t cu_q = __ldg(it + kItCuQ), q_len = __ldg(it + kItQLen), kv_len = __ldg(it + kItKvLen);
  if (!work_matches(h_magic, h_b, h_n, a.B, a.n_items)) {  // uniform over the CTA
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBadWork);
    return;
  }
  const int32_t G = a.Hq / a.Hkv;
  const int lg = __ffs(G) - 1;  // G divides 64: a power of two
  const int32_t rows = q_len * G;
  const int32_t n_rt = (rows + kRowsB - 1) / kRowsB;  // row tiles of the sequence
  // every key below kv_len gets a gradient (zero if no row sees it)
  TileSeq tiles;
  tiles.ib = ItemBlocks{wv.blocks() + __ldg(it + kItBlockOff),
                        a.block_table + static_cast<int64_t>(seq) * a.max_blocks_per_seq, __ldg(it + kItBlockCnt),
                        a.block_len, a.max_blocks_per_seq, kv_len, kv_len, a.n_pool_blocks};
  // this CTA's key tiles: ordinals split, split + key_split, ... of the item's tiles
  auto next_mine = [&](TileSeq& w, int32_t& ord, int32_t* pos0, int32_t* nv, int32_t* tok) -> bool {
    while (w.next(pos0, nv, tok)) {
      if (ord++ % key_split == split) return true;
    }
    return false;
  };
  if (n_rt == 0) return;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar->kv_full, 1);
    for (int s = 0; s < kQdStages; ++s) {
      ptx::mbar_init(&bar->qd_full[s], 1);
      ptx::mbar_init(&bar->qd_free[s], 1);
    }
    for (int b = 0; b < 2; ++b) ptx::mbar_init(&bar->s_full[b], 1);
    ptx::mbar_init(&bar->kv_free, 1);
    ptx::mbar_init(&bar->o_done, 1);
    ptx::mbar_init(&bar->drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == kKvMmaWarp) {
    tc::tmem_alloc(&bar->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bar->tmem_base;

  // Row tiles are numbered g = 0, 1, ... over all of this CTA's key tiles (n_rt a
  // key tile); tile g uses ring slot g % kQdStages and the TMEM pair of parity g & 1.
  if (warp == kKvProducerWarp) {
    // ------------------------------------------------------------- producer
    // Per key tile: K and V, once the previous key tile's last S^T / dP^T have
    // completed (kv_free; the dV / dK MMAs read neither), then every row tile's Q, dO by
    // TMA and L, D by the warp's lanes.  The next key tile's K and V are
    // prefetched into L2 when a key tile starts.
    if (lane == 0) {
      ptx::prefetch_tmap(&tmap_q);
      ptx::prefetch_tmap(&tmap_do);
      ptx::prefetch_tmap(&tmap_k);
      ptx::prefetch_tmap(&tmap_v);
    }
    TileSeq walk = tiles;
    int32_t ord = 0, pos0, nv, tok, kt = 0, rt = 0, kv_issued = 0;
    bool ok = true;
    bool have = next_mine(walk, ord, &pos0, &nv, &tok);
    while (ok && have) {
      const int32_t cur_tok = tok;
      int32_t p2 = 0, nv2 = 0, tok2 = 0;
      const bool have_next = next_mine(walk, ord, &p2, &nv2, &tok2);
      // one kv_free phase per key tile, in order: the wait for phase kt - 1
      // follows the load that needed phase kt - 2
      if (kt > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait(&bar->kv_free, (kt - 1) & 1))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&bar->kv_full, 2 * kTileBytes);
        ptx::tma_load_3d(sk, &tmap_k, 0, kvh, cur_tok, &bar->kv_full);
        ptx::tma_load_3d(sk + kHalfBytes, &tmap_k, 64, kvh, cur_tok, &bar->kv_full);
        ptx::tma_load_3d(sv, &tmap_v, 0, kvh, cur_tok, &bar->kv_full);
        ptx::tma_load_3d(sv + kHalfBytes, &tmap_v, 64, kvh, cur_tok, &bar->kv_full);
        if (have_next) {
          ptx::tma_prefetch_3d(&tmap_k, 0, kvh, tok2);
          ptx::tma_prefetch_3d(&tmap_k, 64, kvh, tok2);
          ptx::tma_prefetch_3d(&tmap_v, 0, kvh, tok2);
          ptx::tma_prefetch_3d(&tmap_v, 64, kvh, tok2);
        }
      }
      ++kv_issued;
      for (int32_t r = 0; r < n_rt; ++r, ++rt) {
        const int s = rt % kQdStages;
        // -L log2(e) and -D of rows r*64 .. r*64+63 (-inf, 0 where no gradient),
        // loaded before the slot is free so that their latency overlaps the wait
        float nl[kRowsB / 32], nd[kRowsB / 32];
#pragma unroll
        for (int u = 0; u < kRowsB / 32; ++u) {
          const int32_t row = r * kRowsB + 32 * u + lane;
          float L = -INFINITY, Dv = 0.f;
          if (row < rows) {
            const int64_t g = static_cast<int64_t>(cu_q + (row >> lg)) * a.Hq + kvh * G + (row & (G - 1));
            L = __ldg(lse + g);
            Dv = __ldg(delta + g);
          }
          nl[u] = L != -INFINITY ? -L * kLog2e : -INFINITY;
          nd[u] = L != -INFINITY ? -Dv : 0.f;
        }
        if (rt >= kQdStages &&
            !__all_sync(0xffffffffu, ptx::mbar_wait(&bar->qd_free[s], ((rt - kQdStages) / kQdStages) & 1))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int u = 0; u < kRowsB / 32; ++u) {
          bar->ld[s][0][32 * u + lane] = nl[u];
          bar->ld[s][1][32 * u + lane] = nd[u];
        }
        __syncwarp();
        if (lane == 0) {
          const int32_t tok0 = cu_q + ((r * kRowsB) >> lg);
          ptx::mbar_arrive_expect_tx(&bar->qd_full[s], 2 * kTile64);
          ptx::tma_load_3d(sq + s * kTile64, &tmap_q, 0, kvh * G, tok0, &bar->qd_full[s]);
          ptx::tma_load_3d(sq + s * kTile64 + kHalf64, &tmap_q, 64, kvh * G, tok0, &bar->qd_full[s]);
          ptx::tma_load_3d(sdo + s * kTile64, &tmap_do, 0, kvh * G, tok0, &bar->qd_full[s]);
          ptx::tma_load_3d(sdo + s * kTile64 + kHalf64, &tmap_do, 64, kvh * G, tok0, &bar->qd_full[s]);
        }
      }
      ++kt;
      have = have_next;
      tok = tok2;
    }
    if (!ok && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
    if (walk.bad_seen && lane == 0) atomicOr(a.status, 1u);
    // every copy issued has landed before shared memory is released
    if (lane == 0) {
      if (kv_issued > 0 && !ptx::mbar_wait(&bar->kv_full, (kv_issued - 1) & 1))
        atomicOr(a.status, ptx::kStatusTimeout);
      for (int32_t v = max(0, rt - kQdStages); v < rt; ++v)
        if (!ptx::mbar_wait(&bar->qd_full[v % kQdStages], (v / kQdStages) & 1)) atomicOr(a.status, ptx::kStatusTimeout);
    }
  } else if (warp == kKvSyncWarp) {
    // ------------------------------------------------------------ sync warp
    // Per row tile g: waits until K, V (first row tile of a key tile) and Q, dO,
    // L, D of tile g have landed, then meets the MMA warp on kBarHand.  It cannot
    // run ahead: each hand-off needs the MMA warp.  Once a wait has run out it
    // stops waiting but keeps taking part in the hand-offs.
    TileSeq walk = tiles;
    int32_t ord = 0, pos0, nv, tok, kt = 0, rt = 0;
    bool ok = true;
    while (next_mine(walk, ord, &pos0, &nv, &tok)) {
      for (int32_t r = 0; r < n_rt; ++r, ++rt) {
        if (ok && r == 0) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->kv_full, kt & 1));
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->qd_full[rt % kQdStages], (rt / kQdStages) & 1));
        ptx::bar_sync(kBarHand, kBarHandThreads);
      }
      ++kt;
    }
    if (!ok && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
  } else if (warp == kKvMmaWarp) {
    // ------------------------------------------------------------------ MMA
    // Row tile g uses the TMEM pair of parity b = g & 1.  S^T(g+1), dP^T(g+1)
    // are issued before the key threads' pass over tile g ends, so the pipe
    // works while they run; then dV += P^T(g) dO(g), dK += dS^T(g) Q(g).
    // S^T(g+2) reuses tile g's columns and is issued after those MMAs (in
    // order).  At the last row tile of a key tile the dV / dK MMAs go first:
    // the next key tile's S^T waits for its K and V, which are loaded only
    // once this tile's last S^T has completed.  The waits are named barriers
    // (no mbarrier wait on this warp).  The other roles keep taking part in
    // every hand-off after a wait of theirs ran out, so this warp needs no
    // abort test: it may then run MMAs on stale operands, which reach no
    // output (the status word reports the timeout).
    const uint32_t idesc_s = tc::idesc_bf16_f32(kN, kRowsB, false, false);
    const uint32_t idesc_acc = tc::idesc_bf16_f32(kN, kD, false, true);
    const tc::Desc dk = tc::split(tc::smem_desc(ptx::smem_addr(sk), 16, 1024, tc::kSwizzle128B));
    const tc::Desc dv = tc::split(tc::smem_desc(ptx::smem_addr(sv), 16, 1024, tc::kSwizzle128B));
    const tc::Desc dq = tc::split(tc::smem_desc(ptx::smem_addr(sq), 16, 1024, tc::kSwizzle128B));
    const tc::Desc ddo = tc::split(tc::smem_desc(ptx::smem_addr(sdo), 16, 1024, tc::kSwizzle128B));
    const tc::Desc dq_mn = tc::split(tc::smem_desc(ptx::smem_addr(sq), kHalf64, 1024, tc::kSwizzle128B));
    const tc::Desc ddo_mn = tc::split(tc::smem_desc(ptx::smem_addr(sdo), kHalf64, 1024, tc::kSwizzle128B));
    // S^T, dP^T of row tile g (after meeting the sync warp: its operands landed);
    // after the last row tile of a key tile, kv_free tells the producer that K
    // and V may be overwritten
    auto hand_and_issue_s = [&](int32_t g, bool last_of_key_tile) {
      ptx::bar_sync(kBarHand, kBarHandThreads);
      tc::fence_after_sync();
      if (tc::elect_one()) {
        const uint32_t qoff = (g % kQdStages) * (kTile64 >> 4);
        const uint32_t b = static_cast<uint32_t>(g & 1);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          tc::mma_ss_fast(tmem + kColST + 64 * b, dk, kstep_off(kk), dq, qoff + kstep_off64(kk), idesc_s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          tc::mma_ss_fast(tmem + kColDPT + 64 * b, dv, kstep_off(kk), ddo, qoff + kstep_off64(kk), idesc_s, kk > 0);
        tc::commit(&bar->s_full[b]);
        if (last_of_key_tile) tc::commit(&bar->kv_free);
      }
      __syncwarp();
    };
    // dV, dK += row tile g (after the key warps handed over its P^T, dS^T)
    auto sync_and_issue_acc = [&](int32_t g, bool first, bool last) {
      const int b = g & 1;
      ptx::bar_sync(kBarDs + b, kBarDsThreads);
      tc::fence_after_sync();
      if (tc::elect_one()) {
        const uint32_t qoff = (g % kQdStages) * (kTile64 >> 4);
#pragma unroll
        for (int kk = 0; kk < kRowsB / 16; ++kk)
          tc::mma_ts_fast(tmem + kColAcc0, tmem + kColST + 64 * b + pt_col(kk), ddo_mn, qoff + kk * (2048 >> 4),
                          idesc_acc, (!first || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kRowsB / 16; ++kk)
          tc::mma_ts_fast(tmem + kColAcc1, tmem + kColDPT + 64 * b + pt_col(kk), dq_mn, qoff + kk * (2048 >> 4),
                          idesc_acc, (!first || kk > 0) ? 1u : 0u);
        tc::commit(&bar->qd_free[g % kQdStages]);
        if (last) tc::commit(&bar->o_done);
      }
      __syncwarp();
    };
    TileSeq walk = tiles;
    int32_t ord = 0, pos0, nv, tok, rt = 0;
    bool have = next_mine(walk, ord, &pos0, &nv, &tok);
    if (have) hand_and_issue_s(0, n_rt == 1);
    while (have) {
      const bool have_next = next_mine(walk, ord, &pos0, &nv, &tok);
      for (int32_t r = 0; r < n_rt; ++r, ++rt) {
        if (r + 1 < n_rt) {
          hand_and_issue_s(rt + 1, r + 2 == n_rt);
          sync_and_issue_acc(rt, r == 0, false);
        } else {
          sync_and_issue_acc(rt, r == 0, true);
          if (have_next) hand_and_issue_s(rt + 1, n_rt == 1);
        }
      }
      have = have_next;
    }
    if (tc::elect_one()) tc::commit(&bar->drain);
    __syncwarp();
    if (!ptx::mbar_wait(&bar->drain, 0) && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
  } else {
    // ------------------------------------------------ key threads (P^T, dS^T)
    const int kq = warp & 3, hh = warp >> 2;  // TMEM lane quarter; 32-row half of each row tile
    const int32_t k = kq * 32 + lane;         // TMEM lane = key of the tile
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(kq * 32) << 16);
    const float c = a.scale * kLog2e;
    TileSeq walk = tiles;
    int32_t ord = 0, pos0, nv, tok, kt = 0, rt = 0;
    bool ok = true;
    while (next_mine(walk, ord, &pos0, &nv, &tok)) {
      // causal: the row (token t, head) sees this key iff t >= pos - (kv_len - q_len)
      const int32_t t_first = a.causal ? min(q_len, max(0, pos0 + k - (kv_len - q_len))) : 0;
      for (int32_t r = 0; r < n_rt; ++r, ++rt) {
        const int s = rt % kQdStages, b = rt & 1;
        if (ok)
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->qd_full[s], (rt / kQdStages) & 1)) &&
               __all_sync(0xffffffffu, ptx::mbar_wait(&bar->s_full[b], (rt >> 1) & 1));
        if (!ok) {
          // no more TMEM work, but every hand-off still takes place (bar.sync
          // keeps this warp in step with the MMA warp)
          ptx::bar_sync(kBarDs + b, kBarDsThreads);
          continue;
        }
        tc::fence_after_sync();
        // this thread's rows are 32 hh + i of the tile; causal: those below
        // t_first * G - r * 64 come before the key
        const int32_t jlo = t_first * G - r * kRowsB - 32 * hh;
        const float* nl = bar->ld[s][0] + 32 * hh;
        const float* nd = bar->ld[s][1] + 32 * hh;
        const uint32_t st_col = kColST + 64 * b + 32 * hh, dpt_col = kColDPT + 64 * b + 32 * hh;
        uint32_t sr[32], dp[32], pk[16], dk2[16];
        tc::tmem_ld32(lane_addr + st_col, sr);
        tc::tmem_ld32(lane_addr + dpt_col, dp);
        tc::tmem_ld_wait();
        if (__all_sync(0xffffffffu, jlo <= 0))
          key_pass<false>(sr, dp, nl, nd, c, jlo, pk, dk2);
        else
          key_pass<true>(sr, dp, nl, nd, c, jlo, pk, dk2);
        // P^T over this half's first 16 S^T columns, dS^T over its first 16 dP^T
        // columns: both already read, and the other half's columns stay intact
        tc::tmem_st16(lane_addr + st_col, pk);
        tc::tmem_st16(lane_addr + dpt_col, dk2);
        tc::tmem_st_wait();
        tc::fence_before_sync();
        ptx::bar_arrive(kBarDs + b, kBarDsThreads);
      }
      // epilogue: this key's dV and dK = scale * sum dS^T Q, by the warps of the
      // first half (one per lane quarter); the others go on to the next key tile
      if (hh == 1) {
        ++kt;
        continue;
      }
      if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->o_done, kt & 1));
      if (!ok) {
        ++kt;
        continue;
      }
      tc::fence_after_sync();
      // Each chunk of 32 columns goes through this warp's 32 x 32 staging block
      // (16-byte slot x of row k at x ^ (k & 7): no bank conflicts either way), then
      // out as whole 128-byte row pieces, four keys per store instruction.
      float4* wst = reinterpret_cast<float4*>(stage + kq * 32 * 32);
#pragma unroll 1
      for (int q4 = 0; q4 < 8; ++q4) {
        const bool is_k = q4 >= 4;
        uint32_t acc[32];
        tc::tmem_ld32(lane_addr + (is_k ? kColAcc1 : kColAcc0) + 32 * (q4 & 3), acc);
        tc::tmem_ld_wait();
        const float f = is_k ? a.scale : 1.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          wst[lane * 8 + (i ^ (lane & 7))] =
              make_float4(__uint_as_float(acc[4 * i]) * f, __uint_as_float(acc[4 * i + 1]) * f,
                          __uint_as_float(acc[4 * i + 2]) * f, __uint_as_float(acc[4 * i + 3]) * f);
        __syncwarp();
        float* pool = is_k ? dk_pool : dv_pool;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int kr = 4 * i + (lane >> 3), x = lane & 7;  // key of the warp, 16-byte slot
          const int key = kq * 32 + kr;
          if (key < nv) {
            const int64_t krow = (static_cast<int64_t>(tok) + key) * a.Hkv + kvh;  // pool token tok + key
            reinterpret_cast<float4*>(pool + krow * kD + 32 * (q4 & 3))[x] = wst[kr * 8 + (x ^ (kr & 7))];
          }
        }
        __syncwarp();
      }
      ++kt;
    }
    if (!ok && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kKvMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Maps over q / dout ([total_q, Hq, d]: boxes of `rows` query rows = rows / G
// tokens x the G heads of a K/V head) and the K / V pools (128-key boxes).
int make_maps(const PartialArgs& a, const void* dout, int rows, CUtensorMap* tq, CUtensorMap* tdo, CUtensorMap* tk,
              CUtensorMap* tv) {
  const int32_t G = a.Hq / a.Hkv;
  const uint64_t qdims[3] = {kD, static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(a.total_q)};
  const uint64_t qstrides[2] = {kD * 2ull, static_cast<uint64_t>(a.Hq) * kD * 2ull};
  const uint32_t qbox[3] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(rows / G)};
  int st = encode_bf16_3d(tq, a.q, qdims, qstrides, qbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == SPLITKV_OK) st = encode_bf16_3d(tdo, dout, qdims, qstrides, qbox, CU_TENSOR_MAP_SWIZZLE_128B);
  const uint64_t kdims[3] = {kD, static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(a.n_pool_blocks) * a.block_len};
  const uint64_t kstrides[2] = {kD * 2ull, static_cast<uint64_t>(a.Hkv) * kD * 2ull};
  const uint32_t kbox[3] = {64, 1, kN};
  if (st == SPLITKV_OK) st = encode_bf16_3d(tk, a.k_pool, kdims, kstrides, kbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == SPLITKV_OK) st = encode_bf16_3d(tv, a.v_pool, kdims, kstrides, kbox, CU_TENSOR_MAP_SWIZZLE_128B);
  return st;
}

}  // namespace

bool bwd_tc_supports(const PartialArgs& a) {
  if (a.dtype != SPLITKV_BF16 || a.d != kD || a.Hkv <= 0 || a.Hq % a.Hkv != 0) return false;
  const int32_t G = a.Hq / a.Hkv;
  return G >= 1 && G <= kRowsB && kRowsB % G == 0 && a.block_len % kN == 0 &&
         static_cast<int64_t>(a.n_pool_blocks) * a.block_len < (1ll << 31);
}

int launch_bwd_tc(const PartialArgs& a, const void* dout, const float* lse, const float* delta, float* dq_part,
                  float* dk_pool, float* dv_pool, cudaStream_t stream) {
  const int32_t G = a.Hq / a.Hkv;
  const int32_t units = (a.max_q_len * G + kRows - 1) / kRows;
  const int64_t grid = static_cast<int64_t>(units) * a.Hkv * a.n_items;
  if (grid == 0) return SPLITKV_OK;
  if (grid > 0x7fffffffLL) return fail(SPLITKV_ERR_UNSUPPORTED, "too many backward units");
  CUtensorMap tq, tdo, tk, tv, tq64, tdo64, tk2, tv2;
  int st = make_maps(a, dout, kRows, &tq, &tdo, &tk, &tv);
  if (st == SPLITKV_OK) st = make_maps(a, dout, kRowsB, &tq64, &tdo64, &tk2, &tv2);
  if (st != SPLITKV_OK) return st;
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kDqSmem));
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "backward smem attribute: %s", cudaGetErrorString(e));
  bwd_dq_tc_kernel<<<static_cast<unsigned>(grid), kThreads, kDqSmem, stream>>>(a, lse, delta, dq_part, units, tq, tdo,
                                                                                 tk, tv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "backward dQ launch: %s", cudaGetErrorString(e));
  // dK/dV CTAs per (item, K/V head): as few as keep about six CTAs per SM in the
  // launch, so each CTA's set-up, first copies and closing stores cover as many key
  // tiles as the grid allows (measured: 16 per pair cost 6-8% on the 64-shard
  // workloads and nearly doubled the decode backward against this choice)
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  const int64_t pairs = static_cast<int64_t>(a.Hkv) * a.n_items;
  const int32_t key_split = static_cast<int32_t>(std::min<int64_t>(16, std::max<int64_t>(1, (6ll * sms + pairs - 1) / pairs)));
  const int64_t grid_kv = static_cast<int64_t>(key_split) * pairs;
  if (grid_kv > 0x7fffffffLL) return fail(SPLITKV_ERR_UNSUPPORTED, "too many backward units");
  e = cudaFuncSetAttribute(bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kKvSmem));
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "backward smem attribute: %s", cudaGetErrorString(e));
  bwd_dkdv_tc_kernel<<<static_cast<unsigned>(grid_kv), kKvThreads, kKvSmem, stream>>>(a, key_split, lse, delta, dk_pool, dv_pool,
                                                                                     tq64, tdo64, tk, tv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "backward dK/dV launch: %s", cudaGetErrorString(e));
  return SPLITKV_OK;
}

}  // namespace splitkv

// Tensor-core partial attention for sm_103a: TMA + tcgen05 (UMMA) + TMEM.
//
// Used when the query rows of a (sequence, K/V head) pair fill tensor-core
// tiles: bf16, d = 128, block_len % 128 == 0, G = Hq / Hkv dividing 128.
// Computes, for every work item (a shard's blocks of one sequence), the
// shard's partial (O_i, L_i) of the Split-KV card's local attention step
// ("Timeline": keys and values stay local; only a query-sized result leaves).
//
// One CTA = one (work item, K/V head, 256 query rows) unit, split into two
// 128-row query tiles A and B that share every K/V tile.  Row r of the unit is
// token r / G, query head kvh*G + r % G.  Warp roles (384 threads, three
// warpgroups; the softmax groups take 216 registers a thread, the third 72):
//   warps 0-3  softmax + epilogue of tile A: thread i owns row i (TMEM lane i);
//   warps 4-7  the same for tile B;
//   warp 8     TMA producer: both Q tiles once, then K and V tiles of 128 keys
//              from the paged pool (3-D maps over [tokens, Hkv, d], 128-byte
//              swizzle, two 64-column halves per tile) into two-stage rings;
//   warp 9     TMEM allocation and MMA issue (one lane, chosen by elect.sync);
//   warp 10    barrier waits for the MMA warp: it waits on the K/V and S
//              barriers, zeroes the V tail of a partial tile and hands each
//              ready point to warp 9 through a named barrier, so the issuing
//              thread never pays an mbarrier wait;
//   warp 11    idle (it completes the third warpgroup).
// TMEM (512 columns): S_A | O_A | S_B | O_B, 128 fp32 columns each.
// Per KV tile j and query tile X:
//   S_X = Q_X K_j^T      tcgen05.mma kind::f16, M = N = 128, fp32 in TMEM;
//   softmax_X            rows read S_X with tcgen05.ld, keep a running max and
//                        sum in base 2, and write P_X = exp2(s*c - m) as bf16
//                        into the first 64 columns of S_X (tcgen05.st);
//   O_X += P_X V_j       tcgen05.mma with A = P_X from TMEM, B = V_j (MN-major);
//                        P_X goes to the MMA warp in two 64-key halves, so the
//                        first half's PV runs while the second is computed.
// The tensor pipe runs S_A, S_B, PV_A, S_A', PV_B, S_B', ...: while one query
// tile's softmax runs, the other tile's MMAs keep the tensor cores busy.  The
// running max is only moved (and O rescaled through TMEM) when it grows by
// more than 2^8, so P stays <= 256 and the common tile needs no O traffic.
//
// Keys past the sequence end (pool slots that may hold anything) get score
// -inf, and their V rows in a partial tile are zeroed in shared memory before
// the P.V MMAs, so they contribute exactly nothing.  Every wait has a time
// limit; on expiry the status word gets bit 2, the warp stops waiting and
// stops its TMEM work, but keeps taking part in every named-barrier hand-off,
// so no other warp blocks on it, and the CTA unwinds at the end.

#include <cmath>

#include "device_common.cuh"
#include "launch.h"
#include "merge_row.cuh"
#include "ptx.cuh"
#include "status.h"
#include "tc_ptx.cuh"
#include "tensor_map.h"

namespace splitkv {
namespace {

constexpr int kD = 128;
constexpr int kMT = 128;      // rows per query tile
constexpr int kM = 2 * kMT;   // rows per CTA
constexpr int kN = 128;       // keys per KV tile
constexpr int kStages = 2;    // K and V ring depth
constexpr int kThreads = 384;
// Register split: launched at 168 a thread (384 x 168 = 64512), the two softmax
// warpgroups grow to 216 and the producer / MMA warpgroup shrinks to 72:
// 2 x 128 x 216 + 128 x 72 = 64512 (per SM sub-partition 216 + 216 + 72 <= 512).
constexpr int kRegsSoftmax = 216, kRegsOther = 72;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kSyncWarp = 10;
// Named barriers (0 is __syncthreads).  The MMA warp syncs on each; the others
// only arrive:  Q and K(0) ready (sync warp);  tile t of query tile A ready:
// P_A(t) written (the four softmax warps of A) and V(t), K(t+1) landed (sync
// warp);  P_B(t) written (the four softmax warps of B).
constexpr int kBarPrologue = 1, kBarTileA = 2, kBarTileB = 3;
constexpr int kBarMerge = 4;  // the softmax warps, around the in-launch merge's ticket
// Second halves of P: keys 64-127 of tile A / B written (the four softmax warps
// of the tile and the MMA warp)
constexpr int kBarTileA2 = 5, kBarTileB2 = 6, kBarHalfThreads = 160;
constexpr int kBarPrologueThreads = 64, kBarTileAThreads = 192, kBarTileBThreads = 160;
constexpr uint32_t kHalfBytes = kN * 64 * 2;     // 128 rows x 64 bf16 (one swizzled half)
constexpr uint32_t kTileBytes = 2 * kHalfBytes;  // 32 KB: one Q, K or V tile
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

// TMEM columns of query tile x: scores (P aliases their first 64) and output.
__host__ __device__ constexpr uint32_t col_s(int x) { return x ? 256u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int x) { return x ? 384u : 128u; }

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[kStages], v_full[kStages];
  // kv_free[j % kStages] completes the j-th release: K tile j and V tile j-1
  // have been consumed by their MMAs.  S(j) of the last query tile is the last
  // MMA to read either, so one softmax thread of that tile arrives once it has
  // seen S(j) complete (MMAs complete in issue order).
  uint64_t kv_free[kStages];
  uint64_t s_full[2], o_done[2];  // per query tile
  uint64_t drain;
  uint32_t tmem_base;
  int32_t first;    // the unit has a key tile (sync warp -> MMA warp, before the prologue barrier)
  int32_t next[2];  // next[t & 1]: tile t + 1 exists (sync warp -> MMA warp, before barrier A of tile t)
  int32_t last;     // in-launch merge: this CTA took the last ticket of its unit
};

constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kTileBytes * (2 + 2 * kStages) + sizeof(Barriers);

// The unit's KV tiles: per block of the item, keys [lo, lo + n) some row of the
// unit can see, cut into kN-key tiles.  All roles walk the same sequence.
struct TileWalk {
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

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

__global__ void __launch_bounds__(kThreads, 1)
    partial_tc_kernel(PartialArgs a, int32_t units_per_item, const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment: the 128-byte swizzle pattern repeats every 8 rows of 128 B.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem;                       // Q_A, Q_B
  uint8_t* sk = smem + 2 * kTileBytes;      // K ring
  uint8_t* sv = sk + kStages * kTileBytes;  // V ring
  Barriers* bar = reinterpret_cast<Barriers*>(sv + kStages * kTileBytes);

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
  const int32_t blk_off = __ldg(it + kItBlockOff), blk_cnt = __ldg(it + kItBlockCnt);
  const int32_t part_row = __ldg(it + kItPartRow);
  const int32_t cu_q = __ldg(it + kItCuQ), q_len = __ldg(it + kItQLen), kv_len = __ldg(it + kItKvLen);
  if (!work_matches(h_magic, h_b, h_n, a.B, a.n_items)) {  // uniform over the CTA
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBadWork);
    return;
  }
  const int32_t G = a.Hq / a.Hkv;
  const int32_t rows = q_len * G;
  const int32_t r0 = utile * kM;
  if (r0 >= rows) return;  // uniform over the CTA
  if (part_row < 0 || static_cast<int64_t>(part_row) + q_len > a.part_rows) {
    if (threadIdx.x == 0) atomicOr(a.status, 2u);
    return;
  }
  const int32_t n_rows = min(kM, rows - r0);
  const bool has_b = n_rows > kMT;  // uniform: the second query tile holds rows
  const int32_t vis_last = visible_keys(q_len, kv_len, (r0 + n_rows - 1) / G, a.causal);
  const TileWalk walk{wv.blocks() + blk_off, a.block_table + static_cast<int64_t>(seq) * a.max_blocks_per_seq,
                      blk_cnt, a.block_len, a.max_blocks_per_seq, kv_len, vis_last, a.n_pool_blocks};

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&bar->k_full[s], 1);
      ptx::mbar_init(&bar->v_full[s], 1);
      ptx::mbar_init(&bar->kv_free[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(&bar->s_full[x], 1);
      ptx::mbar_init(&bar->o_done[x], 1);
    }
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

  if (warp >= 8) {
  // Each role's code sits under its own register-budget change, so the
  // compiler sizes every role for the budget it runs with.
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmap_q);
      ptx::prefetch_tmap(&tmap_k);
      ptx::prefetch_tmap(&tmap_v);
      ptx::mbar_arrive_expect_tx(&bar->q_full, (has_b ? 2 : 1) * kTileBytes);
      for (int x = 0; x < (has_b ? 2 : 1); ++x) {
        const int32_t tok0 = cu_q + (r0 + x * kMT) / G;
        ptx::tma_load_3d(sq + x * kTileBytes, &tmap_q, 0, kvh * G, tok0, &bar->q_full);
        ptx::tma_load_3d(sq + x * kTileBytes + kHalfBytes, &tmap_q, 64, kvh * G, tok0, &bar->q_full);
      }
      int32_t t = 0;
      bool ok = true;
      for (int32_t bi = 0; bi < blk_cnt && ok; ++bi) {
        int32_t lo, n;
        bool bad;
        const int32_t phys = walk.block(bi, &lo, &n, &bad);
        if (bad) atomicOr(a.status, 1u);
        if (phys < 0) continue;
        for (int32_t off = 0; off < n; off += kN, ++t) {
          const int32_t tok = phys * a.block_len + off;
          const int s = t % kStages;
          // K(t) reuses K(t - kStages)'s slot: release t - kStages; V(t) reuses
          // V(t - kStages)'s slot: release t - kStages + 1
          if (t >= kStages && !ptx::mbar_wait(&bar->kv_free[s], ((t - kStages) / kStages) & 1)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&bar->k_full[s], kTileBytes);
          ptx::tma_load_3d(sk + s * kTileBytes, &tmap_k, 0, kvh, tok, &bar->k_full[s]);
          ptx::tma_load_3d(sk + s * kTileBytes + kHalfBytes, &tmap_k, 64, kvh, tok, &bar->k_full[s]);
          if (t >= kStages &&
              !ptx::mbar_wait(&bar->kv_free[(t + 1) % kStages], ((t - kStages + 1) / kStages) & 1)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&bar->v_full[s], kTileBytes);
          ptx::tma_load_3d(sv + s * kTileBytes, &tmap_v, 0, kvh, tok, &bar->v_full[s]);
          ptx::tma_load_3d(sv + s * kTileBytes + kHalfBytes, &tmap_v, 64, kvh, tok, &bar->v_full[s]);
        }
      }
      if (!ok) atomicOr(a.status, ptx::kStatusTimeout);
      // every copy issued has landed before shared memory is released
      if (!ptx::mbar_wait(&bar->q_full, 0)) atomicOr(a.status, ptx::kStatusTimeout);
      for (int32_t v = max(0, t - kStages); v < t; ++v) {
        if (!ptx::mbar_wait(&bar->k_full[v % kStages], (v / kStages) & 1)) atomicOr(a.status, ptx::kStatusTimeout);
        if (!ptx::mbar_wait(&bar->v_full[v % kStages], (v / kStages) & 1)) atomicOr(a.status, ptx::kStatusTimeout);
      }
    }
  } else if (warp == kMmaWarp || warp == kSyncWarp) {
    // The MMA warp and the sync warp walk the same tile sequence.
    int32_t bi = 0, off = 0, n = 0;
    bool have = false;
    auto next_tile = [&](int32_t* nvalid) -> bool {
      while (true) {
        if (have && off + kN < n) {
          off += kN;
          *nvalid = min(kN, n - off);
          return true;
        }
        have = false;
        while (bi < blk_cnt) {
          int32_t lo;
          bool bad;
          const int32_t phys = walk.block(bi++, &lo, &n, &bad);
          if (phys >= 0) {
            have = true;
            off = 0;
            *nvalid = min(kN, n);
            return true;
          }
        }
        return false;
      }
    };
    if (warp == kSyncWarp) {
      // ------------------------------------------------------------ sync warp
      // Takes every mbarrier wait off the MMA warp.  Arrives on the prologue
      // barrier once Q and K(0) have landed (publishing whether the unit has a
      // key tile), then per tile t on barrier A once S_A(t) has completed and
      // V(t), K(t+1) have landed, publishing whether tile t+1 exists.  Seeing
      // S_A(t) complete keeps it from running a tile ahead: S_A(t) is issued
      // only after the MMA warp passed barrier A of tile t-1.  In a partial
      // tile it zeroes the V rows of keys past the end (P is 0 there, and the
      // slots may hold anything, NaN included).  Once a wait has run out it
      // stops waiting and zeroing but still takes part in every hand-off, with
      // bar.sync so that it stays in step with the MMA warp.
      bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->q_full, 0));
      int32_t nv_cur = 0, nv_next = 0;
      bool has_cur = next_tile(&nv_cur);
      if (ok && has_cur) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->k_full[0], 0));
      if (lane == 0) bar->first = has_cur ? 1 : 0;
      __syncwarp();
      ptx::bar_arrive(kBarPrologue, kBarPrologueThreads);
      int32_t t = 0;
      while (has_cur) {
        const bool has_next = next_tile(&nv_next);
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->s_full[0], t & 1));
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->v_full[t % kStages], (t / kStages) & 1));
        if (ok && has_next)
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->k_full[(t + 1) % kStages], ((t + 1) / kStages) & 1));
        if (ok && nv_cur < kN) {
          uint8_t* vtile = sv + (t % kStages) * kTileBytes;
          const int cc = lane & 15;  // 16-byte piece of a 256-byte row (two swizzled halves)
          for (int r = nv_cur + (lane >> 4); r < kN; r += 2)
            reinterpret_cast<uint4*>(vtile + (cc < 8 ? 0 : kHalfBytes) + r * 128)[cc & 7] = make_uint4(0, 0, 0, 0);
          tc::fence_proxy_async_smem();  // visible to the tensor cores' reads
        }
        if (lane == 0) bar->next[t & 1] = has_next ? 1 : 0;
        __syncwarp();
        if (ok)
          ptx::bar_arrive(kBarTileA, kBarTileAThreads);
        else
          ptx::bar_sync(kBarTileA, kBarTileAThreads);
        ++t;
        has_cur = has_next;
        nv_cur = nv_next;
      }
      if (!ok && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
    } else {
    // ------------------------------------------------------------------ MMA
    // One elected lane issues every tcgen05.mma and commit (elect.sync keeps
    // the operands on the uniform datapath: an MMA then costs the issuing
    // thread about 17 clk against 48 under a lane test, next to the 64 clk the
    // tensor pipe takes to run it).  The loop does nothing else per tile: four named-barrier waits (cheap once
    // the hand-off is there; one per half of each P), one shared-memory word, the
    // PV halves and the next S of tiles A and B written out with their tile index
    // fixed, two commits.  Partial tiles need no
    // branch here (the sync warp zeroed their tail of V); the roles whose waits
    // ran out keep taking part in the hand-offs, so no abort test either.
    const uint32_t idesc_qk = tc::idesc_bf16_f32(kMT, kN, false, false);
    const uint32_t idesc_pv = tc::idesc_bf16_f32(kMT, kD, false, true);
    // Descriptors of every operand tile, built once; an MMA only adds an offset.
    const tc::Desc desc_q0 = tc::split(tc::smem_desc(ptx::smem_addr(sq), 16, 1024, tc::kSwizzle128B));
    const tc::Desc desc_k0 = tc::split(tc::smem_desc(ptx::smem_addr(sk), 16, 1024, tc::kSwizzle128B));
    const tc::Desc desc_v0 = tc::split(tc::smem_desc(ptx::smem_addr(sv), kHalfBytes, 1024, tc::kSwizzle128B));
    constexpr uint32_t kTile16 = kTileBytes >> 4;  // one tile, in descriptor address units
    // S_X = Q_X K^T for KV tile t (K in stage t % kStages); lane 0 only
    auto issue_s = [&](const int x, const int32_t t) {
      const uint32_t qoff = x * kTile16, koff = (t % kStages) * kTile16;
      const uint32_t d_col = tmem + col_s(x);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
        tc::mma_ss_fast(d_col, desc_q0, qoff + off, desc_k0, koff + off, idesc_qk, kk > 0);
      }
      tc::commit(&bar->s_full[x]);
    };
    // O_X (+)= P_X V(t) over keys 16 k0 .. 16 k1 - 1, P_X from TMEM, V in stage
    // t % kStages; tile 0 starts the sum
    auto issue_pv = [&](const int x, const int32_t t, const int k0, const int k1) {
      const uint32_t o_col = tmem + col_o(x), p_col = tmem + col_s(x), voff = (t % kStages) * kTile16;
#pragma unroll
      for (int kk = k0; kk < k1; ++kk)
        tc::mma_ts_fast(o_col, p_col + 8 * kk, desc_v0, voff + kk * (2048 >> 4), idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
    };
    ptx::bar_sync(kBarPrologue, kBarPrologueThreads);  // Q, K(0); bar->first
    if (*reinterpret_cast<volatile int32_t*>(&bar->first) != 0) {
      tc::fence_after_sync();
      if (tc::elect_one()) {
        issue_s(0, 0);
        if (has_b) issue_s(1, 0);
      }
      __syncwarp();
      for (int32_t t = 0;; ++t) {
        ptx::bar_sync(kBarTileA, kBarTileAThreads);  // P_A(t) keys 0-63; V(t), K(t+1) landed; bar->next
        const bool more = *reinterpret_cast<volatile int32_t*>(&bar->next[t & 1]) != 0;
        tc::fence_after_sync();
        if (tc::elect_one()) issue_pv(0, t, 0, 4);
        __syncwarp();
        ptx::bar_sync(kBarTileA2, kBarHalfThreads);  // P_A(t) keys 64-127
        tc::fence_after_sync();
        if (tc::elect_one()) {
          // While tiles follow, the next S_X commit also covers this PV_X (a
          // commit tracks every earlier MMA of this thread); only the last PV
          // needs its own signal, for the epilogue.
          issue_pv(0, t, 4, 8);
          if (more)
            issue_s(0, t + 1);
          else
            tc::commit(&bar->o_done[0]);
        }
        __syncwarp();
        if (has_b) {
          ptx::bar_sync(kBarTileB, kBarTileBThreads);  // P_B(t) keys 0-63
          tc::fence_after_sync();
          if (tc::elect_one()) issue_pv(1, t, 0, 4);
          __syncwarp();
          ptx::bar_sync(kBarTileB2, kBarHalfThreads);  // P_B(t) keys 64-127
          tc::fence_after_sync();
          if (tc::elect_one()) {
            issue_pv(1, t, 4, 8);
            if (more)
              issue_s(1, t + 1);
            else
              tc::commit(&bar->o_done[1]);
          }
          __syncwarp();
        }
        if (!more) break;
      }
    }
    // all MMAs issued by this warp have completed before TMEM is released (the
    // warp is converged at every elect, so the elected lane is always the same)
    if (tc::elect_one()) tc::commit(&bar->drain);
    __syncwarp();
    if (!ptx::mbar_wait(&bar->drain, 0) && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
    }
  }
  } else {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
  if (warp < 4 || has_b) {
    // --------------------------------------------------- softmax + epilogue
    const int x = warp >> 2;           // query tile
    const int wq = warp & 3;           // TMEM lane quarter
    const int32_t row = x * kMT + wq * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t s_addr = lane_addr + col_s(x), o_addr = lane_addr + col_o(x);
    const bool row_valid = row < n_rows;
    const bool release_kv = wq == 0 && x == (has_b ? 1 : 0);
    const int32_t my_vis = row_valid ? visible_keys(q_len, kv_len, (r0 + row) / G, a.causal) : 0;
    // every row of this query tile sees the keys below vis_first (uniform over the tile)
    const int32_t vis_first = visible_keys(q_len, kv_len, (r0 + x * kMT) / G, a.causal);
    const float c = a.scale * kLog2e;  // scores -> base-2 exponent
    float m_used = -INFINITY;          // raw-score max the exponentials are taken against
    float l = 0.f;
    int32_t t = 0;
    bool ok = true;
    for (int32_t bi = 0; bi < blk_cnt; ++bi) {
      int32_t lo, n;
      bool bad;
      const int32_t phys = walk.block(bi, &lo, &n, &bad);
      if (phys < 0) continue;
      for (int32_t off = 0; off < n; off += kN, ++t) {
        const int32_t pos0 = lo + off;
        const int32_t nvalid = min(kN, n - off);
        // waits and TMEM accesses stay warp-uniform (tcgen05.ld/st are warp-collective)
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bar->s_full[x], t & 1));
        if (!ok) {
          // a wait ran out: no more TMEM work, but every hand-off still takes
          // place (bar.sync keeps this warp in step with the MMA warp)
          ptx::bar_sync(x ? kBarTileB : kBarTileA, x ? kBarTileBThreads : kBarTileAThreads);
          ptx::bar_sync(x ? kBarTileB2 : kBarTileA2, kBarHalfThreads);
          continue;
        }
        if (release_kv && lane == 0) ptx::mbar_arrive(&bar->kv_free[t % kStages]);  // release t
        tc::fence_after_sync();
        uint32_t sr[4][32];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tc::tmem_ld32(s_addr + 32 * q4, sr[q4]);
        tc::tmem_ld_wait();
        // visible keys of this row inside the tile: [0, lim)
        const int32_t lim = min(nvalid, my_vis - pos0);
        const bool whole = pos0 + kN <= vis_first && nvalid == kN;  // uniform: no masking needed
        if (!whole) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * q4 + i >= lim) sr[q4][i] = __float_as_uint(-INFINITY);
        }
        // row max: eight independent 3-input max chains, then a small tree
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int i = 0; i < 32; i += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mx8[k] = max3(mx8[k], __uint_as_float(sr[q4][i + 2 * k]), __uint_as_float(sr[q4][i + 2 * k + 1]));
        const float mx = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        bool need = false;
        float alpha = 1.f;
        if (mx != -INFINITY) {
          if (m_used == -INFINITY) {
            m_used = mx;  // nothing accumulated yet: O and l are zero
          } else if ((mx - m_used) * c > kRescaleThreshold) {
            need = true;
            alpha = fast_exp2((m_used - mx) * c);
            m_used = mx;
            l *= alpha;
          }
        }
        if (__any_sync(0xffffffffu, need)) {
          // O holds P_{t-1} V_{t-1}: S_t completed, and PV_{t-1} was issued
          // before it, so it completed too; PV_t waits for P_t.
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t orr[32];
            tc::tmem_ld32(o_addr + 32 * q4, orr);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tc::tmem_st32(o_addr + 32 * q4, orr);
          }
          tc::tmem_st_wait();
        }
        const float mc = (m_used == -INFINITY) ? 0.f : m_used * c;
        // p = 2^(s*c - m*c) in pairs (packed FMA), row sum in four packed partial sums
        const float2 c2 = make_float2(c, c), nmc2 = make_float2(-mc, -mc);
        float2 sum4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) sum4[k] = make_float2(0.f, 0.f);
        // P in two halves (keys 0-63 over S columns 0-31, keys 64-127 over 32-63, all
        // already in registers), each handed to the MMA warp once written, so the
        // first half's PV runs while the second half is computed.  P_t overwrites
        // P_{t-1}, which PV_{t-1} read: done, as it was issued before S_t, which
        // has completed.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pw[32];
#pragma unroll
          for (int qq = 0; qq < 2; ++qq)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int q4 = 2 * h + qq;
              const float2 xx = ptx::ffma2(make_float2(__uint_as_float(sr[q4][2 * i]), __uint_as_float(sr[q4][2 * i + 1])),
                                           c2, nmc2);
              const float2 pp = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
              sum4[i & 3] = add2(sum4[i & 3], pp);
              pw[16 * qq + i] = pack_bf16(pp.x, pp.y);
            }
          tc::tmem_st32(s_addr + 32 * h, pw);
          tc::tmem_st_wait();
          tc::fence_before_sync();
          __syncwarp();
          if (h == 0)
            ptx::bar_arrive(x ? kBarTileB : kBarTileA, x ? kBarTileBThreads : kBarTileAThreads);
          else
            ptx::bar_arrive(x ? kBarTileB2 : kBarTileA2, kBarHalfThreads);
        }
        const float2 s4 = add2(add2(sum4[0], sum4[1]), add2(sum4[2], sum4[3]));
        l += s4.x + s4.y;
      }
    }
    // epilogue: O / l and the log-sum-exp of this row; o_done_x is committed
    // once, after the last PV_x
    if (ok && t > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait(&bar->o_done[x], 0))) ok = false;
    if (!ok && lane == 0) atomicOr(a.status, ptx::kStatusTimeout);
    tc::fence_after_sync();
    const int64_t orow = static_cast<int64_t>(part_row + (r0 + row) / G) * a.Hq + kvh * G + (r0 + row) % G;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    // Q_x's tile is free once o_done_x is seen (every MMA that reads it has
    // completed): each warp passes 32 rows x 32 columns at a time through its 4 KB
    // of it (16-byte slot y of row k at y ^ (k & 7): no bank conflicts either way)
    // and stores whole 128-byte row pieces, four rows per instruction.  A unit with
    // no key tile (t == 0) never waits for its Q copy, so it writes its zero rows
    // directly, as does a unit whose waits ran out.
    if (ok && t > 0) {
      float4* wst = reinterpret_cast<float4*>(sq + x * kTileBytes + wq * 4096);
      int64_t orow_k[8];
      bool valid_k[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int32_t rk = x * kMT + wq * 32 + 4 * i + (lane >> 3);
        valid_k[i] = rk < n_rows;
        orow_k[i] = static_cast<int64_t>(part_row + (r0 + rk) / G) * a.Hq + kvh * G + (r0 + rk) % G;
      }
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t orr[32];
        if (t > 0) {
          tc::tmem_ld32(o_addr + 32 * q4, orr);
          tc::tmem_ld_wait();
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (t > 0 && l > 0.f)
            v = make_float4(__uint_as_float(orr[4 * i]) * inv, __uint_as_float(orr[4 * i + 1]) * inv,
                            __uint_as_float(orr[4 * i + 2]) * inv, __uint_as_float(orr[4 * i + 3]) * inv);
          wst[lane * 8 + (i ^ (lane & 7))] = v;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int kr = 4 * i + (lane >> 3), y = lane & 7;
          if (valid_k[i])
            reinterpret_cast<float4*>(a.o_part + orow_k[i] * kD + 32 * q4)[y] = wst[kr * 8 + (y ^ (kr & 7))];
        }
        __syncwarp();
      }
    } else {
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t orr[32];
        if (t > 0) {
          tc::tmem_ld32(o_addr + 32 * q4, orr);
          tc::tmem_ld_wait();
        }
        if (row_valid) {
          float4* dst = reinterpret_cast<float4*>(a.o_part + orow * kD + 32 * q4);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t > 0 && l > 0.f)
              v = make_float4(__uint_as_float(orr[4 * i]) * inv, __uint_as_float(orr[4 * i + 1]) * inv,
                              __uint_as_float(orr[4 * i + 2]) * inv, __uint_as_float(orr[4 * i + 3]) * inv);
            dst[i] = v;
          }
        }
      }
    }
    if (row_valid) a.lse_part[orow] = l > 0.f ? (m_used * c + __log2f(l)) * kLn2 : -INFINITY;

    if (a.fused) {
      // ---- in-launch merge: the last CTA of each (sequence, K/V head, 256-row
      // unit) merges the unit's rows over the sequence's items.  The softmax
      // warps wrote this CTA's partial rows; each publishes them (fence), then
      // one thread takes a ticket from the unit's counter (the usual
      // fence-then-count pattern).  No CTA waits for another.
      const int merge_threads = has_b ? 2 * kMT : kMT;
      __threadfence();
      ptx::bar_sync(kBarMerge, merge_threads);
      // the unit's coordinates again, from the launch index (nothing kept live across the main loop)
      const int64_t um = blockIdx.x;
      const int32_t m_utile = static_cast<int32_t>(um % units_per_item);
      const int32_t m_kvh = static_cast<int32_t>((um / units_per_item) % a.Hkv);
      const WorkView mv(a.work, a.B, a.n_items);  // rebuilt from the arguments: nothing kept live across the loop
      const int32_t* m_it = mv.item(static_cast<int32_t>(um / (static_cast<int64_t>(units_per_item) * a.Hkv)));
      const int32_t m_seq = __ldg(m_it + kItSeq);
      const int32_t m_cu = __ldg(m_it + kItCuQ);
      const int32_t m_r0 = m_utile * kM;
      const int32_t m_rows = min(kM, __ldg(m_it + kItQLen) * G - m_r0);
      const int32_t p0 = __ldg(mv.seq(m_seq) + kSqItemPtr), p1 = __ldg(mv.seq(m_seq + 1) + kSqItemPtr);
      uint32_t* ticket = a.tickets + (static_cast<int64_t>(m_seq) * a.Hkv + m_kvh) * units_per_item + m_utile;
      if (threadIdx.x == 0) {
        const uint32_t taken = atomicAdd(ticket, 1u);
        const bool last = taken == static_cast<uint32_t>(p1 - p0 - 1);
        if (last) *ticket = 0u;  // every item's CTA has counted: ready for the next launch
        __threadfence();
        bar->last = last ? 1 : 0;
      }
      ptx::bar_sync(kBarMerge, merge_threads);
      if (*reinterpret_cast<volatile int32_t*>(&bar->last) != 0) {
        // one warp per (token, head) row of the unit, the partials read through L2
        for (int32_t r = warp; r < m_rows; r += merge_threads / 32) {
          const int32_t rr = m_r0 + r, tok = rr / G, h = m_kvh * G + rr % G;
          merge_row<__nv_bfloat16, kD, true>(a.o_part, a.lse_part, mv, p0, p1, tok, h, a.Hq,
                                             static_cast<int64_t>(m_cu + tok) * a.Hq + h,
                                             static_cast<__nv_bfloat16*>(a.out), a.lse_out);
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

}  // namespace

bool tc_supports(const PartialArgs& a) {
  if (a.dtype != SPLITKV_BF16 || a.d != kD || a.Hkv <= 0 || a.Hq % a.Hkv != 0) return false;
  const int32_t G = a.Hq / a.Hkv;
  return G >= 1 && G <= kMT && kMT % G == 0 && a.block_len % kN == 0 &&
         static_cast<int64_t>(a.n_pool_blocks) * a.block_len < (1ll << 31);
}

int tc_blocks_per_sm(const PartialArgs& a, int* blocks, int32_t* units_per_item) {
  *units_per_item = (a.max_q_len * (a.Hq / a.Hkv) + kM - 1) / kM * a.Hkv;
  cudaError_t e = cudaFuncSetAttribute(partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, partial_tc_kernel, kThreads, kSmemBytes);
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "tc occupancy: %s", cudaGetErrorString(e));
  return SPLITKV_OK;
}

int launch_partial_tc(const PartialArgs& a, cudaStream_t stream) {
  const int32_t G = a.Hq / a.Hkv;
  const int32_t units = (a.max_q_len * G + kM - 1) / kM;
  const int64_t grid = static_cast<int64_t>(units) * a.Hkv * a.n_items;
  if (grid == 0) return SPLITKV_OK;
  if (grid > 0x7fffffffLL) return fail(SPLITKV_ERR_UNSUPPORTED, "too many work units");
  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {kD, static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(a.total_q)};
    const uint64_t strides[2] = {kD * 2ull, static_cast<uint64_t>(a.Hq) * kD * 2ull};
    const uint32_t box[3] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(kMT / G)};
    const int st = encode_bf16_3d(&tq, a.q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != SPLITKV_OK) return st;
  }
  {
    const uint64_t dims[3] = {kD, static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(a.n_pool_blocks) * a.block_len};
    const uint64_t strides[2] = {kD * 2ull, static_cast<uint64_t>(a.Hkv) * kD * 2ull};
    const uint32_t box[3] = {64, 1, kN};
    int st = encode_bf16_3d(&tk, a.k_pool, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != SPLITKV_OK) return st;
    st = encode_bf16_3d(&tv, a.v_pool, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != SPLITKV_OK) return st;
  }
  cudaError_t e = cudaFuncSetAttribute(partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "tc smem attribute: %s", cudaGetErrorString(e));
  partial_tc_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(a, units, tq, tk, tv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "tc launch: %s", cudaGetErrorString(e));
  return SPLITKV_OK;
}

}  // namespace splitkv

// Host side of the split-KV path: block costing, LPT allocation, work lists.
//
// Follows the Split-KV knowledge card (kongchang.com), "Timeline" and "All
// Facts": context KV blocks go to the CP shards by a cost-aware
// longest-processing-time-first rule.  The card leaves the cost and the tie
// order open; this file takes cost = visible (query, key) pairs of a block,
// ties by lower global block index and then lower shard id.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "splitkv.h"
#include "status.h"
#include "work_layout.h"

using splitkv::fail;

namespace {

// Visible (query, key) pairs of keys [lo, hi) for q_len queries whose token t
// sees keys [0, a0 + t) (causal tail) - the sum over t of clamp(a0+t-lo, 0, hi-lo),
// in closed form: the terms are 0, then rise by one per query, then saturate.
int64_t causal_pairs(int64_t q_len, int64_t a0, int64_t lo, int64_t hi) {
  const int64_t w = hi - lo;
  const int64_t a = a0 - lo;  // term of query 0 before clamping
  auto clampi = [](int64_t x, int64_t l, int64_t h) { return x < l ? l : (x > h ? h : x); };
  const int64_t t_rise = clampi(-a + 1, 0, q_len);  // queries whose term is <= 0
  const int64_t t_sat = clampi(w - a, 0, q_len);    // first query whose term is >= w
  int64_t total = (q_len - t_sat) * w;
  if (t_sat > t_rise) {
    const int64_t n = t_sat - t_rise;
    total += n * a + (t_sat * (t_sat - 1) - t_rise * (t_rise - 1)) / 2;
  }
  return total;
}

bool check_lengths(const int32_t* q_len, const int32_t* kv_len, int32_t B, int32_t block_len,
                   int* status) {
  if (!q_len || !kv_len) { *status = fail(SPLITKV_ERR_INVALID, "null length array"); return false; }
  if (B <= 0) { *status = fail(SPLITKV_ERR_INVALID, "B must be positive (got %d)", B); return false; }
  if (block_len <= 0) {
    *status = fail(SPLITKV_ERR_INVALID, "block_len must be positive (got %d)", block_len);
    return false;
  }
  for (int32_t b = 0; b < B; ++b) {
    if (q_len[b] < 0 || kv_len[b] < 0 || q_len[b] > kv_len[b]) {
      *status = fail(SPLITKV_ERR_INVALID,
                     "sequence %d: need 0 <= q_len (%d) <= kv_len (%d)", b, q_len[b], kv_len[b]);
      return false;
    }
  }
  return true;
}

}  // namespace

extern "C" int64_t splitkv_num_blocks(const int32_t* kv_len, int32_t B, int32_t block_len) {
  if (!kv_len || B <= 0 || block_len <= 0)
    return fail(SPLITKV_ERR_INVALID, "splitkv_num_blocks: bad arguments");
  int64_t n = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (kv_len[b] < 0) return fail(SPLITKV_ERR_INVALID, "negative kv_len");
    n += (static_cast<int64_t>(kv_len[b]) + block_len - 1) / block_len;
  }
  splitkv::clear_error();
  return n;
}

extern "C" int splitkv_block_costs(const int32_t* q_len, const int32_t* kv_len, int32_t B,
                                   int32_t block_len, int32_t causal, int64_t* block_cost,
                                   int64_t n_blocks) {
  int st = 0;
  if (!check_lengths(q_len, kv_len, B, block_len, &st)) return st;
  if (!block_cost) return fail(SPLITKV_ERR_INVALID, "null block_cost");
  int64_t g = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t lq = q_len[b], lk = kv_len[b];
    const int64_t nb = (lk + block_len - 1) / block_len;
    if (g + nb > n_blocks)
      return fail(SPLITKV_ERR_CAPACITY, "block_cost holds %lld blocks, batch has more",
                  (long long)n_blocks);
    for (int64_t j = 0; j < nb; ++j) {
      const int64_t lo = j * block_len;
      const int64_t hi = std::min<int64_t>(lk, lo + block_len);
      block_cost[g++] = causal ? causal_pairs(lq, lk - lq + 1, lo, hi) : lq * (hi - lo);
    }
  }
  if (g != n_blocks)
    return fail(SPLITKV_ERR_INVALID, "n_blocks = %lld but the batch has %lld blocks",
                (long long)n_blocks, (long long)g);
  splitkv::clear_error();
  return SPLITKV_OK;
}

namespace {

// Indices 0..n-1 by (signed 64-bit) key descending, equal keys in ascending index
// order: a least-significant-digit radix sort (8-bit digits) of the complemented keys.  Each pass is
// stable, so indices of equal keys keep the ascending order they start in; digits
// that are the same in every key are skipped (costs usually span a few bytes).
// O(n) per pass, against O(n log n) comparisons of a comparison sort.
template <typename Index, typename KeyOf>
void order_desc_stable(int64_t n, KeyOf key_of, std::vector<Index>& order) {
  // per-thread buffers kept across calls: a planner run each step reuses their pages
  thread_local std::vector<uint64_t> key, key2;
  thread_local std::vector<Index> order2;
  order.resize(static_cast<size_t>(n));
  key.resize(static_cast<size_t>(n));
  uint64_t any = 0, all = ~uint64_t{0};
  bool sorted = true;
  for (int64_t i = 0; i < n; ++i) {
    // sign bit flipped: unsigned order = signed order; complemented: descending
    key[i] = ~(static_cast<uint64_t>(static_cast<int64_t>(key_of(i))) ^ (uint64_t{1} << 63));
    any |= key[i];
    all &= key[i];
    order[i] = static_cast<Index>(i);
    if (i > 0 && key[i] < key[i - 1]) sorted = false;
  }
  if (sorted) return;  // already non-increasing: the index order is the answer
  order2.resize(static_cast<size_t>(n));
  key2.resize(static_cast<size_t>(n));
  for (int shift = 0; shift < 64; shift += 8) {
    if ((((any ^ all) >> shift) & 0xffu) == 0) continue;  // this digit is equal in every key
    int64_t start[257] = {0};
    for (int64_t i = 0; i < n; ++i) ++start[((key[i] >> shift) & 0xffu) + 1];
    for (int d = 0; d < 256; ++d) start[d + 1] += start[d];
    for (int64_t i = 0; i < n; ++i) {
      const int64_t at = start[(key[i] >> shift) & 0xffu]++;
      order2[at] = order[i];
      key2[at] = key[i];
    }
    order.swap(order2);
    key.swap(key2);
  }
}

// Longest first; equal costs keep ascending block index.
void lpt_order(const int64_t* block_cost, int64_t n_blocks, std::vector<int64_t>& order) {
  order_desc_stable<int64_t>(n_blocks, [&](int64_t g) { return block_cost[g]; }, order);
}

// Each block in `order` goes to the least-loaded shard, the smallest
// (load, id) pair: a binary min-heap on that pair.  Shards 0..n-1 with zero
// load already form a valid heap (a parent's index, hence id, is lower).  When
// the total cost leaves room, the pair is packed as load * 2^bits + id into one
// unsigned key, which orders exactly like the pair.
template <typename Key, typename Less, typename Add, typename IdOf>
void sift_assign(const std::vector<int64_t>& order, const int64_t* block_cost, int32_t n, std::vector<Key>& heap,
                 Less less, Add add, IdOf id_of, int32_t* shard_of_block) {
  for (int64_t g : order) {
    shard_of_block[g] = id_of(heap[0]);
    const Key top = add(heap[0], block_cost[g]);
    int32_t i = 0;
    for (;;) {
      const int32_t l = 2 * i + 1, r = l + 1;
      if (l >= n) break;
      const int32_t m = (r < n && less(heap[r], heap[l])) ? r : l;
      if (!less(heap[m], top)) break;
      heap[i] = heap[m];
      i = m;
    }
    heap[i] = top;
  }
}

void lpt_assign_sorted(const std::vector<int64_t>& order, const int64_t* block_cost, int32_t n_shards,
                       int32_t* shard_of_block, int64_t* shard_load) {
  int bits = 1;
  while ((int64_t{1} << bits) < n_shards) ++bits;
  uint64_t total = 0;
  for (int64_t g : order) total += static_cast<uint64_t>(block_cost[g]);
  if (total < (uint64_t{1} << (63 - bits))) {
    const uint64_t mask = (uint64_t{1} << bits) - 1;
    std::vector<uint64_t> heap(static_cast<size_t>(n_shards));
    for (int32_t k = 0; k < n_shards; ++k) heap[k] = static_cast<uint64_t>(k);
    sift_assign(
        order, block_cost, n_shards, heap, [](uint64_t x, uint64_t y) { return x < y; },
        [bits](uint64_t x, int64_t c) { return x + (static_cast<uint64_t>(c) << bits); },
        [mask](uint64_t x) { return static_cast<int32_t>(x & mask); }, shard_of_block);
    for (int32_t k = 0; k < n_shards; ++k) shard_load[heap[k] & mask] = static_cast<int64_t>(heap[k] >> bits);
    return;
  }
  using Slot = std::pair<int64_t, int32_t>;
  std::vector<Slot> heap(static_cast<size_t>(n_shards));
  for (int32_t k = 0; k < n_shards; ++k) heap[k] = {0, k};
  sift_assign(
      order, block_cost, n_shards, heap, [](const Slot& x, const Slot& y) { return x < y; },
      [](const Slot& x, int64_t c) { return Slot{x.first + c, x.second}; },
      [](const Slot& x) { return x.second; }, shard_of_block);
  for (int32_t k = 0; k < n_shards; ++k) shard_load[heap[k].second] = heap[k].first;
}

}  // namespace

extern "C" int splitkv_plan(const int64_t* block_cost, int64_t n_blocks, int32_t n_shards,
                            int32_t* shard_of_block, int64_t* shard_load) {
  if (n_blocks < 0 || (n_blocks > 0 && (!block_cost || !shard_of_block)))
    return fail(SPLITKV_ERR_INVALID, "splitkv_plan: bad block arrays");
  if (n_shards <= 0 || !shard_load)
    return fail(SPLITKV_ERR_INVALID, "splitkv_plan: n_shards must be positive (got %d)", n_shards);
  for (int64_t g = 0; g < n_blocks; ++g)
    if (block_cost[g] < 0) return fail(SPLITKV_ERR_INVALID, "negative cost at block %lld", (long long)g);

  thread_local std::vector<int64_t> order;  // kept across calls (see order_desc_stable)
  lpt_order(block_cost, n_blocks, order);
  lpt_assign_sorted(order, block_cost, n_shards, shard_of_block, shard_load);
  splitkv::clear_error();
  return SPLITKV_OK;
}

extern "C" int splitkv_imbalance(const int64_t* shard_load, int32_t n_shards, double* rate) {
  if (!shard_load || !rate || n_shards <= 0)
    return fail(SPLITKV_ERR_INVALID, "splitkv_imbalance: need the loads of n_shards > 0 shards");
  int64_t total = 0, mx = 0;
  for (int32_t s = 0; s < n_shards; ++s) {
    if (shard_load[s] < 0) return fail(SPLITKV_ERR_INVALID, "negative load on shard %d", s);
    if (shard_load[s] > (int64_t(1) << 53) - 1 - total)
      return fail(SPLITKV_ERR_INVALID, "splitkv_imbalance: loads sum past 2^53");
    total += shard_load[s];
    mx = std::max(mx, shard_load[s]);
  }
  // max / mean - 1 with mean = total / n; total < 2^53, so both conversions are exact
  const double mean = static_cast<double>(total) / static_cast<double>(n_shards);
  *rate = total == 0 ? 0.0 : static_cast<double>(mx) / mean - 1.0;
  splitkv::clear_error();
  return SPLITKV_OK;
}

extern "C" int64_t splitkv_work_words(int64_t n_blocks, int32_t B) {
  if (n_blocks < 0 || B <= 0) return fail(SPLITKV_ERR_INVALID, "splitkv_work_words: bad arguments");
  return splitkv::kHeaderWords + splitkv::kSeqWords * (static_cast<int64_t>(B) + 1) +
         (splitkv::kItemWords + 2) * n_blocks;
}

namespace {

// How a plan's (shard, sequence) runs of blocks become work items.
//   max_item_blocks > 0: every run is cut into items of at most that many blocks.
//   tail: with units_per_item CTAs launched per item and `slots` CTAs resident at
//   once, the items whose CTAs fall in the last, partly filled wave (launch order)
//   are each cut into up to `pieces` runs of consecutive blocks.
struct ItemCut {
  int32_t max_item_blocks = 0;
  int32_t units_per_item = 0, slots = 0, pieces = 0;
};

// Work lists of a plan, with items cut as `cut` says (default: one item per pair).
int build_work(const int32_t* q_len, const int32_t* kv_len, int32_t B, int32_t block_len,
               const int64_t* block_cost, const int32_t* shard_of_block, int64_t n_blocks, int32_t n_shards,
               const ItemCut& cut, int32_t* work, int64_t work_words, int32_t* n_items_out,
               int64_t* part_rows_out) {
  const int32_t max_item_blocks = cut.max_item_blocks;
  using namespace splitkv;
  int st = 0;
  if (!check_lengths(q_len, kv_len, B, block_len, &st)) return st;
  if (!work || !n_items_out || !part_rows_out || (n_blocks > 0 && (!block_cost || !shard_of_block)))
    return fail(SPLITKV_ERR_INVALID, "splitkv_build_work: null argument");
  if (n_shards <= 0) return fail(SPLITKV_ERR_INVALID, "n_shards must be positive");
  if (max_item_blocks < 0) return fail(SPLITKV_ERR_INVALID, "max_item_blocks must be >= 0");
  if (cut.units_per_item < 0 || cut.slots < 0 || cut.pieces < 0)
    return fail(SPLITKV_ERR_INVALID, "units_per_item, slots and pieces must be >= 0");
  const int64_t need = splitkv_work_words(n_blocks, B);
  if (need < 0) return static_cast<int>(need);
  if (work_words < need)
    return fail(SPLITKV_ERR_CAPACITY, "work buffer holds %lld words, needs %lld",
                (long long)work_words, (long long)need);

  // Global block g -> (sequence, logical block).
  // per-thread buffers kept across calls (a planner run each step reuses their pages)
  thread_local std::vector<int32_t> seq_of, blk_of;
  seq_of.resize(static_cast<size_t>(n_blocks));
  blk_of.resize(static_cast<size_t>(n_blocks));
  int64_t g = 0;
  int64_t total_q = 0;
  int32_t max_q = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t nb = (static_cast<int64_t>(kv_len[b]) + block_len - 1) / block_len;
    if (g + nb > n_blocks) return fail(SPLITKV_ERR_INVALID, "n_blocks is smaller than the batch");
    for (int64_t j = 0; j < nb; ++j, ++g) {
      seq_of[g] = b;
      blk_of[g] = static_cast<int32_t>(j);
    }
    total_q += q_len[b];
    max_q = std::max(max_q, q_len[b]);
  }
  if (g != n_blocks) return fail(SPLITKV_ERR_INVALID, "n_blocks does not match kv_len/block_len");
  if (total_q > INT32_MAX) return fail(SPLITKV_ERR_UNSUPPORTED, "total_q exceeds int32");
  for (int64_t i = 0; i < n_blocks; ++i)
    if (shard_of_block[i] < 0 || shard_of_block[i] >= n_shards)
      return fail(SPLITKV_ERR_INVALID, "shard_of_block[%lld] = %d out of range", (long long)i,
                  shard_of_block[i]);

  // Group blocks by (shard, sequence); within a group blocks stay ascending.  A
  // counting sort on shard * B + sequence when there are not many more groups
  // than blocks, else a stable comparison sort: the same order either way.
  thread_local std::vector<int64_t> idx;
  idx.resize(static_cast<size_t>(n_blocks));
  const int64_t groups = static_cast<int64_t>(n_shards) * B;
  if (groups <= 4 * n_blocks + 4096) {
    thread_local std::vector<int64_t> start;
    start.assign(static_cast<size_t>(groups) + 1, 0);
    for (int64_t i = 0; i < n_blocks; ++i) ++start[static_cast<int64_t>(shard_of_block[i]) * B + seq_of[i] + 1];
    for (int64_t k = 0; k < groups; ++k) start[k + 1] += start[k];
    for (int64_t i = 0; i < n_blocks; ++i) idx[start[static_cast<int64_t>(shard_of_block[i]) * B + seq_of[i]]++] = i;
  } else {
    for (int64_t i = 0; i < n_blocks; ++i) idx[i] = i;
    std::stable_sort(idx.begin(), idx.end(), [&](int64_t x, int64_t y) {
      if (shard_of_block[x] != shard_of_block[y]) return shard_of_block[x] < shard_of_block[y];
      return seq_of[x] < seq_of[y];
    });
  }
  struct Item {
    int32_t shard, seq;
    int64_t first, count, cost;
  };
  thread_local std::vector<Item> items;
  items.clear();
  for (int64_t i = 0; i < n_blocks;) {
    int64_t j = i;
    Item it{shard_of_block[idx[i]], seq_of[idx[i]], i, 0, 0};
    while (j < n_blocks && shard_of_block[idx[j]] == it.shard && seq_of[idx[j]] == it.seq &&
           (max_item_blocks == 0 || j - i < max_item_blocks)) {
      it.cost += block_cost[idx[j]];
      ++j;
    }
    it.count = j - i;
    items.push_back(it);
    i = j;
  }
  // Launch order: largest item first, then shard, then sequence.
  thread_local std::vector<int32_t> order;
  order_desc_stable<int32_t>(static_cast<int64_t>(items.size()), [&](int64_t i) { return items[i].cost; }, order);
  // Tail cut: the items of the last partial wave, in launch order, each become up
  // to `pieces` items of consecutive blocks, launched last (piece order kept).
  const int64_t units = static_cast<int64_t>(items.size()) * cut.units_per_item;
  if (cut.units_per_item > 0 && cut.slots > 0 && cut.pieces > 1 && units > cut.slots && units % cut.slots != 0) {
    const int64_t tail = (units % cut.slots + cut.units_per_item - 1) / cut.units_per_item;
    const int64_t n0 = static_cast<int64_t>(items.size());
    std::vector<int64_t> rank(static_cast<size_t>(n0));
    for (int64_t r = 0; r < n0; ++r) rank[order[r]] = r;
    std::vector<Item> cut_items;
    std::vector<int64_t> key;  // launch position: parent rank * pieces + piece
    for (int64_t i = 0; i < n0; ++i) {
      const Item& it = items[i];
      const int64_t p = rank[i] >= n0 - tail ? std::min<int64_t>(cut.pieces, it.count) : 1;
      int64_t first = it.first;
      for (int64_t k = 0; k < p; ++k) {
        const int64_t cnt = it.count / p + (k < it.count % p ? 1 : 0);
        Item piece{it.shard, it.seq, first, cnt, 0};
        for (int64_t j = first; j < first + cnt; ++j) piece.cost += block_cost[idx[j]];
        cut_items.push_back(piece);
        key.push_back(rank[i] * cut.pieces + k);
        first += cnt;
      }
    }
    items.swap(cut_items);
    order.resize(items.size());
    for (size_t i = 0; i < items.size(); ++i) order[i] = static_cast<int32_t>(i);
    std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return key[x] < key[y]; });
  }

  const int32_t n_items = static_cast<int32_t>(items.size());
  const int64_t off_seq = work_off_seq();
  const int64_t off_items = work_off_items(B);
  const int64_t off_blocks = work_off_blocks(B, n_items);
  const int64_t off_seq_items = off_blocks + n_blocks;
  std::memset(work, 0, sizeof(int32_t) * static_cast<size_t>(off_seq_items + n_items));

  int32_t* hdr = work;
  hdr[kMagic] = kWorkMagic;
  hdr[kB] = B;
  hdr[kNItems] = n_items;
  hdr[kNShards] = n_shards;
  hdr[kBlockLen] = block_len;
  hdr[kTotalQ] = static_cast<int32_t>(total_q);
  hdr[kMaxQ] = max_q;
  hdr[kOffSeq] = static_cast<int32_t>(off_seq);
  hdr[kOffItems] = static_cast<int32_t>(off_items);
  hdr[kOffBlocks] = static_cast<int32_t>(off_blocks);
  hdr[kOffSeqItems] = static_cast<int32_t>(off_seq_items);
  hdr[kNBlocks] = static_cast<int32_t>(n_blocks);
  if (off_seq_items + n_items > INT32_MAX) return fail(SPLITKV_ERR_UNSUPPORTED, "work descriptor too large");

  int64_t part_row = 0;
  int64_t blk_cursor = 0;
  std::vector<int32_t> cu_q(static_cast<size_t>(B), 0);
  for (int32_t b = 1; b < B; ++b) cu_q[b] = cu_q[b - 1] + q_len[b - 1];
  thread_local std::vector<int32_t> rank_of;
  rank_of.resize(items.size());
  for (int32_t r = 0; r < n_items; ++r) {
    const Item& it = items[order[r]];
    rank_of[order[r]] = r;
    int32_t* w = work + off_items + kItemWords * static_cast<int64_t>(r);
    w[kItShard] = it.shard;
    w[kItSeq] = it.seq;
    w[kItBlockOff] = static_cast<int32_t>(blk_cursor);
    w[kItBlockCnt] = static_cast<int32_t>(it.count);
    if (part_row > INT32_MAX) return fail(SPLITKV_ERR_UNSUPPORTED, "partial rows exceed int32");
    w[kItPartRow] = static_cast<int32_t>(part_row);
    w[kItQLen] = q_len[it.seq];
    w[kItKvLen] = kv_len[it.seq];
    w[kItCuQ] = cu_q[it.seq];
    w[kItCostLo] = static_cast<int32_t>(static_cast<uint64_t>(it.cost) & 0xffffffffu);
    w[kItCostHi] = static_cast<int32_t>(static_cast<uint64_t>(it.cost) >> 32);
    for (int64_t k = 0; k < it.count; ++k) work[off_blocks + blk_cursor + k] = blk_of[idx[it.first + k]];
    blk_cursor += it.count;
    part_row += q_len[it.seq];
  }
  // Per sequence: its items, ascending shard (items were built shard-major).
  std::vector<int32_t> per_seq_count(B, 0);
  for (const Item& it : items) per_seq_count[it.seq]++;
  int32_t ptr = 0;
  int64_t cu = 0;
  for (int32_t b = 0; b < B; ++b) {
    int32_t* s = work + off_seq + kSeqWords * b;
    s[0] = static_cast<int32_t>(cu);
    s[1] = q_len[b];
    s[2] = kv_len[b];
    s[3] = ptr;
    ptr += per_seq_count[b];
    cu += q_len[b];
  }
  int32_t* last = work + off_seq + kSeqWords * B;
  last[0] = static_cast<int32_t>(total_q);
  last[3] = n_items;
  std::vector<int32_t> fill(B, 0);
  for (size_t i = 0; i < items.size(); ++i) {
    const int32_t b = items[i].seq;
    const int32_t base = work[off_seq + kSeqWords * b + 3];
    work[off_seq_items + base + fill[b]++] = rank_of[i];
  }
  *n_items_out = n_items;
  *part_rows_out = part_row;
  splitkv::clear_error();
  return SPLITKV_OK;
}

}  // namespace

extern "C" int splitkv_build_work(const int32_t* q_len, const int32_t* kv_len, int32_t B,
                                  int32_t block_len, const int64_t* block_cost,
                                  const int32_t* shard_of_block, int64_t n_blocks,
                                  int32_t n_shards, int32_t* work, int64_t work_words,
                                  int32_t* n_items_out, int64_t* part_rows_out) {
  return build_work(q_len, kv_len, B, block_len, block_cost, shard_of_block, n_blocks, n_shards, ItemCut{}, work,
                    work_words, n_items_out, part_rows_out);
}

extern "C" int splitkv_build_work_split(const int32_t* q_len, const int32_t* kv_len, int32_t B,
                                        int32_t block_len, const int64_t* block_cost,
                                        const int32_t* shard_of_block, int64_t n_blocks, int32_t n_shards,
                                        int32_t max_item_blocks, int32_t* work, int64_t work_words,
                                        int32_t* n_items_out, int64_t* part_rows_out) {
  ItemCut cut;
  cut.max_item_blocks = max_item_blocks;
  return build_work(q_len, kv_len, B, block_len, block_cost, shard_of_block, n_blocks, n_shards, cut, work,
                    work_words, n_items_out, part_rows_out);
}

extern "C" int splitkv_build_work_tail(const int32_t* q_len, const int32_t* kv_len, int32_t B,
                                       int32_t block_len, const int64_t* block_cost,
                                       const int32_t* shard_of_block, int64_t n_blocks, int32_t n_shards,
                                       int32_t units_per_item, int32_t slots, int32_t pieces, int32_t* work,
                                       int64_t work_words, int32_t* n_items_out, int64_t* part_rows_out) {
  ItemCut cut;
  cut.units_per_item = units_per_item;
  cut.slots = slots;
  cut.pieces = pieces;
  return build_work(q_len, kv_len, B, block_len, block_cost, shard_of_block, n_blocks, n_shards, cut, work,
                    work_words, n_items_out, part_rows_out);
}

extern "C" int splitkv_plan_dcp(const int32_t* q_len, const int32_t* kv_len, int32_t B, int32_t block_len,
                                int32_t causal, int32_t max_shards, double alpha, double beta, double gamma,
                                int32_t* shard_of_block, int64_t n_blocks, int64_t* shard_load,
                                int32_t* n_shards_used, double* modeled_time) {
  // Split selection that models attention completion together with the reduction
  // that depends on it (LiquidCP abstract: MegaDCP).  For every shard count s the
  // blocks are planned with the same LPT rule; the shards run concurrently, so
  // attention completes with the slowest one - compute (alpha per unit of block
  // cost) plus K/V streaming (gamma per token) - and the reduction combines one
  // partial row per (shard, sequence) pair and query token:
  //     T(s) = max_k (alpha * load_k + gamma * tokens_k) + beta * partial_rows(s)
  // (each product rounded on its own: this file is compiled without FP
  // contraction).  The smallest s reaching the least T wins.
  int st = 0;
  if (!check_lengths(q_len, kv_len, B, block_len, &st)) return st;
  if (max_shards <= 0 || !shard_of_block || !shard_load || !n_shards_used || !modeled_time)
    return fail(SPLITKV_ERR_INVALID, "splitkv_plan_dcp: bad arguments");
  std::vector<int64_t> costs(static_cast<size_t>(n_blocks));
  st = splitkv_block_costs(q_len, kv_len, B, block_len, causal, costs.data(), n_blocks);
  if (st != SPLITKV_OK) return st;
  std::vector<int32_t> seq_of(static_cast<size_t>(n_blocks));
  std::vector<int64_t> tokens(static_cast<size_t>(n_blocks));
  {
    int64_t g = 0;
    for (int32_t b = 0; b < B; ++b)
      for (int64_t j = 0; j < (static_cast<int64_t>(kv_len[b]) + block_len - 1) / block_len; ++j) {
        seq_of[g] = b;
        tokens[g++] = std::min<int64_t>(block_len, kv_len[b] - j * block_len);
      }
  }
  std::vector<int32_t> sob(static_cast<size_t>(n_blocks)), best_sob;
  std::vector<int64_t> load(static_cast<size_t>(max_shards)), best_load;
  std::vector<uint8_t> held(static_cast<size_t>(max_shards));
  std::vector<int64_t> shard_tok(static_cast<size_t>(max_shards));
  int32_t best_s = 0;
  double best_t = 0.0;
  std::vector<int64_t> order;
  lpt_order(costs.data(), n_blocks, order);  // the LPT order does not depend on s

  // Shard counts are tried from the largest down, so the first smaller s whose
  // lower bound exceeds the best T found ends the search: every shard count
  // below it has a larger bound.  The bound holds for non-negative
  // coefficients: the slowest shard is at least the mean (alpha*C + gamma*N)/s
  // over all cost C and tokens N, and each sequence with keys adds at least one
  // partial row per query token.  The relative margin covers the rounding of
  // both sides, so the chosen s is the one the exhaustive search picks.
  const bool prune = alpha >= 0.0 && beta >= 0.0 && gamma >= 0.0;
  int64_t cost_sum = 0, tok_sum = 0, rows_min = 0;
  for (int64_t g = 0; g < n_blocks; ++g) {
    cost_sum += costs[g];
    tok_sum += tokens[g];
  }
  for (int32_t b = 0; b < B; ++b)
    if (kv_len[b] > 0) rows_min += q_len[b];
  const double att_sum = alpha * static_cast<double>(cost_sum) + gamma * static_cast<double>(tok_sum);
  for (int32_t s = max_shards; s >= 1; --s) {
    if (prune && best_s != 0 && best_t > 0.0 &&
        att_sum / s + beta * static_cast<double>(rows_min) > best_t * (1.0 + 1e-9))
      break;
    lpt_assign_sorted(order, costs.data(), s, sob.data(), load.data());
    std::fill(shard_tok.begin(), shard_tok.begin() + s, 0);
    for (int64_t g = 0; g < n_blocks; ++g) shard_tok[sob[g]] += tokens[g];
    double t_att = 0.0;
    for (int32_t k = 0; k < s; ++k) {
      const double tk = alpha * static_cast<double>(load[k]) + gamma * static_cast<double>(shard_tok[k]);
      if (k == 0 || tk > t_att) t_att = tk;
    }
    // partial rows: blocks are sequence-major, so one pass with a per-sequence shard mask
    int64_t rows = 0;
    for (int64_t g = 0; g < n_blocks;) {
      const int32_t b = seq_of[g];
      std::fill(held.begin(), held.begin() + s, 0);
      int32_t distinct = 0;
      for (; g < n_blocks && seq_of[g] == b; ++g)
        if (!held[sob[g]]) {
          held[sob[g]] = 1;
          ++distinct;
        }
      rows += static_cast<int64_t>(distinct) * q_len[b];
    }
    const double t = t_att + beta * static_cast<double>(rows);
    if (best_s == 0 || t <= best_t) {  // s is decreasing: a tie goes to the smaller s
      best_s = s;
      best_t = t;
      best_sob = sob;
      best_load.assign(load.begin(), load.begin() + s);
    }
  }
  std::copy(best_sob.begin(), best_sob.end(), shard_of_block);
  for (int32_t k = 0; k < max_shards; ++k) shard_load[k] = k < best_s ? best_load[k] : 0;
  *n_shards_used = best_s;
  *modeled_time = best_t;
  splitkv::clear_error();
  return SPLITKV_OK;
}

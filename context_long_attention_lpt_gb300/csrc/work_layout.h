// Word layout of the int32 work descriptor (documented in include/splitkv.h,
// splitkv_build_work).  Shared by the host builder and the device kernels.
#pragma once

#include <cstdint>

namespace splitkv {

constexpr int32_t kWorkMagic = 0x534B5632;  // "SKV2"

// header words
constexpr int kMagic = 0, kB = 1, kNItems = 2, kNShards = 3, kBlockLen = 4, kTotalQ = 5, kMaxQ = 6,
              kOffSeq = 7, kOffItems = 8, kOffBlocks = 9, kOffSeqItems = 10, kNBlocks = 11;
constexpr int64_t kHeaderWords = 16;

// per-sequence row: {cu_q, q_len, kv_len, seq_item_ptr}
constexpr int64_t kSeqWords = 4;
constexpr int kSqCuQ = 0, kSqQLen = 1, kSqKvLen = 2, kSqItemPtr = 3;

// per-item row: the item's own words, then a copy of its sequence's lengths so that a
// kernel starting on an item needs one row of the descriptor, not two
constexpr int64_t kItemWords = 12;
constexpr int kItShard = 0, kItSeq = 1, kItBlockOff = 2, kItBlockCnt = 3, kItPartRow = 4, kItQLen = 5,
              kItKvLen = 6, kItCuQ = 7, kItCostLo = 8, kItCostHi = 9;

// The sections sit at fixed offsets given by B and n_items (the header repeats them), so
// a kernel finds an item's row from its launch arguments without reading the header first.
constexpr int64_t work_off_seq() { return kHeaderWords; }
constexpr int64_t work_off_items(int64_t B) { return kHeaderWords + kSeqWords * (B + 1); }
constexpr int64_t work_off_blocks(int64_t B, int64_t n_items) { return work_off_items(B) + kItemWords * n_items; }

}  // namespace splitkv

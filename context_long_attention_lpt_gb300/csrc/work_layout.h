// Word layout of the int32 work descriptor (documented in include/splitkv.h,
// splitkv_build_work).  Shared by the host builder and the device kernels.
#pragma once

#include <cstdint>

namespace splitkv {

constexpr int32_t kWorkMagic = 0x534B5631;  // "SKV1"

// header words
constexpr int kMagic = 0, kB = 1, kNItems = 2, kNShards = 3, kBlockLen = 4, kTotalQ = 5, kMaxQ = 6,
              kOffSeq = 7, kOffItems = 8, kOffBlocks = 9, kOffSeqItems = 10, kNBlocks = 11;
constexpr int64_t kHeaderWords = 16;

// per-sequence row: {cu_q, q_len, kv_len, seq_item_ptr}
constexpr int64_t kSeqWords = 4;
constexpr int kSqCuQ = 0, kSqQLen = 1, kSqKvLen = 2, kSqItemPtr = 3;

// per-item row
constexpr int64_t kItemWords = 8;
constexpr int kItShard = 0, kItSeq = 1, kItBlockOff = 2, kItBlockCnt = 3, kItPartRow = 4,
              kItCostLo = 5, kItCostHi = 6;

}  // namespace splitkv

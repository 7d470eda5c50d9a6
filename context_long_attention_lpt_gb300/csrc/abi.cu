// extern "C" device-side entry points: argument validation, kernel choice, launch.

#include <algorithm>
#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "launch.h"
#include "splitkv.h"
#include "status.h"

using splitkv::fail;

namespace {

// Bit 0: a block-table entry outside the pool was skipped.
__device__ unsigned int g_device_status = 0;

unsigned int* status_word(int* err) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_device_status);
  if (e != cudaSuccess) {
    *err = fail(SPLITKV_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
    return nullptr;
  }
  return static_cast<unsigned int*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Decode kernel for a handful of query rows per K/V head, tensor cores once the
// rows fill MMA tiles, the generic CUDA-core kernel for everything else.
int pick_kernel(const splitkv::PartialArgs& a, int32_t requested) {
  if (requested != SPLITKV_KERNEL_AUTO) return requested;
  if (splitkv::decode_supports(a)) return SPLITKV_KERNEL_DECODE;
  if (splitkv::tc_supports(a)) return SPLITKV_KERNEL_TC;
  return SPLITKV_KERNEL_SIMT;
}

}  // namespace

extern "C" int splitkv_auto_kernel(int32_t Hq, int32_t Hkv, int32_t d, int32_t block_len,
                                   int32_t max_q_len, int32_t dtype) {
  splitkv::PartialArgs a{};
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.block_len = block_len;
  a.max_q_len = max_q_len;
  a.dtype = dtype;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return fail(SPLITKV_ERR_INVALID, "bad head counts");
  return pick_kernel(a, SPLITKV_KERNEL_AUTO);
}

extern "C" int splitkv_partial_slots(int32_t Hq, int32_t Hkv, int32_t d, int32_t block_len, int32_t max_q_len,
                                     int32_t dtype, int32_t kernel, int32_t* units_per_item) {
  splitkv::PartialArgs a{};
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.block_len = block_len;
  a.max_q_len = max_q_len;
  a.dtype = dtype;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_q_len <= 0) return fail(SPLITKV_ERR_INVALID, "bad shape");
  if (!units_per_item) return fail(SPLITKV_ERR_INVALID, "splitkv_partial_slots: null argument");
  const int k = pick_kernel(a, kernel);
  int blocks = 0, st = SPLITKV_OK;
  if (k == SPLITKV_KERNEL_DECODE && splitkv::decode_supports(a)) {
    *units_per_item = Hkv;
    st = splitkv::decode_blocks_per_sm(a, &blocks);
  } else if (k == SPLITKV_KERNEL_TC && splitkv::tc_supports(a)) {
    st = splitkv::tc_blocks_per_sm(a, &blocks, units_per_item);
  } else {
    return fail(SPLITKV_ERR_UNSUPPORTED, "splitkv_partial_slots: only the decode and tensor-core kernels");
  }
  if (st != SPLITKV_OK) return st;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  splitkv::clear_error();
  return blocks * sms;
}

extern "C" int splitkv_backward_kernel(int32_t Hq, int32_t Hkv, int32_t d, int32_t block_len, int32_t dtype) {
  splitkv::PartialArgs a{};
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.block_len = block_len;
  a.dtype = dtype;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return fail(SPLITKV_ERR_INVALID, "bad head counts");
  return splitkv::bwd_tc_supports(a) ? SPLITKV_KERNEL_TC : SPLITKV_KERNEL_SIMT;
}

extern "C" int splitkv_plan_batch(const int32_t* q_len, const int32_t* kv_len, int32_t B, int32_t block_len,
                                  int32_t causal, int32_t n_shards, int32_t units_per_item, int32_t slots,
                                  int32_t pieces, int64_t* block_cost, int32_t* shard_of_block, int64_t n_blocks,
                                  int64_t* shard_load, int32_t* work_host, int32_t* work_dev, int64_t work_words, int32_t* n_items, int64_t* part_rows, void* stream) {
  int st = splitkv_block_costs(q_len, kv_len, B, block_len, causal, block_cost, n_blocks);
  if (st != SPLITKV_OK) return st;
  st = splitkv_plan(block_cost, n_blocks, n_shards, shard_of_block, shard_load);
  if (st != SPLITKV_OK) return st;
  st = splitkv_build_work_tail(q_len, kv_len, B, block_len, block_cost, shard_of_block, n_blocks, n_shards,
                               units_per_item, slots, pieces, work_host, work_words, n_items, part_rows);
  if (st != SPLITKV_OK) return st;
  if (work_dev) {
    const cudaError_t e = cudaMemcpyAsync(work_dev, work_host, static_cast<size_t>(work_words) * sizeof(int32_t),
                                          cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "work descriptor upload: %s", cudaGetErrorString(e));
  }
  splitkv::clear_error();
  return SPLITKV_OK;
}

namespace {

// Validates the arguments shared by the partial-attention entry points and fills `a`.
int make_partial_args(splitkv::PartialArgs* a, const void* q, const void* k_pool, const void* v_pool,
                      int64_t n_pool_blocks, const int32_t* block_table, int32_t max_blocks_per_seq,
                      const int32_t* work, int32_t n_items, int32_t B, int32_t total_q, int32_t max_q_len,
                      int32_t Hq, int32_t Hkv, int32_t d, int32_t block_len, float scale, int32_t causal,
                      int32_t dtype, float* o_part, float* lse_part, int64_t part_rows, int32_t kernel) {
  if (dtype != SPLITKV_F32 && dtype != SPLITKV_BF16)
    return fail(SPLITKV_ERR_INVALID, "dtype must be SPLITKV_F32 or SPLITKV_BF16 (got %d)", dtype);
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return fail(SPLITKV_ERR_INVALID, "need B > 0 and Hq a positive multiple of Hkv (B=%d Hq=%d Hkv=%d)",
                B, Hq, Hkv);
  if (d != 64 && d != 128) return fail(SPLITKV_ERR_UNSUPPORTED, "head dim %d not supported (64, 128)", d);
  if (block_len <= 0 || n_pool_blocks < 0 || max_blocks_per_seq < 0 || n_items < 0 || total_q < 0 ||
      max_q_len < 0 || part_rows < 0)
    return fail(SPLITKV_ERR_INVALID, "negative size argument");
  if (!std::isfinite(scale)) return fail(SPLITKV_ERR_INVALID, "scale must be finite");
  if (n_items > 0 && (!q || !k_pool || !v_pool || !block_table || !work || !o_part || !lse_part))
    return fail(SPLITKV_ERR_INVALID, "null device pointer");
  if (!work) return fail(SPLITKV_ERR_INVALID, "null work descriptor");
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o_part))
    return fail(SPLITKV_ERR_INVALID, "q, k_pool, v_pool and o_part must be 16-byte aligned");
  if (kernel < SPLITKV_KERNEL_AUTO || kernel > SPLITKV_KERNEL_TC)
    return fail(SPLITKV_ERR_INVALID, "unknown kernel %d", kernel);
  int err = 0;
  *a = splitkv::PartialArgs{q, k_pool, v_pool, n_pool_blocks, block_table, max_blocks_per_seq, work,
                            n_items, B, total_q, max_q_len, Hq, Hkv, d, block_len, scale, causal ? 1 : 0,
                            dtype, o_part, lse_part, part_rows, nullptr, 0, nullptr, nullptr, nullptr};
  a->status = status_word(&err);
  if (!a->status) return err;
  return SPLITKV_OK;
}

int launch_partial(const splitkv::PartialArgs& a, int k, cudaStream_t s) {
  int st = SPLITKV_OK;
  switch (k) {
    case SPLITKV_KERNEL_TC:
      if (!splitkv::tc_supports(a))
        return fail(SPLITKV_ERR_UNSUPPORTED, "tensor-core kernel needs bf16, d=128, block_len %% 128 == 0, "
                    "G dividing 128");
      st = splitkv::launch_partial_tc(a, s);
      break;
    case SPLITKV_KERNEL_DECODE:
      if (!splitkv::decode_supports(a))
        return fail(SPLITKV_ERR_UNSUPPORTED, "decode kernel needs bf16, d=128, q_len*G <= 8, block_len %% 64 == 0");
      st = splitkv::launch_partial_decode(a, s);
      break;
    default: {
      const cudaError_t e = splitkv::launch_partial_simt(a, s);
      if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "partial launch: %s", cudaGetErrorString(e));
      break;
    }
  }
  return st;
}

int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" int splitkv_attn_partial(const void* q, const void* k_pool, const void* v_pool,
                                    int64_t n_pool_blocks, const int32_t* block_table,
                                    int32_t max_blocks_per_seq, const int32_t* work,
                                    int32_t n_items, int32_t B, int32_t total_q,
                                    int32_t max_q_len, int32_t Hq, int32_t Hkv, int32_t d,
                                    int32_t block_len, float scale, int32_t causal,
                                    int32_t dtype, float* o_part, float* lse_part,
                                    int64_t part_rows, int32_t kernel, void* stream) {
  splitkv::PartialArgs a;
  int st = make_partial_args(&a, q, k_pool, v_pool, n_pool_blocks, block_table, max_blocks_per_seq, work, n_items, B,
                             total_q, max_q_len, Hq, Hkv, d, block_len, scale, causal, dtype, o_part, lse_part,
                             part_rows, kernel);
  if (st != SPLITKV_OK) return st;
  if (n_items == 0) {
    splitkv::clear_error();
    return SPLITKV_OK;
  }
  st = launch_partial(a, pick_kernel(a, kernel), static_cast<cudaStream_t>(stream));
  if (st != SPLITKV_OK) return st;
  splitkv::clear_error();
  return SPLITKV_OK;
}

extern "C" int splitkv_fused_launches(int32_t Hq, int32_t Hkv, int32_t d, int32_t block_len, int32_t max_q_len,
                                      int32_t n_items, int32_t dtype, int32_t kernel) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return fail(SPLITKV_ERR_INVALID, "bad head counts");
  splitkv::PartialArgs a{};
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.block_len = block_len;
  a.max_q_len = max_q_len;
  a.n_items = n_items;
  a.dtype = dtype;
  const int k = pick_kernel(a, kernel);
  splitkv::clear_error();
  return ((k == SPLITKV_KERNEL_DECODE && splitkv::decode_fuses(a)) || k == SPLITKV_KERNEL_TC) ? 1 : 2;
}

extern "C" int64_t splitkv_ticket_count(int32_t B, int32_t Hq, int32_t Hkv, int32_t max_q_len) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_q_len < 0)
    return fail(SPLITKV_ERR_INVALID, "splitkv_ticket_count: bad arguments");
  splitkv::clear_error();
  return static_cast<int64_t>(B) * Hkv * std::max<int64_t>(1, div_up(static_cast<int64_t>(max_q_len) * (Hq / Hkv), 256));
}

extern "C" int splitkv_attn_fused(const void* q, const void* k_pool, const void* v_pool, int64_t n_pool_blocks,
                                  const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* work,
                                  int32_t n_items, int32_t B, int32_t total_q, int32_t max_q_len, int32_t Hq,
                                  int32_t Hkv, int32_t d, int32_t block_len, float scale, int32_t causal,
                                  int32_t dtype, float* o_part, float* lse_part, int64_t part_rows,
                                  uint32_t* tickets, int64_t n_tickets, void* out, float* lse_out, int32_t kernel,
                                  void* stream) {
  splitkv::PartialArgs a;
  int st = make_partial_args(&a, q, k_pool, v_pool, n_pool_blocks, block_table, max_blocks_per_seq, work, n_items, B,
                             total_q, max_q_len, Hq, Hkv, d, block_len, scale, causal, dtype, o_part, lse_part,
                             part_rows, kernel);
  if (st != SPLITKV_OK) return st;
  if (total_q > 0 && (!out || !lse_out)) return fail(SPLITKV_ERR_INVALID, "null output pointer");
  const int64_t need = splitkv_ticket_count(B, Hq, Hkv, max_q_len);
  if (need < 0) return static_cast<int>(need);
  if (!tickets || n_tickets < need)
    return fail(SPLITKV_ERR_CAPACITY, "tickets holds %lld counters, needs %lld", (long long)n_tickets, (long long)need);
  if (n_items == 0) {
    splitkv::clear_error();
    return SPLITKV_OK;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int k = pick_kernel(a, kernel);
  if ((k == SPLITKV_KERNEL_DECODE && splitkv::decode_fuses(a)) || k == SPLITKV_KERNEL_TC) {
    a.fused = 1;
    a.tickets = tickets;
    a.out = out;
    a.lse_out = lse_out;
    st = launch_partial(a, k, s);
  } else {
    // kernels without an in-kernel merge: the same two launches as the separate calls
    st = launch_partial(a, k, s);
    if (st == SPLITKV_OK) {
      const cudaError_t e = splitkv::launch_merge(o_part, lse_part, part_rows, work, B, total_q, Hq, d, dtype, out,
                                                  lse_out, a.status, s);
      if (e != cudaSuccess) st = fail(SPLITKV_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
    }
  }
  if (st != SPLITKV_OK) return st;
  splitkv::clear_error();
  return SPLITKV_OK;
}

extern "C" int splitkv_merge(const float* o_part, const float* lse_part, int64_t part_rows,
                             const int32_t* work, int32_t B, int32_t total_q, int32_t Hq, int32_t d,
                             int32_t dtype, void* out, float* lse_out, void* stream) {
  if (dtype != SPLITKV_F32 && dtype != SPLITKV_BF16)
    return fail(SPLITKV_ERR_INVALID, "dtype must be SPLITKV_F32 or SPLITKV_BF16 (got %d)", dtype);
  if (d != 64 && d != 128) return fail(SPLITKV_ERR_UNSUPPORTED, "head dim %d not supported (64, 128)", d);
  if (B <= 0 || Hq <= 0 || total_q < 0) return fail(SPLITKV_ERR_INVALID, "bad sizes");
  if (total_q > 0 && (!o_part || !lse_part || !work || !out || !lse_out))
    return fail(SPLITKV_ERR_INVALID, "null device pointer");
  if (!aligned16(o_part)) return fail(SPLITKV_ERR_INVALID, "o_part must be 16-byte aligned");
  if (part_rows < 0) return fail(SPLITKV_ERR_INVALID, "negative part_rows");
  int err = 0;
  unsigned int* status = status_word(&err);
  if (!status) return err;
  const cudaError_t e = splitkv::launch_merge(o_part, lse_part, part_rows, work, B, total_q, Hq, d,
                                              dtype, out, lse_out, status,
                                              static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
  splitkv::clear_error();
  return SPLITKV_OK;
}

extern "C" int splitkv_device_status(uint32_t* status, int32_t clear) {
  if (!status) return fail(SPLITKV_ERR_INVALID, "null status pointer");
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
  }
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "device status: %s", cudaGetErrorString(e));
  *status = v;
  splitkv::clear_error();
  return SPLITKV_OK;
}

extern "C" int splitkv_bwd_delta(const void* o, const void* dout, int32_t total_q, int32_t Hq, int32_t d,
                                 int32_t dtype, float* delta, void* stream) {
  if (dtype != SPLITKV_F32 && dtype != SPLITKV_BF16) return fail(SPLITKV_ERR_INVALID, "bad dtype");
  if (total_q < 0 || Hq <= 0 || (d != 64 && d != 128)) return fail(SPLITKV_ERR_INVALID, "bad sizes");
  if (total_q > 0 && (!o || !dout || !delta)) return fail(SPLITKV_ERR_INVALID, "null device pointer");
  const cudaError_t e = splitkv::launch_bwd_delta(o, dout, static_cast<int64_t>(total_q) * Hq, d, dtype, delta,
                                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "delta launch: %s", cudaGetErrorString(e));
  splitkv::clear_error();
  return SPLITKV_OK;
}

extern "C" int splitkv_attn_backward(const void* q, const void* k_pool, const void* v_pool, int64_t n_pool_blocks,
                                     const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* work,
                                     int32_t n_items, int32_t B, int32_t total_q, int32_t max_q_len, int32_t Hq,
                                     int32_t Hkv, int32_t d, int32_t block_len, float scale, int32_t causal,
                                     int32_t dtype, const void* dout, const float* lse, const float* delta,
                                     float* dq_part, int64_t part_rows, float* dk_pool, float* dv_pool,
                                     void* stream) {
  splitkv::PartialArgs a;
  int st = make_partial_args(&a, q, k_pool, v_pool, n_pool_blocks, block_table, max_blocks_per_seq, work, n_items, B,
                             total_q, max_q_len, Hq, Hkv, d, block_len, scale, causal, dtype, dq_part,
                             /* lse_part: unused */ dq_part, part_rows, SPLITKV_KERNEL_SIMT);
  if (st != SPLITKV_OK) return st;
  if (n_items > 0 && (!dout || !lse || !delta || !dk_pool || !dv_pool))
    return fail(SPLITKV_ERR_INVALID, "null device pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n_items > 0 && splitkv::bwd_tc_supports(a)) {
    // tensor cores: every partial dQ row and every key's dK / dV written once
    st = splitkv::launch_bwd_tc(a, dout, lse, delta, dq_part, dk_pool, dv_pool, s);
    if (st != SPLITKV_OK) return st;
    splitkv::clear_error();
    return SPLITKV_OK;
  }
  // CUDA cores: the partial dQ rows collect atomic adds from every key tile of their item
  cudaError_t e = cudaMemsetAsync(dq_part, 0, static_cast<size_t>(part_rows) * Hq * d * sizeof(float), s);
  if (e == cudaSuccess && n_items > 0) e = splitkv::launch_bwd_partial(a, dout, lse, delta, dq_part, dk_pool, dv_pool, s);
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
  splitkv::clear_error();
  return SPLITKV_OK;
}

extern "C" int splitkv_dq_reduce(const float* dq_part, int64_t part_rows, const int32_t* work, int32_t B,
                                 int32_t total_q, int32_t Hq, int32_t d, float* dq, void* stream) {
  if (B <= 0 || Hq <= 0 || total_q < 0 || part_rows < 0 || (d != 64 && d != 128))
    return fail(SPLITKV_ERR_INVALID, "bad sizes");
  if (total_q > 0 && (!dq_part || !work || !dq)) return fail(SPLITKV_ERR_INVALID, "null device pointer");
  int err = 0;
  unsigned int* status = status_word(&err);
  if (!status) return err;
  const cudaError_t e = splitkv::launch_dq_reduce(dq_part, part_rows, work, B, total_q, Hq, d, dq, status,
                                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "dq reduce launch: %s", cudaGetErrorString(e));
  splitkv::clear_error();
  return SPLITKV_OK;
}

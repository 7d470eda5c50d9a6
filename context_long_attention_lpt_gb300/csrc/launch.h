// Internal launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "splitkv.h"

namespace splitkv {

// Arguments of one partial-attention launch, already validated by the ABI layer.
struct PartialArgs {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  int64_t n_pool_blocks;
  const int32_t* block_table;
  int32_t max_blocks_per_seq;
  const int32_t* work;
  int32_t n_items;
  int32_t B;
  int32_t total_q;
  int32_t max_q_len;
  int32_t Hq;
  int32_t Hkv;
  int32_t d;
  int32_t block_len;
  float scale;
  int32_t causal;
  int32_t dtype;
  float* o_part;
  float* lse_part;
  int64_t part_rows;
  unsigned int* status;  // device status word (bit 0: block-table entry out of range)
  // Fused merge (decode kernel): the last CTA of each (sequence, K/V head) group,
  // found by an atomic ticket, merges the group's partials into out / lse_out.
  int32_t fused;
  uint32_t* tickets;  // one counter per (sequence, K/V head), zero between launches
  void* out;
  float* lse_out;
};

// Each launcher returns cudaSuccess or the launch error.
cudaError_t launch_partial_simt(const PartialArgs& a, cudaStream_t stream);
// The specialised kernels return a SPLITKV_* status (they also encode TMA maps).
int launch_partial_decode(const PartialArgs& a, cudaStream_t stream);
int launch_partial_tc(const PartialArgs& a, cudaStream_t stream);

// CTAs of the specialised kernels one SM keeps resident (and, for the tensor-core
// kernel, CTAs launched per work item); SPLITKV_* status.
int decode_blocks_per_sm(const PartialArgs& a, int* blocks);
int tc_blocks_per_sm(const PartialArgs& a, int* blocks, int32_t* units_per_item);

// Shape limits of the specialised kernels (checked before launching them).
bool decode_supports(const PartialArgs& a);
bool decode_fuses(const PartialArgs& a);  // the decode kernel can merge in the same launch
bool tc_supports(const PartialArgs& a);

// Backward pass (backward.cu).
cudaError_t launch_bwd_delta(const void* o, const void* dout, int64_t n_rows, int32_t d, int32_t dtype, float* delta,
                             cudaStream_t stream);
// Tensor-core backward (bf16, d = 128, block_len % 128 == 0, G | 128).
bool bwd_tc_supports(const PartialArgs& a);
int launch_bwd_tc(const PartialArgs& a, const void* dout, const float* lse, const float* delta, float* dq_part,
                  float* dk_pool, float* dv_pool, cudaStream_t stream);
cudaError_t launch_bwd_partial(const PartialArgs& a, const void* dout, const float* lse, const float* delta,
                               float* dq_part, float* dk_pool, float* dv_pool, cudaStream_t stream);
cudaError_t launch_dq_reduce(const float* dq_part, int64_t part_rows, const int32_t* work, int32_t B, int32_t total_q,
                             int32_t Hq, int32_t d, float* dq, unsigned int* status, cudaStream_t stream);

cudaError_t launch_merge(const float* o_part, const float* lse_part, int64_t part_rows,
                         const int32_t* work, int32_t B, int32_t total_q, int32_t Hq, int32_t d,
                         int32_t dtype, void* out, float* lse_out, unsigned int* status,
                         cudaStream_t stream);

}  // namespace splitkv

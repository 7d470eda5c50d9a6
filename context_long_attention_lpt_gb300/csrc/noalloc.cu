// Split-KV attention in one call that allocates no memory.
//
// Some callers cannot call cudaMalloc: code running inside a host that owns
// all device memory (an inference server or framework plugin with a fixed
// arena, where a raw allocation bypasses its accounting), latency-critical
// loops that must not risk allocation stalls or out-of-memory failures midway,
// and embedders that only ever hand this library buffers they already own.
// This entry point serves them: the caller passes inputs and outputs, and the
// intermediate buffers of the path (the work descriptor and the per-item
// partials) live in one fixed-size array that the library itself declares in
// device memory.  The array is part of the library image, so every GPU that
// loads the library holds it until the process exits.

#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "launch.h"
#include "splitkv.h"
#include "status.h"
#include "work_layout.h"

namespace splitkv {
namespace {

constexpr int kMaxDevices = 64;

// Device address of the scratch, looked up once per device (in host code the
// array's name is only a host-side stand-in, not a device address).
unsigned char* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace

// The shared scratch: work descriptor, then partial outputs, then partial LSEs.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPLITKV_NOALLOC_SCRATCH_BYTES];

namespace {

int scratch_for_current_device(unsigned char** scratch) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(SPLITKV_ERR_UNSUPPORTED, "device index %d too large", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *scratch = g_scratch_ptr[dev];
  return SPLITKV_OK;
}

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

}  // namespace
}  // namespace splitkv

extern "C" int splitkv_attention_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                         int64_t n_pool_blocks, const int32_t* block_table,
                                         int32_t max_blocks_per_seq, const int32_t* work_host,
                                         int64_t work_words, int32_t n_items, int32_t B,
                                         int32_t total_q, int32_t max_q_len, int32_t Hq, int32_t Hkv,
                                         int32_t d, int32_t block_len, float scale, int32_t causal,
                                         int32_t dtype, int64_t part_rows, void* out, float* lse_out,
                                         void* stream) {
  using namespace splitkv;
  if (!work_host || work_words < 16 || work_host[0] != kWorkMagic)
    return fail(SPLITKV_ERR_INVALID, "work_host is not a work descriptor from splitkv_build_work");
  if (n_items < 0 || part_rows < 0 || Hq <= 0 || (d != 64 && d != 128))
    return fail(SPLITKV_ERR_INVALID, "bad sizes for splitkv_attention_noalloc");
  // The descriptor's used length, from its own offsets.
  const int64_t used_words = static_cast<int64_t>(work_host[kOffSeqItems]) + work_host[kNItems];
  if (used_words > work_words || work_host[kNItems] != n_items || work_host[kB] != B)
    return fail(SPLITKV_ERR_INVALID, "work descriptor does not match n_items / B / work_words");
  const int64_t work_bytes = align256(used_words * 4);
  const int64_t o_bytes = align256(part_rows * Hq * static_cast<int64_t>(d) * 4);
  const int64_t l_bytes = align256(part_rows * static_cast<int64_t>(Hq) * 4);
  const int64_t need = work_bytes + o_bytes + l_bytes;
  if (need > SPLITKV_NOALLOC_SCRATCH_BYTES)
    return fail(SPLITKV_ERR_CAPACITY,
                "splitkv_attention_noalloc needs %lld bytes of scratch, the fixed array holds %lld "
                "(use splitkv_attn_partial + splitkv_merge with caller buffers)",
                (long long)need, (long long)SPLITKV_NOALLOC_SCRATCH_BYTES);
  unsigned char* scratch = nullptr;
  int st = scratch_for_current_device(&scratch);
  if (st != SPLITKV_OK) return st;
  int32_t* work_dev = reinterpret_cast<int32_t*>(scratch);
  float* o_part = reinterpret_cast<float*>(scratch + work_bytes);
  float* lse_part = reinterpret_cast<float*>(scratch + work_bytes + o_bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Copying the plan in allocates nothing; the host buffer is read before this returns
  // when it is pageable, and must stay unchanged until the copy runs when it is pinned.
  cudaError_t e = cudaMemcpyAsync(work_dev, work_host, used_words * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "work upload: %s", cudaGetErrorString(e));
  st = splitkv_attn_partial(q, k_pool, v_pool, n_pool_blocks, block_table, max_blocks_per_seq, work_dev, n_items,
                            B, total_q, max_q_len, Hq, Hkv, d, block_len, scale, causal, dtype, o_part, lse_part,
                            part_rows, SPLITKV_KERNEL_AUTO, stream);
  if (st != SPLITKV_OK) return st;
  return splitkv_merge(o_part, lse_part, part_rows, work_dev, B, total_q, Hq, d, dtype, out, lse_out, stream);
}

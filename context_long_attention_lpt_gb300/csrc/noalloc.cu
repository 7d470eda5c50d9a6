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

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "splitkv.h"
#include "status.h"
#include "work_layout.h"

namespace splitkv {
namespace {

constexpr int kMaxDevices = 64;

// Device address of the scratch per device, with the id of the context it was
// looked up in (in host code the array's name is only a host-side stand-in, not
// a device address).  A device whose context was destroyed and created again
// (cudaDeviceReset) loads the module at a new address, so a changed context id
// triggers a new lookup.
struct ScratchAddr {
  unsigned char* ptr;
  unsigned long long ctx_id;
};
ScratchAddr g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void lookup_ctx_fns() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
}

// Id of the calling thread's current context, 0 if it cannot be told.
unsigned long long current_ctx_id() {
  std::call_once(g_ctx_once, lookup_ctx_fns);
  if (!g_ctx_current || !g_ctx_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

}  // namespace

// The shared scratch: work descriptor, then partial outputs, then partial LSEs.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPLITKV_NOALLOC_SCRATCH_BYTES];

namespace {

// Set-up: the array's device address for the current device, looked up with that
// device current on its first use (and again after its context changed).
int scratch_for_current_device(unsigned char** scratch) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(SPLITKV_ERR_UNSUPPORTED, "device index %d too large", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_ctx_id();
  ScratchAddr& c = g_scratch[dev];
  if (!c.ptr || id == 0 || c.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail(SPLITKV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    c.ptr = static_cast<unsigned char*>(p);
    c.ctx_id = current_ctx_id();  // the lookup made the device's context current if it was not yet
  }
  *scratch = c.ptr;
  return SPLITKV_OK;
}

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Checks the host work descriptor against the call's sizes and returns, in
// *rows_needed, the partial rows its items address (largest part_row + q_len).
int check_descriptor(const int32_t* w, int64_t words, int32_t n_items, int32_t B, int32_t total_q,
                     int32_t max_q_len, int64_t* rows_needed) {
  if (!w || words < kHeaderWords || w[kMagic] != kWorkMagic)
    return fail(SPLITKV_ERR_INVALID, "work_host is not a work descriptor from splitkv_build_work");
  if (w[kNItems] != n_items || w[kB] != B || w[kTotalQ] != total_q || w[kMaxQ] != max_q_len)
    return fail(SPLITKV_ERR_INVALID,
                "work descriptor does not match the call (n_items %d/%d, B %d/%d, total_q %d/%d, max_q_len %d/%d)",
                w[kNItems], n_items, w[kB], B, w[kTotalQ], total_q, w[kMaxQ], max_q_len);
  const int64_t off_seq = w[kOffSeq], off_items = w[kOffItems], off_blocks = w[kOffBlocks],
                off_seq_items = w[kOffSeqItems], n_blocks = w[kNBlocks];
  if (off_seq != work_off_seq() || off_items != work_off_items(B) || off_blocks != work_off_blocks(B, n_items))
    return fail(SPLITKV_ERR_INVALID, "work descriptor sections are not where its B and n_items place them");
  if (off_seq_items < 0 || n_blocks < 0 ||
      off_seq + (static_cast<int64_t>(B) + 1) * kSeqWords > words ||
      off_items + static_cast<int64_t>(n_items) * kItemWords > words || off_blocks + n_blocks > words ||
      off_seq_items + n_items > words)
    return fail(SPLITKV_ERR_INVALID, "work descriptor offsets fall outside work_words");
  int64_t need = 0;
  for (int32_t i = 0; i < n_items; ++i) {
    const int32_t* it = w + off_items + static_cast<int64_t>(i) * kItemWords;
    const int32_t seq = it[kItSeq], prow = it[kItPartRow];
    if (seq < 0 || seq >= B || prow < 0)
      return fail(SPLITKV_ERR_INVALID, "work item %d has sequence %d / partial row %d out of range", i, seq, prow);
    const int32_t lq = it[kItQLen];  // the kernels take the item row's copy of q_len
    if (lq < 0 || lq > max_q_len || lq != w[off_seq + static_cast<int64_t>(seq) * kSeqWords + kSqQLen])
      return fail(SPLITKV_ERR_INVALID, "work item %d has q_len %d (sequence %d)", i, lq, seq);
    need = std::max<int64_t>(need, static_cast<int64_t>(prow) + lq);
  }
  *rows_needed = need;
  return SPLITKV_OK;
}

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
  if (n_items < 0 || part_rows < 0 || B <= 0 || total_q < 0 || max_q_len < 0 || Hq <= 0 || (d != 64 && d != 128))
    return fail(SPLITKV_ERR_INVALID, "bad sizes for splitkv_attention_noalloc");
  int64_t rows_needed = 0;
  int st = check_descriptor(work_host, work_words, n_items, B, total_q, max_q_len, &rows_needed);
  if (st != SPLITKV_OK) return st;
  if (part_rows != rows_needed)
    return fail(SPLITKV_ERR_INVALID, "part_rows %lld does not match the work descriptor's %lld partial rows",
                (long long)part_rows, (long long)rows_needed);
  // Bound the row count before any product, so the byte counts below cannot overflow.
  const int64_t row_bytes = 4 * static_cast<int64_t>(Hq) * (d + 1);
  const int64_t used_words = static_cast<int64_t>(work_host[kOffSeqItems]) + n_items;
  if (part_rows > SPLITKV_NOALLOC_SCRATCH_BYTES / row_bytes || used_words > SPLITKV_NOALLOC_SCRATCH_BYTES / 4)
    return fail(SPLITKV_ERR_CAPACITY,
                "splitkv_attention_noalloc: %lld partial rows of %lld bytes exceed the fixed scratch array of %lld "
                "bytes (use splitkv_attn_partial + splitkv_merge with caller buffers)",
                (long long)part_rows, (long long)row_bytes, (long long)SPLITKV_NOALLOC_SCRATCH_BYTES);
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
  st = scratch_for_current_device(&scratch);
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

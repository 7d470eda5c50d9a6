/*
 * splitkv.h - C ABI of the split-KV attention library (libsplitkv.so).
 *
 * Exact split-KV attention for very short queries against very long contexts,
 * after the "Split-KV" knowledge card (kongchang.com):
 *   - intro / "Timeline": K/V shards stay local to their device and each layer's
 *     attention exchanges only tensors the size of the queries;
 *   - "Timeline" / "All Facts": context KV blocks are allocated to the shards by
 *     a cost-aware longest-processing-time-first (LPT) rule, load imbalance < 1%;
 *   - "All Facts": the result is exact, strictly equal to the unsharded one.
 * Here the shards are emulated as KV splits on one GPU.  The path is:
 *   splitkv_block_costs -> splitkv_plan -> splitkv_build_work   (host, C++)
 *   splitkv_attn_partial -> splitkv_merge                        (device, CUDA)
 *
 * Conventions shared by every call
 *   - Query tensor q: [total_q, Hq, d], sequences concatenated; sequence b owns
 *     rows cu_q[b] .. cu_q[b]+q_len[b]-1 (cu_q = prefix sum of q_len).
 *   - K/V pools: [n_pool_blocks, block_len, Hkv, d], row-major; a sequence's
 *     logical block j lives in physical block block_table[b*max_blocks_per_seq+j].
 *   - GQA: query head h reads K/V head h / (Hq/Hkv).
 *   - Query token t of sequence b sits at key position kv_len[b]-q_len[b]+t
 *     (queries appended after the context).  causal != 0: key j is visible iff
 *     j <= that position; causal == 0: all kv_len[b] keys are visible.
 *   - Scores are scale * q.k; LSE values are natural-log log-sum-exp of the
 *     visible scaled scores, -inf where nothing is visible.
 *   - dtype: SPLITKV_F32 (fp32 Q/K/V, fp32 arithmetic) or SPLITKV_BF16 (bf16
 *     Q/K/V, fp32 accumulation).
 *   - Ownership: the caller owns every buffer.  Host calls take host pointers;
 *     device calls take device pointers and a cudaStream_t passed as void*.
 *     No call allocates device memory.  Device calls are asynchronous on the
 *     stream and never synchronise.
 *   - Errors: every call returns 0 (SPLITKV_OK) or a negative status, never
 *     aborts; splitkv_last_error() gives a message for the calling thread.
 *     Arguments are validated on the host before any launch.
 */
#ifndef SPLITKV_H
#define SPLITKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPLITKV_OK 0
#define SPLITKV_ERR_INVALID (-1)     /* bad pointer, size or argument */
#define SPLITKV_ERR_UNSUPPORTED (-2) /* shape the chosen kernel cannot run */
#define SPLITKV_ERR_CUDA (-3)        /* a CUDA runtime / driver call failed */
#define SPLITKV_ERR_CAPACITY (-4)    /* an output buffer is too small */

#define SPLITKV_F32 0
#define SPLITKV_BF16 1

/* kernel choice for splitkv_attn_partial */
#define SPLITKV_KERNEL_AUTO 0   /* pick the fastest kernel that supports the shape */
#define SPLITKV_KERNEL_SIMT 1   /* generic CUDA-core kernel: any shape, fp32 or bf16 */
#define SPLITKV_KERNEL_DECODE 2 /* CUDA-core decode kernel: bf16, d=128, q_len*G <= 8, block_len%64==0 */
#define SPLITKV_KERNEL_TC 3     /* TMA + tcgen05/TMEM kernel: bf16, d=128, block_len%128==0 */

/* ---------------------------------------------------------------- host side */

/* Number of KV blocks of the batch: sum over b of ceil(kv_len[b] / block_len).
 * Returns the count (>= 0) or a negative status. */
int64_t splitkv_num_blocks(const int32_t* kv_len, int32_t B, int32_t block_len);

/* Step 1, block costing ("cost-aware" LPT, Split-KV card, "Timeline").
 * block_cost[g] (out, host, n_blocks entries) = number of (query, key) pairs of
 * global block g left visible by the mask.  Blocks are numbered sequence after
 * sequence, logical block order within a sequence.  A fully visible block costs
 * q_len * tokens; a block holding a causal tail counts the triangle.
 * q_len, kv_len: host [B].  n_blocks must equal splitkv_num_blocks(). */
int splitkv_block_costs(const int32_t* q_len, const int32_t* kv_len, int32_t B,
                        int32_t block_len, int32_t causal, int64_t* block_cost,
                        int64_t n_blocks);

/* Step 2, LPT allocation (Split-KV card, "Timeline" / "All Facts").
 * Blocks are taken by cost, largest first (equal costs: lower global index
 * first); each goes to the shard with the smallest load so far (equal loads:
 * lower shard id).  Out (host): shard_of_block[n_blocks] in [0, n_shards),
 * shard_load[n_shards] = summed cost per shard.  Integer only: bit-exact. */
int splitkv_plan(const int64_t* block_cost, int64_t n_blocks, int32_t n_shards,
                 int32_t* shard_of_block, int64_t* shard_load);

/* Load imbalance of a plan (Split-KV card, "Timeline" / "All Facts": the LPT
 * allocation keeps it below 1%).  The card gives no definition; the rate here is
 * max load / mean load - 1, with mean = (sum of the loads) / n_shards, in IEEE
 * double (0 when every load is 0).  In (host): shard_load[n_shards], each >= 0,
 * summing below 2^53 (so the sum converts to double exactly).  Out: *rate. */
int splitkv_imbalance(const int64_t* shard_load, int32_t n_shards, double* rate);

/* Step 2, alternative planner: split selection that models the completion of
 * attention together with the reduction that depends on it (after the LiquidCP
 * abstract, PaperTrail: its MegaDCP selects history-KV splits this way; the
 * abstract gives no formula, this is the plainest reading).  For every shard
 * count s in 1..max_shards the blocks are planned with splitkv_plan's LPT rule;
 * attention completes with the slowest shard - alpha per unit of its block cost
 * plus gamma per K/V token it streams - and the reduction combines one partial
 * row per (shard, sequence) pair and query token, so
 *     T(s) = max_k (alpha*load_k + gamma*tokens_k) + beta*partial_rows(s)
 * (IEEE double, each product rounded separately) where partial_rows(s) = sum
 * over distinct (shard, sequence) pairs of q_len.
 * The smallest s reaching the least T is chosen.  Out (host): shard_of_block
 * [n_blocks] (ids < *n_shards_used), shard_load[max_shards] (0 past the chosen
 * count), *n_shards_used, *modeled_time.  alpha: time per unit of block cost on
 * one shard; beta: time per partial row to merge (any consistent unit). */
int splitkv_plan_dcp(const int32_t* q_len, const int32_t* kv_len, int32_t B, int32_t block_len,
                     int32_t causal, int32_t max_shards, double alpha, double beta, double gamma,
                     int32_t* shard_of_block, int64_t n_blocks, int64_t* shard_load,
                     int32_t* n_shards_used, double* modeled_time);

/* Upper bound, in int32 words, of the work descriptor built below. */
int64_t splitkv_work_words(int64_t n_blocks, int32_t B);

/* Step 2b, work lists.  Groups the plan into work items, one per (shard,
 * sequence) pair that holds at least one block, and writes the int32 work
 * descriptor consumed by splitkv_attn_partial / splitkv_merge (host buffer of
 * work_words words; the caller copies it to the device).  Layout:
 *   [0..15]  header: magic 0x534B5632, B, n_items, n_shards, block_len,
 *            total_q, max_q_len, off_seq, off_items, off_blocks, off_seq_items,
 *            n_blocks, 0...
 *   off_seq = 16   (B+1) x 4: {cu_q[b], q_len[b], kv_len[b], seq_item_ptr[b]};
 *                  row B = {total_q, 0, 0, n_items}
 *   off_items = 16 + 4(B+1)
 *                  n_items x 12: {shard, seq, block_off, block_cnt, part_row,
 *                  q_len[seq], kv_len[seq], cu_q[seq], cost_lo, cost_hi, 0, 0};
 *                  items sorted by cost (largest first, then shard, then
 *                  sequence) - the launch order
 *   off_blocks = off_items + 12 n_items
 *                  n_blocks: logical block indices, grouped by item, ascending
 *   off_seq_items = off_blocks + n_blocks
 *                  n_items: item indices grouped by sequence, ascending shard
 * The kernels find the sequence rows, item rows and block lists at these fixed
 * offsets from their B and n_items arguments (a CTA's first read is its item
 * row, which repeats its sequence's lengths); a launch whose B or n_items
 * differ from the header's does no work and sets bit 3 of the status word.
 * Item i's partial output occupies rows part_row .. part_row+q_len[seq]-1 of
 * the partial buffers; *part_rows (out) is the total row count (sum over items
 * of q_len of its sequence) and *n_items (out) the number of items. */
int splitkv_build_work(const int32_t* q_len, const int32_t* kv_len, int32_t B,
                       int32_t block_len, const int64_t* block_cost,
                       const int32_t* shard_of_block, int64_t n_blocks, int32_t n_shards,
                       int32_t* work, int64_t work_words, int32_t* n_items,
                       int64_t* part_rows);

/* splitkv_build_work with every (shard, sequence) run of blocks cut into items
 * of at most max_item_blocks blocks (in the run's ascending block order; 0: no
 * cut, the same descriptor as splitkv_build_work).  The plan is unchanged:
 * each item still belongs to one shard, and the merge reduces the extra
 * partial rows exactly like those of other shards (Split-KV card, "All
 * Facts": any split of a sequence's keys merges to the unsharded result).
 * More, shorter items give the device more, shorter units of work: the last
 * partly filled wave of CTAs gets shorter.  Same buffers and statuses as
 * splitkv_build_work; splitkv_work_words bounds the size for any cut. */
int splitkv_build_work_split(const int32_t* q_len, const int32_t* kv_len, int32_t B,
                             int32_t block_len, const int64_t* block_cost,
                             const int32_t* shard_of_block, int64_t n_blocks, int32_t n_shards,
                             int32_t max_item_blocks, int32_t* work, int64_t work_words,
                             int32_t* n_items, int64_t* part_rows);

/* splitkv_build_work with the items of the last, partly filled wave of CTAs cut
 * into pieces.  Each item launches units_per_item CTAs, and `slots` CTAs run at
 * once (both from splitkv_partial_slots).  If the item count times
 * units_per_item is above `slots` and not a multiple of it, the last
 * ceil((units mod slots) / units_per_item) items in launch order are each cut
 * into min(pieces, blocks) items of consecutive blocks, launched last.  The
 * plan is unchanged (every piece belongs to its shard; the merge reduces the
 * extra partial rows exactly, Split-KV card, "All Facts"); the last wave's
 * work is spread over all resident CTAs instead of a few.  units_per_item,
 * slots or pieces of 0 (or pieces 1): no cut.  Same buffers and statuses as
 * splitkv_build_work. */
int splitkv_build_work_tail(const int32_t* q_len, const int32_t* kv_len, int32_t B,
                            int32_t block_len, const int64_t* block_cost,
                            const int32_t* shard_of_block, int64_t n_blocks, int32_t n_shards,
                            int32_t units_per_item, int32_t slots, int32_t pieces, int32_t* work,
                            int64_t work_words, int32_t* n_items, int64_t* part_rows);

/* Steps 1-2 and the descriptor upload of one batch in one call: block costs
 * (Split-KV card, "Timeline": cost-aware), the LPT plan and the work lists,
 * exactly as splitkv_block_costs -> splitkv_plan -> splitkv_build_work_tail
 * (units_per_item, slots, pieces as there; pieces <= 1: no cut, the descriptor
 * of splitkv_build_work), then an asynchronous copy of the descriptor's work_words words from work_host to
 * work_dev on `stream` (a cudaStream_t; NULL is the legacy default stream).
 * For callers that plan every step, where one call instead of three keeps the
 * host ahead of the device.
 *   block_cost [n_blocks], shard_of_block [n_blocks], shard_load [n_shards]:
 *     host outputs, as from the two planning calls; n_blocks must equal
 *     splitkv_num_blocks().
 *   work_host [work_words]: host output, the descriptor.  Page-locked memory
 *     makes the copy asynchronous; the caller keeps it unchanged until the copy
 *     has completed (e.g. an event recorded on `stream` after this call).
 *   work_dev [work_words]: device buffer, or NULL to skip the copy (then
 *     `stream` is unused and the call needs no CUDA device).
 *   *n_items, *part_rows (out): as from splitkv_build_work.
 * Statuses: those of the three calls (nothing is copied when one fails),
 * SPLITKV_ERR_CUDA when the copy cannot be queued. */
int splitkv_plan_batch(const int32_t* q_len, const int32_t* kv_len, int32_t B, int32_t block_len,
                       int32_t causal, int32_t n_shards, int32_t units_per_item, int32_t slots,
                       int32_t pieces, int64_t* block_cost, int32_t* shard_of_block,
                       int64_t n_blocks, int64_t* shard_load,
                       int32_t* work_host, int32_t* work_dev, int64_t work_words,
                       int32_t* n_items, int64_t* part_rows, void* stream);

/* CTAs the partial kernel for a shape keeps resident on the current device at
 * once (occupancy x SM count), returned, and *units_per_item (out) = CTAs it
 * launches per work item.  kernel: SPLITKV_KERNEL_* (AUTO picks as the
 * partial call does).  Decode and tensor-core kernels only; other kernels
 * give SPLITKV_ERR_UNSUPPORTED.  Needs a CUDA device; negative status on error. */
int splitkv_partial_slots(int32_t Hq, int32_t Hkv, int32_t d, int32_t block_len, int32_t max_q_len,
                          int32_t dtype, int32_t kernel, int32_t* units_per_item);

/* Which kernel SPLITKV_KERNEL_AUTO picks for a shape (a SPLITKV_KERNEL_* value). */
int splitkv_auto_kernel(int32_t Hq, int32_t Hkv, int32_t d, int32_t block_len,
                        int32_t max_q_len, int32_t dtype);

/* -------------------------------------------------------------- device side */

/* Step 3, per-shard partial attention (Split-KV card, intro / "Timeline": each
 * shard attends only over its local KV blocks and emits a query-sized partial).
 * For every work item (shard s, sequence b), every query token t of b and every
 * query head h:
 *     m = max_j s_j,  l = sum_j exp(s_j - m),
 *     o_part[part_row+t, h, :] = sum_j exp(s_j - m) v_j / l,
 *     lse_part[part_row+t, h]  = m + ln l          (-inf, o = 0 if none visible)
 * over the keys j of s's blocks of b that token t sees; s_j = scale * q.k_j.
 * In (device): q, k_pool, v_pool (dtype), block_table int32 [B, max_blocks_per_seq],
 * work (the descriptor above, copied to the device).  Out (device, fp32):
 * o_part [part_rows, Hq, d], lse_part [part_rows, Hq].  n_items, B, total_q,
 * max_q_len and part_rows must match the descriptor.  kernel: SPLITKV_KERNEL_*.
 * A block-table entry outside [0, n_pool_blocks) is not read: the block is
 * skipped and bit 0 of the device status word is set (splitkv_device_status). */
int splitkv_attn_partial(const void* q, const void* k_pool, const void* v_pool,
                         int64_t n_pool_blocks, const int32_t* block_table,
                         int32_t max_blocks_per_seq, const int32_t* work, int32_t n_items,
                         int32_t B, int32_t total_q, int32_t max_q_len, int32_t Hq,
                         int32_t Hkv, int32_t d, int32_t block_len, float scale,
                         int32_t causal, int32_t dtype, float* o_part, float* lse_part,
                         int64_t part_rows, int32_t kernel, void* stream);

/* Counters splitkv_attn_fused needs: B * Hkv * max(1, ceil(max_q_len*(Hq/Hkv)/256)). */
int64_t splitkv_ticket_count(int32_t B, int32_t Hq, int32_t Hkv, int32_t max_q_len);

/* Launches splitkv_attn_fused makes for a shape and kernel choice: 1 when the
 * chosen kernel merges inside its own launch (decode kernel with at most 2048
 * items, tensor-core kernel), 2 otherwise (partial, then merge).  Negative
 * status for bad head counts. */
int splitkv_fused_launches(int32_t Hq, int32_t Hkv, int32_t d, int32_t block_len, int32_t max_q_len,
                           int32_t n_items, int32_t dtype, int32_t kernel);

/* Steps 3 and 4 in one call (Split-KV card, "All Facts": exact, "Timeline":
 * query-sized partials): the partial attention of splitkv_attn_partial and the
 * merge of splitkv_merge, with the same arguments and results.  With the decode
 * and tensor-core kernels both happen in ONE launch: each CTA writes its
 * partial rows, publishes them (memory fence) and takes a ticket from the
 * counter of its group with an atomic add - a (sequence, K/V head) for the
 * decode kernel, a (sequence, K/V head, 256-row unit) for the tensor-core
 * kernel; the CTA that takes the last ticket sets the counter back to zero and
 * merges the group's partials into out / lse_out.  No CTA waits for another.
 * The tensor-core kernel's merge computes each row exactly as splitkv_merge
 * does, so the two paths give the same bits.  The generic CUDA-core kernel runs
 * the partial and merge launches in turn (splitkv_fused_launches tells which).
 *   tickets (device, caller-owned): n_tickets >= splitkv_ticket_count(...)
 *   uint32 counters, all zero before the first call; every completed call leaves
 *   them zero again.  After a call that reported a device error (status word),
 *   zero them before the next call.  Calls that overlap on the GPU must use
 *   different ticket buffers (and partial buffers). */
int splitkv_attn_fused(const void* q, const void* k_pool, const void* v_pool,
                       int64_t n_pool_blocks, const int32_t* block_table,
                       int32_t max_blocks_per_seq, const int32_t* work, int32_t n_items,
                       int32_t B, int32_t total_q, int32_t max_q_len, int32_t Hq, int32_t Hkv,
                       int32_t d, int32_t block_len, float scale, int32_t causal, int32_t dtype,
                       float* o_part, float* lse_part, int64_t part_rows, uint32_t* tickets,
                       int64_t n_tickets, void* out, float* lse_out, int32_t kernel, void* stream);

/* Step 4, exact merge of the partials (Split-KV card, "All Facts": identical to
 * the unsharded result).  For every query row r of sequence b and head h, over
 * the items i of b:  L = ln sum_i exp(L_i),  O = sum_i exp(L_i - L) O_i;
 * items with L_i = -inf carry weight 0.  Only query-sized tensors are read.
 * In (device): o_part, lse_part as written by splitkv_attn_partial (part_rows
 * rows), work.  A partial row outside part_rows is not read (bit 1 of the
 * device status word is set).
 * Out (device): out [total_q, Hq, d] in dtype, lse_out fp32 [total_q, Hq]. */
int splitkv_merge(const float* o_part, const float* lse_part, int64_t part_rows,
                  const int32_t* work, int32_t B, int32_t total_q, int32_t Hq, int32_t d,
                  int32_t dtype, void* out, float* lse_out, void* stream);

/* Size in bytes of the fixed device array used by splitkv_attention_noalloc. */
#define SPLITKV_NOALLOC_SCRATCH_BYTES (64ll << 20)

/* The whole device path (partial attention, then merge) in one call that
 * allocates nothing - no cudaMalloc, cudaFree or allocating library routine.
 * The pages have no counterpart to it.  It is for callers that cannot allocate
 * device memory themselves: plugins inside a host that owns all device memory
 * through its own arena, loops that must not stall or fail on an allocation,
 * embedders that only pass buffers they already own.  The caller passes the
 * inputs and outputs of splitkv_attn_partial / splitkv_merge, and the work
 * descriptor as the HOST buffer from splitkv_build_work (work_words words); the
 * descriptor copy and the partials live in one fixed array of
 * SPLITKV_NOALLOC_SCRATCH_BYTES bytes declared by the library in device memory,
 * which every GPU that loads the library holds until the process exits.
 *   - Needs 4*words + 4*part_rows*Hq*(d+1) bytes (each part rounded up to 256);
 *     larger problems are rejected with SPLITKV_ERR_CAPACITY before any work.
 *   - work_host is checked on the host before any work: its n_items, B,
 *     total_q and max_q_len must equal the arguments, its offsets must lie
 *     inside work_words, and part_rows must equal the rows its items address
 *     (largest part_row + q_len); otherwise SPLITKV_ERR_INVALID.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current; again after that device's context was
 *     destroyed and created anew); make that first call before any stream
 *     capture.
 *   - Every call shares the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero (each partial row read is written
 *     first).  Calls whose GPU work overlaps - on different streams, or from
 *     different host threads - race on the array and give wrong results.
 *   - A pinned work_host must stay unchanged until the stream has run the copy;
 *     a pageable one is read before the call returns.
 * Kernel choice is SPLITKV_KERNEL_AUTO.  Returns 0 or a negative status. */
int splitkv_attention_noalloc(const void* q, const void* k_pool, const void* v_pool,
                              int64_t n_pool_blocks, const int32_t* block_table,
                              int32_t max_blocks_per_seq, const int32_t* work_host,
                              int64_t work_words, int32_t n_items, int32_t B, int32_t total_q,
                              int32_t max_q_len, int32_t Hq, int32_t Hkv, int32_t d,
                              int32_t block_len, float scale, int32_t causal, int32_t dtype,
                              int64_t part_rows, void* out, float* lse_out, void* stream);

/* ------------------------------------------------------------ backward pass
 * The Split-KV card presents the method for training (intro: asymmetric
 * training with very short queries and very long contexts) and as exact ("All
 * Facts").  With the merged forward's O and L, each shard needs only
 * query-sized tensors (Q, dO, L, D) to compute the exact dK, dV of its own keys
 * and a query-sized partial dQ; the partials sum to dQ.  Chain rule through
 * s = scale q.k, P = exp(s - L), O = P V, for every visible (row r, key j):
 *   dV_j += P_rj dO_r, dP_rj = dO_r.V_j, dS_rj = P_rj (dP_rj - D_r),
 *   dQ_r += scale dS_rj K_j, dK_j += scale dS_rj Q_r.                        */

/* D[row, h] = sum_c O[row, h, c] * dO[row, h, c].  In (device, dtype): o, dout
 * [total_q, Hq, d] (O = splitkv_merge's output).  Out (device): delta fp32
 * [total_q, Hq]. */
int splitkv_bwd_delta(const void* o, const void* dout, int32_t total_q, int32_t Hq, int32_t d,
                      int32_t dtype, float* delta, void* stream);

/* Per-shard backward over the work items of splitkv_build_work.  Tensor cores
 * (tcgen05) for bf16, d = 128, block_len % 128 == 0 and Hq/Hkv dividing 64;
 * CUDA cores otherwise.
 * In (device): q, k_pool, v_pool, block_table, work as for the forward; dout
 * [total_q, Hq, d] (dtype); lse fp32 [total_q, Hq] (splitkv_merge's lse_out);
 * delta fp32 [total_q, Hq].  Out (device, fp32): dq_part [part_rows, Hq, d]
 * (item i's partial dQ in its part_row slab; every row written by this call),
 * dk_pool / dv_pool [n_pool_blocks, block_len, Hkv, d]: the gradient of
 * every key position < kv_len of every sequence is written; other positions
 * are left untouched.  The pages give the backward no formula; this is the
 * chain rule through the forward with the merged L saved (card intro:
 * training with short queries and long contexts). */
/* Which kernel splitkv_attn_backward runs for a shape: SPLITKV_KERNEL_TC or
 * SPLITKV_KERNEL_SIMT (a negative status for bad head counts). */
int splitkv_backward_kernel(int32_t Hq, int32_t Hkv, int32_t d, int32_t block_len, int32_t dtype);

int splitkv_attn_backward(const void* q, const void* k_pool, const void* v_pool, int64_t n_pool_blocks,
                          const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* work,
                          int32_t n_items, int32_t B, int32_t total_q, int32_t max_q_len, int32_t Hq,
                          int32_t Hkv, int32_t d, int32_t block_len, float scale, int32_t causal,
                          int32_t dtype, const void* dout, const float* lse, const float* delta,
                          float* dq_part, int64_t part_rows, float* dk_pool, float* dv_pool,
                          void* stream);

/* dQ[row, h] = sum over the items of the row's sequence of their partial dQ
 * rows (the backward's query-sized exchange).  Out (device): dq fp32
 * [total_q, Hq, d]. */
int splitkv_dq_reduce(const float* dq_part, int64_t part_rows, const int32_t* work, int32_t B,
                      int32_t total_q, int32_t Hq, int32_t d, float* dq, void* stream);

/* Reads and optionally clears the device status word: bit 0, a logical block
 * past max_blocks_per_seq or a block-table entry outside the pool was skipped;
 * bit 1, a work item's partial rows fell outside part_rows (item skipped);
 * bit 2, a wait of a pipelined kernel ran out its time limit (that launch's
 * outputs are not valid); bit 3, a work descriptor did not match the launch's
 * B and n_items (the launch did nothing).  Synchronises the device. */
int splitkv_device_status(uint32_t* status, int32_t clear);

/* Message of the last failed call on this thread ("" if none). */
const char* splitkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPLITKV_H */

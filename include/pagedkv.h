/*
 * pagedkv.h -- C ABI of the GB300 paged KV cache library (libpagedkv.so).
 *
 * Two planes sit behind this header, as in "MiniPaged-Qwen: Paged KV Cache
 * 与 KV Block Manager" (blog.zsmgc.love) §8: a host-side metadata plane (the
 * block manager, plain C++) and a device data plane (per-layer K/V caches and
 * the CUDA kernels that write and read them, sm_103a).
 *
 * Conventions for every entry point:
 *   - The return value is a kv_status_t; KV_OK (0) means success.  No C++
 *     exception crosses this boundary.  kv_status_string() names each code.
 *   - Host pointers: caller-owned host memory, read or written only during
 *     the call.  Device pointers: caller-owned device memory (for example
 *     torch tensors); the library never frees them.
 *   - Kernel entry points are asynchronous on the given stream (a
 *     cudaStream_t passed as void*; NULL is the legacy default stream).  They
 *     validate arguments on the host, launch, and report launch errors as
 *     KV_ERR_CUDA without synchronising.  Device-side bounds violations are
 *     recorded in a device error word (see kv_device_error) and the offending
 *     access is skipped; nothing traps.
 *   - Tensors are dense and row-major unless a stride argument says
 *     otherwise.  Cache layout, per layer: [num_blocks, block_size,
 *     num_kv_heads, head_dim], elements of the given dtype.
 *   - Integers that index tokens, slots or blocks are int32 on the device
 *     (block tables, seq_lens, slot_mapping), so a pool holds at most
 *     2^31 - 1 slots.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */

typedef enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = 1,   /* bad sizes, ids, dtype or head_dim; LLM-algo ch.22 rejects
                               request_id < 0 and prompt_len <= 0 (Step 4, Request) */
  KV_ERR_OOM = 2,           /* not enough free blocks; state unchanged (LLM-algo ch.22
                               Step 4: atomic prefill, decode rollback) */
  KV_ERR_UNKNOWN_SEQ = 3,   /* the sequence id is not live */
  KV_ERR_DUPLICATE_SEQ = 4, /* second prefill of a live sequence (LLM-algo ch.22) */
  KV_ERR_DOUBLE_FREE = 5,   /* release of an already released sequence ("从零实现一个
                               mini vLLM: Block Manager", section on releasing blocks) */
  KV_ERR_INVARIANT = 6,     /* manager state violates an invariant (MiniPaged-Qwen §15) */
  KV_ERR_CUDA = 7,          /* a CUDA runtime call or launch failed */
  KV_ERR_DEVICE_BOUNDS = 8, /* a kernel met a block index or slot outside the pool */
  KV_ERR_WORKSPACE = 9,     /* the workspace passed is smaller than required */
  KV_ERR_DEVICE_TIMEOUT = 10,/* a bounded device-side wait gave up */
  KV_ERR_DEVICE_STEP = 11   /* paged_decode_step: a sequence's new-token row is not written
                               to that sequence's newest slot (inconsistent step metadata) */
} kv_status_t;

/* Static, NUL-terminated text for a status code (never NULL).  No passage:
 * the pages raise Python exceptions with messages; this is their C form. */
const char* kv_status_string(int status);

typedef enum { KV_DTYPE_F32 = 0, KV_DTYPE_F16 = 1, KV_DTYPE_BF16 = 2 } kv_dtype_t;

/* ------------------------------------------------- host metadata plane */
/*
 * The block manager: MiniPaged-Qwen §8 (SequenceState, KVBlockManager),
 * §9 (append_token), §15 (invariants); "从零实现一个 mini vLLM: Block
 * Manager" (allocate_for_prefill, append_slot_for_decode, free_sequence,
 * can_allocate, can_append_slots); LLM-algo ch.22 Step 4 (atomic prefill,
 * decode rollback, release validation, allocation report).
 *
 * Free-list policy: blocks are taken from the front of the free list;
 * released blocks are appended at the back in block-table order.  The
 * handle is not thread-safe: serialise calls on one handle.
 */
typedef struct kvbm_s* kvbm_t;

/* Create a manager over blocks 0..num_blocks-1 of block_size slots each.
 * initial_free_order: NULL for 0..num_blocks-1, else a host array of
 * num_blocks int32 that must be a permutation of the pool (else
 * KV_ERR_INVALID_ARG).  num_blocks * block_size must fit in int32.
 * *out receives the handle; release it with kvbm_destroy.  The pool of
 * MiniPaged-Qwen §8 (KVBlockManager(num_blocks, block_size)) and LLM-algo
 * ch.22 Step 4 (KVCacheManager: every block free at the start). */
int kvbm_create(int64_t num_blocks, int32_t block_size, const int32_t* initial_free_order,
                kvbm_t* out);
/* Release the handle and everything it holds (h may be NULL).  No passage:
 * the pages' managers are Python objects their runtime frees; a C ABI needs
 * an explicit release. */
int kvbm_destroy(kvbm_t h);

/* *ok = 1 iff ceil(num_tokens / block_size) blocks are free (num_tokens >= 1):
 * can_allocate of "从零实现一个 mini vLLM: Block Manager" (prefill admission). */
int kvbm_can_allocate(kvbm_t h, int64_t num_tokens, int* ok);

/* Prefill: allocate ceil(num_tokens / block_size) blocks at once for a new
 * sequence seq_id (>= 0) holding num_tokens (>= 1) tokens.  slots_out, if not
 * NULL, receives num_tokens int32 slots: slot[t] = table[t / bs] * bs + t % bs
 * (MiniPaged-Qwen §3).  All or nothing: on KV_ERR_OOM nothing changes.
 * KV_ERR_DUPLICATE_SEQ if seq_id is live. */
int kvbm_allocate_for_prefill(kvbm_t h, int64_t seq_id, int64_t num_tokens, int32_t* slots_out);

/* Decode append (MiniPaged-Qwen §9): *slot_out = slot of position L (the
 * current length), allocating a block only when L / bs == len(table); then
 * L += 1.  On KV_ERR_OOM the length and table are unchanged. */
int kvbm_append_slot_for_decode(kvbm_t h, int64_t seq_id, int32_t* slot_out);

/* num_tokens consecutive appends to a live sequence (chunked prefill), all
 * or nothing on OOM.  slots_out (nullable) receives num_tokens slots.  The
 * chunk of a chunked prefill in "从零实现一个 mini vLLM: Block Manager" takes
 * its slots this way: MiniPaged-Qwen §9's append, num_tokens times. */
int kvbm_append_slots(kvbm_t h, int64_t seq_id, int64_t num_tokens, int32_t* slots_out);

/* Prefix sharing ("paged-attention-impl-detail", section Copy-on-Write共享:
 * requests with a common prompt prefix share its physical blocks, each
 * block counting its sharers).  A new sequence child_id (>= 0, not live)
 * starts as the first prefix_len tokens of live sequence parent_id
 * (1 <= prefix_len <= parent's length): its table is the parent's first
 * ceil(prefix_len / bs) entries and each of those blocks gains a
 * reference.  No block is taken.  Copy-on-write (same section): when a
 * sequence's next write lands in a block that another table also holds
 * (only possible while prefix_len % bs != 0 left it partly filled), the
 * append first takes a free block, queues a copy old -> new of the whole
 * block (see kvbm_take_copies), drops one reference from the old block and
 * writes into the new one.  Appends count that block in their OOM check.
 * Released blocks return to the free list when no table refers to them.
 * KV_ERR_UNKNOWN_SEQ (parent not live), KV_ERR_DUPLICATE_SEQ (child live),
 * KV_ERR_INVALID_ARG (prefix_len out of range). */
int kvbm_fork(kvbm_t h, int64_t parent_id, int64_t child_id, int64_t prefix_len);

/* Copy-on-write copies queued since the last call, oldest first: block
 * src[i] must be copied to block dst[i] (K and V, every layer) on the
 * device before the cache writes of the slots returned by the appends that
 * queued them, and before any attention over those sequences
 * (paged_copy_blocks).  *n_out = the number queued.  With src and dst both
 * NULL the call only reports that number; otherwise the queue is copied
 * out and emptied when it fits in cap (else KV_ERR_INVALID_ARG and nothing
 * changes). */
int kvbm_take_copies(kvbm_t h, int32_t* src, int32_t* dst, int64_t cap, int64_t* n_out);

/* *out = the number of table entries (over all live sequences) that refer
 * to block (0 = free): the per-block reference count of
 * "paged-attention-impl-detail", section Copy-on-Write共享. */
int kvbm_block_refcount(kvbm_t h, int32_t block, int32_t* out);

/* *ok = 1 iff one decode append to each listed sequence fits in the free
 * blocks (counts sequences whose next write opens a new block or copies a
 * shared one): can_append_slots of "从零实现一个 mini vLLM: Block
 * Manager" (decode admission). */
int kvbm_can_append_slots(kvbm_t h, const int64_t* seq_ids, int64_t n, int* ok);

/* One decode step for n distinct live sequences: append one slot to each
 * (slots_out[n], nullable), then export their tables and lengths as
 * kvbm_export does (block_tables / seq_lens nullable).  All or nothing on
 * OOM (LLM-algo ch.22 Step 4, decode rollback).  A repeated id is
 * KV_ERR_INVALID_ARG.  MiniPaged-Qwen §9 (append) then §16.2 (export). */
int kvbm_decode_step(kvbm_t h, const int64_t* seq_ids, int64_t n, int64_t max_blocks,
                     int32_t* slots_out, int32_t* block_tables, int32_t* seq_lens);

/* One serving step's host metadata in a single call ("从零实现一个 mini vLLM:
 * Block Manager", section on the ModelRunner: slot mapping, block tables and
 * context lengths built from the manager's state):
 *   1. release free_ids (e.g. the previous step's finished sequences);
 *   2. prefill-allocate each new sequence prefill_ids[i] of prefill_lens[i]
 *      tokens, as kvbm_allocate_for_prefill;
 *   3. append one decode slot to each of decode_ids;
 *   4. write slot_mapping[n_slots], n_slots = sum(prefill_lens) + n_decode +
 *      n_pad: the prefill slots in order, then the decode slots, with -1 at
 *      the strictly increasing positions pad_positions[n_pad];
 *   5. export the decode sequences' tables and lengths as kvbm_export.
 * Steps 2-3 are all or nothing: everything is validated (ids, lengths,
 * padding, free blocks) before any allocation, so on an error only the
 * releases of step 1 have happened.  Outputs are nullable. */
int kvbm_prepare_step(kvbm_t h, const int64_t* free_ids, int64_t n_free, const int64_t* prefill_ids,
                      const int64_t* prefill_lens, int64_t n_prefill, const int64_t* decode_ids,
                      int64_t n_decode, const int64_t* pad_positions, int64_t n_pad, int64_t max_blocks,
                      int32_t* slot_mapping, int32_t* block_tables, int32_t* seq_lens);

/* Release every block of seq_id once (MiniPaged-Qwen §5.3): each loses one
 * reference and returns to the back of the free list, in table order, when
 * none is left.  The table is validated first; a corrupt table gives
 * KV_ERR_INVARIANT and changes nothing.  KV_ERR_DOUBLE_FREE for an id
 * already released (and not prefilled again), KV_ERR_UNKNOWN_SEQ for an id
 * never seen. */
int kvbm_free_sequence(kvbm_t h, int64_t seq_id);

/* *out = the number of free blocks: get_num_free_blocks, one of the three
 * actions of the minimal block manager ("从零实现一个 mini vLLM: Block
 * Manager", section "Block Manager 要维护哪些东西"). */
int kvbm_num_free_blocks(kvbm_t h, int64_t* out);

/* Copy the free list, front first, into out[cap]; *n_out = its length.
 * KV_ERR_INVALID_ARG if cap is too small.  The free_blocks list of
 * MiniPaged-Qwen §8 and LLM-algo ch.22 Step 4, for inspection and tests. */
int kvbm_get_free_list(kvbm_t h, int32_t* out, int64_t cap, int64_t* n_out);

/* *out = seq_id's length (MiniPaged-Qwen §8 SequenceState.length).
 * KV_ERR_UNKNOWN_SEQ if it is not live. */
int kvbm_seq_len(kvbm_t h, int64_t seq_id, int64_t* out);

/* Copy seq_id's block table into out[cap]; *n_out = its length
 * (MiniPaged-Qwen §8 SequenceState.block_table).  KV_ERR_UNKNOWN_SEQ if it
 * is not live, KV_ERR_INVALID_ARG if cap is too small. */
int kvbm_get_block_table(kvbm_t h, int64_t seq_id, int32_t* out, int64_t cap, int64_t* n_out);

/* Metadata export (MiniPaged-Qwen §16.2 get_block_table_tensor /
 * get_seq_lens_tensor): block_tables[n][max_blocks] row-major, padded with
 * -1; seq_lens[n].  Either output may be NULL.  KV_ERR_INVALID_ARG if a
 * table is longer than max_blocks. */
int kvbm_export(kvbm_t h, const int64_t* seq_ids, int64_t n, int64_t max_blocks,
                int32_t* block_tables, int32_t* seq_lens);

/* kvbm_export's block tables (MiniPaged-Qwen §16.2) written as an update of
 * a buffer that already holds an earlier export: for row i, prev_ids[i] and prev_nblocks[i] say
 * which sequence the row held and how many of its entries were blocks (the
 * rest -1), as this call left them (initialise prev_ids to -1 for a buffer
 * never exported into).  A row that held the same sequence gets its block
 * entries written and -1 only over entries that were blocks before; any
 * other row is written in full.  The result equals kvbm_export's, with
 * the same max_blocks for every call on one buffer.  prev_ids /
 * prev_nblocks are updated.  All caller-owned host memory; validation and
 * errors as kvbm_export (nothing written on an error). */
int kvbm_export_update(kvbm_t h, const int64_t* seq_ids, int64_t n, int64_t max_blocks, int32_t* block_tables,
                       int64_t* prev_ids, int32_t* prev_nblocks);

/* KV_OK iff: every table entry is in range and appears once in its table,
 * each block's reference count equals the table entries referring to it,
 * the free list holds exactly the unreferenced blocks once each, referenced
 * + free = the pool, len(table) = ceil(L / bs) (MiniPaged-Qwen §15;
 * LLM-algo ch.22 Step 3; a block is shared across sequences only through
 * kvbm_fork, as "从零实现一个 mini vLLM: Block Manager" allows for prefix
 * caching and copy-on-write).  Else KV_ERR_INVARIANT. */
int kvbm_check_invariants(kvbm_t h);

typedef struct {
  int64_t num_blocks;
  int64_t block_size;
  int64_t num_free_blocks;
  int64_t num_sequences;
  int64_t logical_tokens;     /* sum of sequence lengths */
  int64_t allocated_tokens;   /* sum of len(table) * block_size */
  int64_t unused_tail_tokens; /* allocated - logical (MiniPaged-Qwen §6.2) */
} kvbm_stats_t;

/* Pool and usage counts: free blocks, live sequences, logical and allocated
 * tokens and the unused block tails between them (MiniPaged-Qwen §6.2;
 * LLM-algo ch.22 Step 4's allocation report, summed over sequences). */
int kvbm_stats(kvbm_t h, kvbm_stats_t* out);

/* *out = the number of ranges of consecutive released ids the manager
 * remembers, so that a second release of an id answers KV_ERR_DOUBLE_FREE
 * (LLM-algo ch.22 Step 4 raises on a second release) until the id is
 * prefilled again.  Released ids are kept as merged ranges, so the memory
 * this takes follows the gaps between released ids, not their number: ids
 * released in order (a serving loop numbering its requests) stay one range. */
int kvbm_released_ranges(kvbm_t h, int64_t* out);

/* LLM-algo ch.22 allocation_report for one sequence: allocated tokens,
 * unused tail tokens, utilisation = logical / allocated. */
int kvbm_allocation_report(kvbm_t h, int64_t seq_id, int64_t* logical_tokens,
                           int64_t* allocated_tokens, int64_t* unused_tail_tokens,
                           double* utilization);

/* Debug aid from "从零实现一个 mini vLLM: Block Manager" (invariants section):
 * out[num_blocks] receives the owning sequence id of each block, -1 if free,
 * -2 if several sequences share it (kvbm_fork). */
int kvbm_owner_table(kvbm_t h, int64_t* out, int64_t cap);

/* KV capacity ledger (LLM-algo ch.22 estimate_kv_cache_bytes; MiniPaged-Qwen
 * §2): bytes/token = 2 * layers * kv_heads * head_dim * dtype_bytes; a block
 * holds block_size tokens; the pool num_blocks blocks.  Outputs nullable. */
int kv_cache_ledger(int64_t num_blocks, int64_t block_size, int64_t num_layers,
                    int64_t num_kv_heads, int64_t head_dim, int64_t dtype_bytes,
                    int64_t* bytes_per_token, int64_t* bytes_per_block, int64_t* total_bytes);

/* ---------------------------------------------------- device data plane */

/* Cache write (MiniPaged-Qwen §12): for each token t < num_tokens with
 * slot = slot_mapping[t] != -1, copy k[t] ([num_kv_heads, head_dim]) to
 * k_cache[slot / block_size][slot % block_size] and v[t] likewise.
 * slot == -1 marks a padded token: nothing is read or written for it.  Any
 * other slot outside [0, num_blocks * block_size) is skipped and recorded as
 * KV_ERR_DEVICE_BOUNDS in the device error word.  Bit-exact copy.
 *   k, v: device, token t at k + t * k_token_stride (elements); the heads of
 *         one token are contiguous ([num_kv_heads, head_dim]).
 *         Pass stride = num_kv_heads * head_dim for a dense [N, Hkv, D].
 *   k_cache, v_cache: device, [num_blocks, block_size, num_kv_heads, head_dim].
 *   slot_mapping: device int32[num_tokens].
 * num_tokens == 0 launches nothing.  Two tokens with the same slot race. */
int paged_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                            const int32_t* slot_mapping, int64_t num_tokens,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int64_t num_blocks, int64_t k_token_stride, int64_t v_token_stride,
                            int dtype, void* stream);

/* paged_reshape_and_cache for num_layers layers in one launch.  One block
 * table and one slot mapping serve every layer ("MiniPaged-Qwen" §16: the
 * step's metadata is built once and read by every layer's attention; the
 * capacity ledger's per-block bytes cover all layers, see kv_cache_ledger).
 *   k, v: layer l's rows at + l * k_layer_stride / v_layer_stride elements,
 *     then as for paged_reshape_and_cache (token stride, dense heads).
 *   k_cache, v_cache: layer l's cache [num_blocks, block_size, num_kv_heads,
 *     head_dim] at + l * cache_layer_stride elements (>= one layer's cache
 *     when num_layers > 1, else KV_ERR_INVALID_ARG).
 * Everything else (padding, bounds, bit-exactness) as paged_reshape_and_cache. */
int paged_reshape_and_cache_layers(const void* k, const void* v, void* k_cache, void* v_cache,
                                   const int32_t* slot_mapping, int64_t num_tokens, int32_t num_layers,
                                   int64_t k_layer_stride, int64_t v_layer_stride,
                                   int64_t cache_layer_stride, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int64_t num_blocks, int64_t k_token_stride,
                                   int64_t v_token_stride, int dtype, void* stream);

/* fp8 KV cache ("paged-attention-impl-detail", 实践建议 4: the KV cache
 * inside a block can be quantised on its own).  Codes are OCP FP8 E4M3
 * bytes in caches [num_blocks, block_size, num_kv_heads, head_dim]; each
 * (token, kv head) row has one float32 scale, stored in scale arrays
 * [num_blocks, num_kv_heads, block_size] (a block's scales are its own).
 * A row is quantised as: scale = amax / 448 (1 for an all-zero row), each
 * value divided by the scale in float32 with one correct rounding, then
 * rounded to E4M3, nearest-even, saturating at +-448.  Its dequantised value
 * is code * scale.  The write replaces paged_reshape_and_cache (same slot
 * rules: -1 skipped, out-of-pool slots skipped and recorded; a padded
 * token's input row, which must exist like every row t < num_tokens, may be
 * read); k, v are
 * fp16 or bf16 (dtype), head_dim 64, 128 or 256, token strides even, k/v
 * 4-byte aligned, caches 8-byte aligned.  Bit-exact against the
 * definition above. */
int paged_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                                float* k_scales, float* v_scales, const int32_t* slot_mapping,
                                int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                int32_t block_size, int64_t num_blocks, int64_t k_token_stride,
                                int64_t v_token_stride, int dtype, void* stream);

/* paged_decode_attention over fp8 caches and their scales: K_j, V_j are the
 * dequantised rows (the fp8 KV cache of "paged-attention-impl-detail",
 * 实践建议 4, read by MiniPaged-Qwen §13's decode attention).  q and out are fp16 or bf16 (dtype); head_dim 128,
 * block_size 16 or 32, at most 16 query heads per kv head and 4096
 * sequences (else KV_ERR_INVALID_ARG).  The stream-K tensor-core kernel:
 * TMA brings the E4M3 rows and the scales, E4M3 pairs convert exactly to
 * the MMA type, each token's K scale multiplies its scores and its V scale
 * its softmax weight.  workspace: paged_decode_workspace_size() bytes for
 * the same sizes and dtype, blocks_per_split 0.  Other arguments, results
 * and errors are those of paged_decode_attention; all pointers 16-byte
 * aligned. */
int paged_decode_attention_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scales, const float* v_scales,
                               const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs,
                               int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
                               int64_t max_seq_len, float scale, int dtype, void* workspace,
                               size_t workspace_bytes, void* stream);

/* paged_decode_step for fp8 caches ("paged-attention-impl-detail", 实践建议
 * 4; MiniPaged-Qwen §12-§13): the step's quantised cache write
 * (exactly as paged_reshape_and_cache_fp8) and decode attention over the
 * fp8 caches (exactly as paged_decode_attention_fp8) in one call, under the
 * requirement and with the checks of paged_decode_step (new_token_row,
 * KV_ERR_DEVICE_STEP).  One launch when the rows of k and v are 8-byte
 * aligned: the consumer warps quantise and scatter the rows, and the tile
 * holding position seq_lens[b] - 1 quantises that token itself with the same
 * float32 steps, so codes, scales and outputs are bit-identical to the two
 * calls in sequence.  Otherwise (rows not 8-byte aligned, or more than two
 * rows per consumer warp of the grid, as with a prefill chunk, where the
 * in-launch quantisation would hold up the first tiles) the two calls in
 * stream order. */
int paged_decode_step_fp8(void* out, const void* q, const void* k, const void* v,
                          const int32_t* slot_mapping, int64_t num_tokens, int64_t k_token_stride,
                          int64_t v_token_stride, const int32_t* new_token_row, void* k_cache,
                          void* v_cache, float* k_scales, float* v_scales, const int32_t* block_tables,
                          const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                          int32_t max_blocks_per_seq, int64_t max_seq_len, float scale, int dtype,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Chunked-prefill attention through block tables ("从零实现一个 mini vLLM:
 * Block Manager": a chunked prefill allocates the chunk's slots, writes its
 * K/V, then attends through the table; "MiniPaged-Qwen" §13-§14).  For each
 * sequence b, its chunk is rows query_start_loc[b] .. query_start_loc[b+1]-1
 * of q and out: the last n_b of its seq_lens[b] = L_b positions, whose K/V
 * the cache write has already stored.  Chunk token t (position
 * p = L_b - n_b + t) attends to keys 0..p of its sequence:
 *   out[r, qh] = sum_{j <= p} softmax_j(scale * q[r, qh] . K_j) V_j,
 *   kvh = qh / (num_heads / num_kv_heads), K_j read through block_tables[b].
 * A chunk of one token is decode.
 *   q, out: device [num_query_tokens, num_heads, head_dim] of dtype (fp16
 *     or bf16), 16-byte aligned; caches as for paged_decode_attention.
 *   query_start_loc: device int32[num_seqs + 1], non-decreasing, every
 *     entry in [0, num_query_tokens].
 *   max_query_len: host upper bound of the chunk lengths (sizes the grid).
 *     A longer chunk's rows past the grid's reach are not computed, and the
 *     launch records KV_ERR_DEVICE_BOUNDS.
 *   head_dim 64 or 128.
 * A chunk longer than its sequence or reaching past num_query_tokens, or a
 * sequence longer than its table row, is recorded as KV_ERR_DEVICE_BOUNDS
 * (the former two's rows are not written).  Block sizes 16, 32, 64 and 128
 * run on the 5th-generation tensor cores (tcgen05, accumulators in tensor
 * memory, K/V tiles by TMA); other block sizes on mma.sync.  fp32
 * accumulation and online softmax, one rounding to dtype. */
int paged_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            const int32_t* query_start_loc, int64_t num_query_tokens, int32_t num_seqs,
                            int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                            int32_t max_blocks_per_seq, int32_t max_query_len, float scale, int dtype,
                            void* stream);

/* Copy-on-write block copies (kvbm_take_copies): for each i < n, block
 * dst[i] of every layer's K and V cache becomes a copy of block src[i]
 * ("paged-attention-impl-detail", copy_on_write: the new block's k and v
 * take the old block's).  One launch for all pairs and layers.
 *   k_cache, v_cache: device, num_layers caches [num_blocks, block_size,
 *     num_kv_heads, head_dim] of dtype, layer l at + l * layer_stride
 *     elements (16-byte aligned; pass 0 for one layer).
 *   src, dst: device int32[n].  A pair with an index outside [0, num_blocks)
 *     is skipped and recorded as KV_ERR_DEVICE_BOUNDS.  A destination that is
 *     also a source of another pair, or two pairs with one destination, race.
 * Bit-exact copies.  n == 0 launches nothing. */
int paged_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int64_t n,
                      int32_t num_layers, int64_t layer_stride, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int64_t num_blocks, int dtype, void* stream);

/* paged_copy_blocks for fp8 (E4M3) caches ("paged-attention-impl-detail",
 * copy_on_write, with the per-block quantisation of 实践建议 4): block
 * dst[i] takes block src[i]'s codes (K and V) and its float32 scales.
 *   k_cache, v_cache: device, num_layers code caches [num_blocks, block_size,
 *     num_kv_heads, head_dim] of bytes, layer l at + l * layer_stride bytes
 *     (>= one layer's codes when num_layers > 1; a multiple of 16).
 *   k_scales, v_scales: device, num_layers scale arrays [num_blocks,
 *     num_kv_heads, block_size] of float32, layer l at
 *     + l * num_blocks * num_kv_heads * block_size floats.
 *   src, dst, n: as for paged_copy_blocks.
 * Each block's codes and scales must be whole 16-byte multiples (else
 * KV_ERR_INVALID_ARG).  Two launches on `stream`; indices outside the pool
 * are recorded as KV_ERR_DEVICE_BOUNDS and skipped. */
int paged_copy_blocks_fp8(void* k_cache, void* v_cache, float* k_scales, float* v_scales, const int32_t* src,
                          const int32_t* dst, int64_t n, int32_t num_layers, int64_t layer_stride,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                          void* stream);

/* Split-K plan for a decode call with these sizes.  blocks_per_split: 0
 * chooses automatically (from the SM count of the current device, the
 * number of (sequence, kv head) pairs and max_seq_len); > 0 forces that many
 * logical blocks per split (split kernels only).  Outputs (each nullable):
 * *kernel_out = 0 for the SIMT split kernel (fp32 and shapes the tensor-core
 * kernels do not take), 1 for the TMA + tensor-core split kernel (forced
 * splits, or more than 4096 sequences), 2 for the TMA + tensor-core
 * stream-K kernel (the fp16/bf16 default: one cooperative wave of
 * persistent CTAs, each taking an equal share of all (sequence, kv head,
 * block) tiles, and combining cut sequences inside the same launch); the
 * blocks per split and number of splits S (split kernels); the workspace
 * bytes.  Kernel 2 launches one kernel; kernels 0 and 1 add a log-sum-exp
 * merge kernel when S > 1.  No passage: the pages' decode attention
 * (MiniPaged-Qwen §13) reads each sequence whole; the partition is this
 * library's, and the merge restates §17.3's online softmax across pieces.
 * max_seq_len is an upper bound of the seq_lens the call will see. */
int paged_decode_plan(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int64_t max_seq_len, int32_t blocks_per_split, int dtype,
                      int32_t* kernel_out, int32_t* blocks_per_split_out, int32_t* num_splits_out,
                      size_t* workspace_bytes_out);

/* Bytes of device workspace paged_decode_attention needs for these sizes
 * (0 when no split is needed); same arguments as paged_decode_plan.  The
 * workspace holds the partial results (acc, m, l) of the library's work
 * partition (split-K, or stream-K ranges that cut a sequence) and its ready
 * flags.  No passage: the pages' decode attention ("MiniPaged-Qwen" §13)
 * reads each sequence whole; the partition is this library's way of
 * keeping every SM busy when the batch alone would not. */
int paged_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, int64_t max_seq_len,
                                int32_t blocks_per_split, int dtype, size_t* bytes_out);

/* Single-query paged decode attention (MiniPaged-Qwen §13, §14, §17.3):
 *   out[b, qh, :] = sum_{j < seq_lens[b]} softmax_j(scale * q[b, qh] . K_j) V_j,
 * with kv head kvh = qh / (num_heads / num_kv_heads) and K_j, V_j read at
 * cache[block_tables[b][j / bs]][j % bs][kvh].  Only the first
 * ceil(seq_lens[b] / bs) table entries are read; slots past seq_lens[b] in
 * the last block are never used, whatever they hold.  seq_lens[b] == 0
 * gives a zero output row.  fp32 accumulation, one rounding to dtype.
 *   out, q: device, [num_seqs, num_heads, head_dim] of dtype, 16-byte aligned.
 *   k_cache, v_cache: device caches as above, 16-byte aligned.
 *   block_tables: device int32 [num_seqs, max_blocks_per_seq].
 *   seq_lens: device int32 [num_seqs], each <= max_seq_len.
 *   max_seq_len: host upper bound of seq_lens; sizes the split-K partition.
 *   blocks_per_split: 0 = automatic, else forced (see paged_decode_plan).
 *   workspace: device, >= paged_decode_workspace_size() bytes, 256-byte
 *     aligned, or NULL when that size is 0 (else KV_ERR_WORKSPACE).
 *     Clobbered; calls that share a workspace must be ordered on one stream.
 *     Its contents need no initialisation: the stream-K kernel's ready flags
 *     carry a tag unique to each call (a random base plus a call counter),
 *     and each flag is cleared by its one reader.  A CUDA graph replays the
 *     tag it captured; after a call reports KV_ERR_DEVICE_TIMEOUT, a late
 *     flag can be left set, so zero the workspace (or capture the graph
 *     again) before replaying a graph that uses it.
 * num_heads must be a multiple of num_kv_heads.  head_dim: fp32 a multiple
 * of 4 up to 256; fp16/bf16 a multiple of 8 up to 256.
 * Bounds violations (a table entry outside [0, num_blocks), a seq_len above
 * max_blocks_per_seq * block_size or above what the split plan covers) are
 * skipped or clamped and recorded as KV_ERR_DEVICE_BOUNDS in the device
 * error word; that row's result is then unspecified. */
int paged_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* seq_lens,
                           int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, int64_t num_blocks,
                           int32_t max_blocks_per_seq, int64_t max_seq_len, float scale,
                           int32_t blocks_per_split, int dtype, void* workspace,
                           size_t workspace_bytes, void* stream);

/* One decode step's device work in one call: the cache write of the step's
 * new tokens (exactly as paged_reshape_and_cache) followed by decode
 * attention over the batch (exactly as paged_decode_attention with
 * blocks_per_split = 0), with the new tokens visible to the attention.
 * "MiniPaged-Qwen" §12 (write the token's K/V at its slot) and §13 (attend
 * over the history including it); "从零实现一个 mini vLLM: Block Manager"
 * (a decode step writes the input token's K/V in its own forward).
 *   k, v, slot_mapping, num_tokens, k/v_token_stride: the step's new tokens,
 *     as for paged_reshape_and_cache (prefill chunks, decode tokens, -1 pads).
 *   new_token_row: device int32[num_seqs]; new_token_row[b] is the row of
 *     k/v holding sequence b's newest token, position seq_lens[b] - 1, or -1
 *     when the step writes no token of sequence b.  May be NULL only when
 *     num_tokens == 0.
 *   The remaining arguments are those of paged_decode_attention.
 * Requirement: the only slots this step writes that the attention reads are
 * those positions seq_lens[b] - 1 named by new_token_row.  When the stream-K
 * kernel applies (paged_decode_plan kernel 2) and the rows of k and v are
 * 16-byte aligned, the call is ONE launch: its warps scatter the rows while
 * the first K/V tiles stream in, and the tile holding position
 * seq_lens[b] - 1 takes that token from row new_token_row[b] rather than
 * from the cache, so no tile depends on a write of the same launch.  The
 * kernel checks that slot_mapping[new_token_row[b]] is that position's slot
 * (block_tables[b][(L - 1) / bs] * bs + (L - 1) % bs) and records
 * KV_ERR_DEVICE_STEP in the device error word when it is not, or when the
 * row is >= num_tokens.  Otherwise the call launches the cache write, then
 * attention, in stream order.  num_seqs == 0 runs the cache write alone.
 * Results are bit-identical to the two calls in sequence: same cache bytes,
 * same attention arithmetic. */
int paged_decode_step(void* out, const void* q, const void* k, const void* v,
                      const int32_t* slot_mapping, int64_t num_tokens, int64_t k_token_stride,
                      int64_t v_token_stride, const int32_t* new_token_row, void* k_cache,
                      void* v_cache, const int32_t* block_tables, const int32_t* seq_lens,
                      int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
                      int64_t max_seq_len, float scale, int dtype, void* workspace,
                      size_t workspace_bytes, void* stream);

/* paged_decode_attention without a workspace argument, for callers that
 * cannot allocate device memory themselves (their GPU memory belongs to
 * another allocator, or allocation is forbidden or too slow where they run).
 * The pages have no counterpart: this is a deployment convenience.
 * Scratch comes from one fixed array the library defines in device memory,
 * paged_decode_static_scratch_bytes() bytes (8 MiB), which every GPU that
 * loads the library holds until the process exits.  The call allocates
 * nothing.  Its first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, synchronous) with that device current: make that
 * first call before any stream capture.  Sizes whose workspace
 * (paged_decode_workspace_size) exceeds the array return KV_ERR_WORKSPACE
 * and launch nothing.  All calls on a device share the array: calls that
 * overlap on the GPU (other streams, other threads) race; order them on one
 * stream.  Nothing in it needs clearing between calls.  The address found
 * by the first call is kept for the life of the process: do not use this
 * entry point after cudaDeviceReset (or any other teardown of the device's
 * primary context) in the same process.  Other arguments, results and
 * errors are those of paged_decode_attention. */
int paged_decode_attention_static_scratch(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          const int32_t* seq_lens, int32_t num_seqs,
                                          int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                          int32_t block_size, int64_t num_blocks,
                                          int32_t max_blocks_per_seq, int64_t max_seq_len,
                                          float scale, int32_t blocks_per_split, int dtype,
                                          void* stream);

/* Size in bytes of the fixed scratch array behind
 * paged_decode_attention_static_scratch (no passage; see that entry). */
size_t paged_decode_static_scratch_bytes(void);

/* Read (and, if reset != 0, clear) the device error word of the current
 * device: *status_out = KV_OK or the first KV_ERR_DEVICE_* code recorded by
 * a kernel since the last reset.  Synchronises the current device.  The
 * device side of LLM-algo ch.22's rule that invalid input raises an error
 * rather than passing silently: kernels record, they do not trap. */
int kv_device_error(int reset, int* status_out);

/* Text of the last CUDA error an entry point of this library met on the
 * calling thread (the cause of its most recent KV_ERR_CUDA); static storage,
 * never NULL.  No passage (diagnostics of the C ABI). */
const char* kv_last_cuda_error(void);

/* ------------------------------------------------ native step runner */
/*
 * One serving decode step of one layer per call ("从零实现一个 mini vLLM:
 * Block Manager", section on the ModelRunner: the CPU builds slot mapping,
 * block tables and context lengths from the manager and hands them to the
 * GPU with the step's K/V; "MiniPaged-Qwen" §8: CPU metadata plane, GPU data
 * plane).  kvstep_run does, in order:
 *   1. kvbm_prepare_step on the manager into a page-locked buffer, each
 *      decode sequence's row in the step's K/V (the prefill tokens come
 *      first, then one token per decode sequence, around the pads), and the
 *      copy-on-write copies the step's appends queued (kvbm_take_copies);
 *   2. one async host-to-device copy of that buffer on a side stream (with
 *      host_io, also the step's q, k and v), so the copy overlaps the
 *      previous step's kernel;
 *   3. on cfg.stream after an event wait on that copy: paged_copy_blocks for
 *      the queued copies (when there are any), then paged_decode_step;
 *   4. with host_io, the output back to the caller's host buffer on a
 *      second side stream.
 * Four metadata buffers rotate between steps; their reuse is ordered by
 * events (the host waits only for work issued four steps earlier).
 * The runner allocates its buffers (page-locked host, device) and two side
 * streams at kvstep_create.  Not thread-safe: one thread drives a runner,
 * and the manager must not be used by anyone else meanwhile.  The device
 * current at kvstep_create must be current at every later call.
 */
typedef struct kvstep_s* kvstep_t;

typedef struct {
  int32_t num_seqs;            /* decode sequences per step (n_decode of every kvstep_run) */
  int32_t num_heads, num_kv_heads, head_dim, block_size;
  int64_t num_blocks;
  int32_t max_blocks_per_seq;  /* columns of the exported block tables */
  int64_t max_seq_len;         /* upper bound of every step's seq_lens */
  float scale;
  int32_t dtype;               /* kv_dtype_t */
  int64_t num_step_tokens;     /* rows of k/v per step = prefill tokens + num_seqs + pads */
  void* k_cache;               /* device caches [num_blocks, block_size, num_kv_heads, head_dim] */
  void* v_cache;
  void* workspace;             /* device, >= paged_decode_workspace_size(..., 0, ...) bytes */
  size_t workspace_bytes;
  void* stream;                /* compute stream (cudaStream_t) */
  int32_t host_io;             /* 0: q/k/v/out given to kvstep_run are device buffers;
                                  1: page-locked host buffers, copied in and out by the runner;
                                  2: q/k/v staged by the caller in the runner's page-locked
                                     buffers (kvstep_stage_buffer) and copied in with the step's
                                     metadata in one copy; out a page-locked host buffer */
  int32_t num_layers;          /* layers sharing the block tables (0 or 1: one) */
  int64_t cache_layer_stride;  /* elements between consecutive layers' caches (num_layers > 1) */
  int32_t cache_fp8;           /* 1: k_cache/v_cache hold E4M3 codes with the scales below; each step
                                  runs paged_decode_step_fp8 per layer (copy-on-write copies are
                                  not supported) */
  float* k_scales;             /* fp8 only: [num_blocks, num_kv_heads, block_size] per layer, */
  float* v_scales;             /*   layers back to back */
} kvstep_config_t;

/* Create a runner over manager mgr (not owned; it must outlive the runner)
 * with the sizes, caches and workspace of cfg (caller-owned device memory).
 * The runner owns its page-locked and device metadata buffers, side
 * streams and events.  KV_ERR_INVALID_ARG for inconsistent sizes or a
 * missing cache; KV_ERR_CUDA if an allocation fails.  The ModelRunner of
 * "从零实现一个 mini vLLM: Block Manager" (above). */
int kvstep_create(kvbm_t mgr, const kvstep_config_t* cfg, kvstep_t* out);

/* Wait for the runner's outstanding work, then release it (no passage: C
 * ABI lifetime). */
int kvstep_destroy(kvstep_t h);

/* One step.  q [num_seqs, num_heads, head_dim], k and v dense
 * [num_step_tokens, num_kv_heads, head_dim], out like q (with num_layers
 * layers, each of the four is that many such tensors back to back, and the
 * step's metadata, built and copied once, serves one fused launch per
 * layer over that layer's cache): device buffers
 * (host_io = 0; read and written in cfg.stream order), page-locked host
 * buffers (host_io = 1; q/k/v are read by the copy issued here, out is
 * written when the step's device-to-host copy completes, see kvstep_join),
 * or, with host_io = 2, q/k/v NULL (the inputs were staged with
 * kvstep_stage_buffer) and out a page-locked host buffer as for host_io = 1.
 * The id arguments are those of kvbm_prepare_step; n_decode must equal
 * cfg.num_seqs, the pads must be strictly increasing and in range, and the
 * step's rows must add up to cfg.num_step_tokens (else KV_ERR_INVALID_ARG,
 * nothing done).  Copies queued on the manager before the call (by appends
 * made outside the runner) must have been taken and applied by the caller:
 * if any are pending the call returns KV_ERR_INVALID_ARG and does nothing.
 * Manager errors are those of kvbm_prepare_step; nothing is launched then. */
int kvstep_run(kvstep_t h, const void* q, const void* k, const void* v, void* out,
               const int64_t* free_ids, int64_t n_free, const int64_t* prefill_ids,
               const int64_t* prefill_lens, int64_t n_prefill, const int64_t* decode_ids,
               int64_t n_decode, const int64_t* pad_positions, int64_t n_pad);

/* host_io = 2: page-locked host addresses where a step's q, k and v are to
 * be written (layouts as for kvstep_run; 256-byte aligned).  The runner
 * rotates four such slots, one per step in turn.  slot = -1: the slot the
 * next kvstep_run copies from, after waiting for the copy that last read
 * it; the caller writes its inputs there, then calls kvstep_run with q, k
 * and v NULL.  slot = 0..3: that slot, without waiting (for filling slots
 * before any step; the caller must not write a slot whose copy may still be
 * running).  slot_out (nullable) receives the slot index.  Any pointer
 * output may be NULL.  KV_ERR_INVALID_ARG for another host_io mode or a
 * slot out of range. */
int kvstep_stage_buffer(kvstep_t h, int32_t slot, void** q, void** k, void** v, int32_t* slot_out);

/* Make `stream` wait for every copy and kernel the runner has issued (an
 * event wait; nothing blocks the host).  No passage: stream ordering of
 * the step runner above. */
int kvstep_join(kvstep_t h, void* stream);

/* Host copies of the last step's metadata (valid until the next
 * kvstep_run): slot mapping, block tables, seq_lens and the decode rows,
 * the ModelRunner's inputs of "从零实现一个 mini vLLM: Block Manager"; for
 * inspection and tests.  Any output may be NULL. */
int kvstep_last_buffers(kvstep_t h, const int32_t** slot_mapping, const int32_t** block_tables,
                        const int32_t** seq_lens, const int32_t** new_token_row);

/* Test controls of the stream-K decode kernel, process-wide, read at each
 * later launch (no counterpart on the pages).  Keys:
 *   KV_DEBUG_WAIT_LIMIT_NS: longest one bounded device wait may take before
 *     the kernel records KV_ERR_DEVICE_TIMEOUT and gives up (value <= 0
 *     restores the default, 1 s).
 *   KV_DEBUG_SKIP_TILE: value >= 0: CTA 0 of each later launch never loads
 *     tile number `value` of its range (counted from 0), so the wait for it
 *     runs out after the wait limit; the launch still ends, records
 *     KV_ERR_DEVICE_TIMEOUT, and its outputs are unspecified.  value < 0:
 *     off.  For tests of the timeout path, which need no GPU fault.
 * KV_ERR_INVALID_ARG for an unknown key. */
enum { KV_DEBUG_WAIT_LIMIT_NS = 1, KV_DEBUG_SKIP_TILE = 2 };
int kv_debug_set(int key, int64_t value);

/* Library version string (static; no passage). */
const char* kv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */

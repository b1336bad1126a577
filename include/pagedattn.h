/*
 * pagedattn.h -- C ABI of libpagedattn.so: paged KV-cache decode attention
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation is single-query decode attention over a KV cache kept in
 * fixed-size physical blocks that a per-sequence block table addresses
 * ("Paged Attention > The PagedAttention Algorithm", Standard Attention vs
 * PagedAttention: softmax(q K^T / sqrt(d_k)) V, with K and V gathered through
 * the block table; "PagedAttention by hand", Forward pass, Steps 2-4). The
 * result equals standard attention over the sequence's tokens in logical
 * order.
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument is DEVICE memory owned by the caller, unless the
 *     parameter says otherwise. The library allocates nothing. Its state is a
 *     thread-local error string, two device-resident counters (rejected
 *     indices, see pa_bad_index_count; waits that gave up, see
 *     pa_wait_timeout_count), a host-side note of which leading bytes of each
 *     recently used split-K workspace are zero (see
 *     pa_decode_workspace_bytes), and the fixed scratch of pa_decode_no_alloc.
 *   - Work is enqueued on `stream` and returns without synchronising. Inputs
 *     must stay valid until the stream reaches the work.
 *   - A negative return value means the call enqueued nothing (or, for
 *     PA_ERR_CUDA, that a launch failed); pa_last_error() then describes it.
 *   - 16-bit elements are IEEE fp16 or bfloat16 (`pa_dtype`), row-major.
 *   - Every tensor pointer must be 16-byte aligned.
 *
 * Layouts (S = num_seqs, Hq / Hkv = query / kv heads, d = head_dim,
 * B = block_size, NB = num_blocks, MB = max_blocks_per_seq):
 *   query, out          [S, Hq, d]       (out: dtype or fp32, see pa_decode)
 *   key_cache,
 *   value_cache         [NB, B, Hkv, d]   (the physical block pool)
 *   block_tables        [S, MB] int32     (physical block ids)
 *   seq_lens            [S] int32
 *   key, value (new)    [T, Hkv, d]
 *   slot_mapping        [T] int64         (physical block * B + offset)
 * Query head hq reads kv head hq / (Hq / Hkv) (contiguous groups).
 */
#ifndef PAGEDATTN_H_
#define PAGEDATTN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_FLOAT16 = 0, PA_BFLOAT16 = 1, PA_FLOAT32 = 2 } pa_dtype;

enum {
  PA_OK = 0,
  PA_ERR_INVALID = -1,     /* a null pointer, a bad size or a misaligned pointer */
  PA_ERR_UNSUPPORTED = -2, /* valid, but outside what the kernels are built for */
  PA_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required */
  PA_ERR_CUDA = -4,        /* a CUDA call failed; the message names it */
  PA_ERR_CAPACITY = -5     /* the block pool or a block table is full (nothing changed) */
};

/*
 * Cache write: for every token i < num_tokens with slot = slot_mapping[i] >= 0,
 * copy the rows key[i, :, :] and value[i, :, :] ([Hkv, d] each) into
 * key_cache[slot / B, slot % B, :, :] and value_cache[...] bit for bit.
 * A negative slot skips token i. This is the write vLLM performs for the new
 * token before the attention kernel runs ("PagedAttention by hand", Setup,
 * Step 1, and the Code section); the slot of logical token t of a sequence is
 * table[t / B] * B + t % B ("The PagedAttention Algorithm", opening: a
 * logical token maps to an offset inside a numbered physical block).
 *
 * Sizes: num_tokens >= 0 (0 is a no-op), num_kv_heads >= 1, head_dim in
 * {64, 128}, block_size a power of two in [1, 64], num_blocks >= 1.
 * A slot >= num_blocks * block_size is not written and is counted by
 * pa_bad_index_count. Two tokens with the same slot race (one of them wins).
 * Errors: PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA.
 */
int pa_reshape_and_cache(const void* key, const void* value,
                         void* key_cache, void* value_cache,
                         const int64_t* slot_mapping, int num_tokens,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         pa_dtype dtype, cudaStream_t stream);

/*
 * Workspace bytes pa_decode needs for these sizes (0 when one partition
 * covers the longest possible sequence, max_blocks_per_seq * block_size).
 * partition_tokens is the value that will be passed to pa_decode (0 = the
 * library's default, see pa_decode). Returns 0 for invalid sizes.
 *
 * Workspace contents: per-(sequence, kv-head) arrival counters at the start,
 * followed by fp32 partial results. Zero-fill a new workspace once, at
 * allocation. Every pa_decode leaves the counters it used at zero. When a
 * later call's counters reach into bytes an earlier call on the same
 * workspace used for partial results (more sequences or heads, or other
 * sizes), pa_decode clears its counter region itself, with one
 * cudaMemsetAsync on the call's stream; the library tracks this per workspace
 * address, so distinct workspaces must not overlap in memory. A call captured
 * in a CUDA graph replays without that check: between replays, use its
 * workspace only with the captured sizes (or zero it again). Calls that share
 * a workspace must not overlap on the GPU.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size,
                                 int partition_tokens);

/*
 * The split-K partition length pa_decode uses for these arguments: the
 * default for partition_tokens = 0 (see pa_decode), else partition_tokens
 * itself. Host-only. Returns PA_ERR_INVALID or PA_ERR_UNSUPPORTED (negative)
 * where pa_decode would reject the value, with pa_last_error set.
 */
int pa_decode_partition_tokens(int partition_tokens, int block_size, int max_blocks_per_seq);

/*
 * Decode attention. For every sequence s and query head hq, with
 * h = hq / (Hq / Hkv) and L = seq_lens[s]:
 *   score_t = scale * <query[s, hq, :], K_t>,        t = 0 .. L-1
 *   out[s, hq, :] = sum_t softmax(score)_t * V_t
 * where K_t / V_t = key_cache / value_cache[block_tables[s, t / B], t % B, h, :].
 * Slots at or past L and table entries at or past ceil(L / B) are never read.
 * L = 0 gives a zero output row. Arithmetic is fp32: q.K takes the 16-bit
 * inputs with fp32 accumulation; each softmax weight enters P.V as the sum of
 * two 16-bit (dtype) parts (its rounding and the rounding of the remainder),
 * again with fp32 accumulation.
 *
 * dtype (PA_FLOAT16 or PA_BFLOAT16) is the type of query and the caches.
 * out_dtype is either dtype (out is rounded to it, nearest even) or
 * PA_FLOAT32 (out holds the fp32 result before that rounding; the 16-bit
 * output of the same call is exactly its nearest-even rounding).
 *
 * The first twelve parameters follow the statement of the problem; the rest
 * give the table's row stride (max_blocks_per_seq), the pool size for index
 * checks (num_blocks), the split-K partition length, the element types, the
 * scratch space and the stream.
 *
 * Split-K: each sequence is cut into partitions of partition_tokens tokens
 * (0 = the default: 1024 when max_blocks_per_seq * block_size >= 4096, else
 * 512; otherwise a multiple of 16 and of block_size, at most 2^20). The
 * kernel is persistent (a few CTAs per SM); each CTA takes a contiguous,
 * token-balanced run of the rows' leading partitions and continues the
 * online softmax across consecutive partitions of one (sequence, kv head);
 * a share of each row's trailing partitions, fixed by the row's length
 * alone, is claimed at run time from a counter in the workspace. Where a
 * row is split into pieces, the pieces are numbered by the data alone and
 * combined by log-sum-exp in piece order inside the same launch, so the call
 * is a single kernel and its result does not depend on which CTA computed
 * which piece.
 * `workspace` must hold pa_decode_workspace_bytes(...) bytes (it may be NULL
 * when that is 0); see there for the zeroing rule.
 *
 * Sizes: num_seqs >= 0 (0 is a no-op) and <= 65535, num_kv_heads in
 * [1, 65535], num_q_heads a multiple of num_kv_heads with at most 16 query
 * heads per kv head, head_dim in {64, 128}, block_size a power of two in
 * [1, 64], max_blocks_per_seq >= 1, num_blocks >= 1 with num_blocks *
 * block_size below 2^32 - 1 slots (PA_ERR_UNSUPPORTED otherwise; such a pool
 * would not fit in one GPU's memory), scale finite.
 * A seq_len above max_blocks_per_seq * block_size is clamped to it, and a
 * block id outside [0, num_blocks) reads as zeros; both are counted by
 * pa_bad_index_count and never fault.
 * Errors: PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA.
 */
int pa_decode(void* out, const void* query,
              const void* key_cache, const void* value_cache,
              const int32_t* block_tables, const int32_t* seq_lens,
              int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
              int block_size, float scale,
              int max_blocks_per_seq, int num_blocks, int partition_tokens,
              pa_dtype dtype, pa_dtype out_dtype, void* workspace, size_t workspace_bytes,
              cudaStream_t stream);

/*
 * The decode step's cache write and attention in one kernel ("PagedAttention
 * by hand", Setup, Step 1: the newest token's key and value are in the cache
 * before attention runs). For every sequence s with L = seq_lens[s] >= 1 and
 * every kv head h, the row new_key[s, h, :] (new_value likewise) is token
 * L-1's K (V): the kernel uses it for that token and stores it into its slot
 * key_cache[block_tables[s, (L-1) / B], (L-1) % B, h, :]. The result and the
 * caches afterwards are those of pa_reshape_and_cache (slot of token L-1 of
 * each sequence) followed by pa_decode. new_key, new_value: DEVICE
 * [S, Hkv, d], 16-byte aligned. The block holding token L-1 must belong to
 * sequence s alone (resolve copy-on-write first, e.g. with pa_bm_append and
 * pa_copy_blocks). Other arguments, sizes and errors as for pa_decode.
 */
int pa_decode_append(void* out, const void* query, const void* new_key, const void* new_value,
                     void* key_cache, void* value_cache,
                     const int32_t* block_tables, const int32_t* seq_lens,
                     int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                     int block_size, float scale,
                     int max_blocks_per_seq, int num_blocks, int partition_tokens,
                     pa_dtype dtype, pa_dtype out_dtype, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/*
 * pa_decode without a caller-provided workspace, for callers that cannot
 * allocate device memory: for example a plugin inside a host runtime that owns
 * every device allocation, or a serving loop that forbids allocation after
 * start-up (cudaMalloc can synchronise the device and can fail under memory
 * pressure). The pages describe no such entry point; it has no counterpart
 * there.
 *
 * Arguments, results and errors are those of pa_decode, without `workspace`
 * and `workspace_bytes`. The split-K scratch is a fixed array of
 * pa_decode_no_alloc_scratch_bytes() bytes (64 MiB) that the library keeps in
 * device memory; every GPU that loads the library holds it until the process
 * exits. Sizes whose pa_decode_workspace_bytes(...) exceed it are rejected
 * with PA_ERR_WORKSPACE.
 *
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * Its first call on a device (with that device current) looks up the array's
 * device address with cudaGetSymbolAddress and caches it; make that first call
 * before any stream capture. Each call clears the scratch's arrival counters
 * with cudaMemsetAsync on `stream`, then runs pa_decode on it.
 *
 * All calls on a device share the one array, which keeps the previous call's
 * contents: calls that can overlap on the GPU (other streams, other threads)
 * race on it and give wrong results. Serialise them.
 */
int pa_decode_no_alloc(void* out, const void* query,
                       const void* key_cache, const void* value_cache,
                       const int32_t* block_tables, const int32_t* seq_lens,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, float scale,
                       int max_blocks_per_seq, int num_blocks, int partition_tokens,
                       pa_dtype dtype, pa_dtype out_dtype, cudaStream_t stream);

/* Size in bytes of the fixed scratch that pa_decode_no_alloc uses. */
size_t pa_decode_no_alloc_scratch_bytes(void);

/*
 * Paged causal prefill (chunked prefill). Sequence s has L = seq_lens[s]
 * tokens in the cache, the last Q_s of which are new (their K/V already
 * written, e.g. with pa_reshape_and_cache); their queries are the rows
 * query_start[s] .. query_start[s+1]-1 of `query`. Query j sits at position
 * L - Q_s + j and attends to tokens 0 .. L - Q_s + j ("PagedAttention"
 * glossary, How It Works: the blockwise formula with query index i, read
 * token by token):
 *   out[query_start[s] + j, hq, :] = sum_{t <= L-Q_s+j} softmax(scale q.K_t)_t V_t
 * with K_t / V_t read through the block table as in pa_decode.
 * query, out: [total_q, Hq, d] (out: dtype or fp32); query_start: DEVICE int32
 * [num_seqs + 1], non-decreasing, query_start[0] = 0; max_query_len: HOST
 * upper bound of Q_s (sizes the grid). A Q_s above L or a length above
 * max_blocks_per_seq * block_size is clamped and counted by
 * pa_bad_index_count. Other sizes and errors as for pa_decode.
 * Runs on the tcgen05 tensor cores (whole blocks of 8..64 tokens copied by
 * TMA, smaller blocks row by row). num_blocks * block_size must be below 2^31
 * (PA_ERR_UNSUPPORTED otherwise).
 * Arithmetic: q.K in the input type with fp32 accumulation. fp16 caches,
 * and bf16 caches given a workspace: every softmax weight enters P.V rounded
 * to fp16, in one product with fp16 V and fp32 accumulation, and each row's
 * sum of weights adds exactly those rounded weights, so a weight's rounding
 * error largely cancels between the weighted sum and the sum (the result is
 * off by at most about 2^-11 * max_t |V_t - out| from that rounding). For
 * bf16 the call first converts the value rows of every sequence to an fp16
 * copy in the workspace (a second kernel on `stream`; a value beyond fp16's
 * range, +-65504, becomes +-inf there). bf16 without a workspace (NULL):
 * every weight enters as the sum of two bf16 parts (its upper half and the
 * rounding of the remainder, relative error below 2^-16), two products, and
 * no copy is made.
 * workspace: DEVICE, 16-byte aligned, pa_prefill_workspace_bytes(...) bytes
 * (contents need no initialisation; calls sharing it must not overlap on the
 * GPU), or NULL. It is ignored when that size is 0 (fp16 caches).
 */
int pa_prefill(void* out, const void* query, const void* key_cache, const void* value_cache,
               const int32_t* block_tables, const int32_t* seq_lens, const int32_t* query_start,
               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
               float scale, int max_blocks_per_seq, int num_blocks, int max_query_len,
               pa_dtype dtype, pa_dtype out_dtype, void* workspace, size_t workspace_bytes,
               cudaStream_t stream);

/*
 * Workspace bytes pa_prefill can use with bf16 caches: an fp16 copy of the
 * value rows, num_seqs * max_blocks_per_seq * block_size * num_kv_heads *
 * head_dim * 2 bytes (rounded up to 256). 0 for fp16 caches, for invalid
 * sizes, and when the copy would have 2^31 slots or more (then pa_prefill
 * runs without it).
 */
size_t pa_prefill_workspace_bytes(int num_seqs, int num_kv_heads, int head_dim,
                                  int max_blocks_per_seq, int block_size, pa_dtype dtype);

/*
 * Block copies inside the pools, the device half of copy-on-write
 * ("PagedAttention by hand", Why divide memory into physical blocks?:
 * allocate a fresh block, copy that one block's contents, write into the
 * copy). For i < num_copies, the whole block src[i] (B * Hkv * d elements)
 * of key_cache and of value_cache is copied onto block dst[i].
 * src, dst: DEVICE int32 arrays of num_copies block ids. A pair with an id
 * outside [0, num_blocks) is skipped and counted by pa_bad_index_count;
 * src == dst is a no-op. Copies whose blocks overlap (a dst that is another
 * pair's src) race. Sizes as for pa_reshape_and_cache.
 * Errors: PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA.
 */
int pa_copy_blocks(void* key_cache, void* value_cache,
                   const int32_t* src, const int32_t* dst, int num_copies,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   pa_dtype dtype, cudaStream_t stream);

/*
 * Block manager: host-side bookkeeping of the pool ("PagedAttention by hand",
 * What is PagedAttention: free blocks are a stack of interchangeable ids, a
 * block table maps each sequence's logical blocks to physical ones; Why divide
 * memory into physical blocks?: reference counts and copy-on-write; the
 * "PagedAttention" glossary: a new block only when the previous one fills).
 * Every pointer here is HOST memory. Not thread-safe: serialise the calls on
 * one manager. Free-stack order: block 0 is handed out first on a fresh pool;
 * a freed sequence pushes its blocks in table order and allocation pops the
 * most recently pushed. Errors: PA_ERR_INVALID (bad id, NULL, duplicates,
 * capacities), PA_ERR_CAPACITY (pool or table full; nothing changed).
 */
typedef struct pa_block_manager pa_block_manager;

/* A manager of num_blocks blocks of block_size slots; tables hold at most
 * max_blocks_per_seq blocks. *out receives the handle. */
int pa_bm_create(int num_blocks, int block_size, int max_blocks_per_seq, pa_block_manager** out);
void pa_bm_destroy(pa_block_manager* bm);

/* A new, empty sequence; its id is written to *seq_id (freed ids are reused). */
int pa_bm_new_sequence(pa_block_manager* bm, int* seq_id);

/* A new sequence sharing all blocks of `parent` (their reference counts + 1),
 * e.g. one more sample of the same prompt. */
int pa_bm_fork(pa_block_manager* bm, int parent, int* child);

/* Drops the sequence: blocks whose reference count reaches 0 become free. */
int pa_bm_free_sequence(pa_block_manager* bm, int seq_id);

/*
 * Reserves slots for num_new[i] new tokens of sequence seq_ids[i], for
 * i < count, in order (a sequence appears at most once). Writes the slot of
 * every new token (block * block_size + offset), in request order, to
 * slot_mapping (room for slot_capacity entries), and the copy-on-write block
 * copies the writes need to copy_src / copy_dst (room for copy_capacity >=
 * count pairs; at most one per sequence), their number to *num_copies. The
 * caller performs those copies (pa_copy_blocks) before writing the tokens
 * (pa_reshape_and_cache with this slot_mapping).
 */
int pa_bm_append(pa_block_manager* bm, const int* seq_ids, const int* num_new, int count,
                 int64_t* slot_mapping, int slot_capacity,
                 int32_t* copy_src, int32_t* copy_dst, int copy_capacity, int* num_copies);

/* Block tables [count, max_blocks_per_seq] (unused entries 0) and lengths
 * [count] of the listed sequences, ready to upload for pa_decode. */
int pa_bm_block_tables(const pa_block_manager* bm, const int* seq_ids, int count,
                       int32_t* block_tables, int32_t* seq_lens);

int pa_bm_num_free_blocks(const pa_block_manager* bm, int* n);
int pa_bm_ref_count(const pa_block_manager* bm, int block, int* count);

/*
 * Message for the most recent non-OK return on the calling thread ("" if
 * none). The pointer stays valid until the next library call on that thread.
 */
const char* pa_last_error(void);

/*
 * Number of out-of-range indices (block ids, slots, sequence lengths) the
 * kernels on the CURRENT device have skipped or clamped since the counter was
 * last cleared. Synchronises the device. Writes the count to *count (a host
 * pointer); clears the counter when `clear` is non-zero.
 * Errors: PA_ERR_INVALID (count is NULL), PA_ERR_CUDA.
 */
int pa_bad_index_count(unsigned long long* count, int clear);

/*
 * Number of bounded waits inside the kernels on the CURRENT device that gave
 * up since the counter was last cleared. The tensor-core prefill kernel's
 * warps wait on each other through shared-memory barriers; every such wait
 * has a limit of about one second, after which the kernel counts it here and
 * winds down instead of hanging (its output is then invalid). Always 0 in
 * correct operation. Synchronises the device; *count is a host pointer;
 * clears the counter when `clear` is non-zero.
 * Errors: PA_ERR_INVALID (count is NULL), PA_ERR_CUDA.
 */
int pa_wait_timeout_count(unsigned long long* count, int clear);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H_ */

/*
 * pa.h -- C ABI of libpa.so, a GB300 (sm_103a) paged KV cache with
 * PagedAttention decode.
 *
 * The KV cache of every sequence lives in fixed-size physical blocks of B
 * token slots, scattered over one shared pool and reached through the
 * sequence's block table: token position pos is stored at offset pos % B of
 * physical block table[pos / B].  ("PagedAttention: Virtual Memory for the KV
 * Cache", section "A block table preserves token order"; "Paged Attention and
 * vLLM", section "Block Table and Logical-to-Physical Mapping".)
 *
 * Conventions for every call below
 * --------------------------------
 *  - Device pointers are owned by the caller (for instance torch tensors),
 *    row-major and contiguous, and must be 16-byte aligned.  The GPU entry
 *    points allocate no device memory; the split-K scratch of pa_decode is
 *    passed in as `workspace`.
 *  - GPU calls work on the calling thread's current device: every device
 *    pointer and the stream of a call must belong to it (the per-device error
 *    word, fixed scratch and cached tensor maps are the current device's).
 *  - GPU calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream).  The returned status covers only
 *    what the host can check (dimensions, dtypes, alignment, supported
 *    shapes, launch errors).
 *  - Bad indices met on the device (a block-table entry outside [0, N), a
 *    context length outside [0, max_blocks_per_seq * B], a slot >= N * B, a
 *    copy pair outside [0, N)) never fault: the offending item is skipped and
 *    a sticky bit is set in a per-device error word read by pa_device_errors.
 *  - Cache layout: k_cache and v_cache are each [N, Hkv, B, D] in kv_dtype;
 *    one (block, kv head) row set is B * D contiguous elements.
 *  - Supported shapes: head_dim D in {64, 128}; block_size B in {16, 32};
 *    group G = Hq / Hkv in {1, 2, 4, 8}; kv_dtype f32, f16 or bf16.  Other
 *    valid shapes return PA_ERR_UNSUPPORTED.
 *  - Host allocator calls (pa_pool_*, pa_seq_*) touch no GPU and are not
 *    thread-safe: one pool is used from one thread at a time.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID = 1,      /* bad argument: null or misaligned pointer, bad sizes */
    PA_ERR_UNSUPPORTED = 2,  /* valid but not compiled: D, B, G or dtype combination */
    PA_ERR_OOM = 3,          /* allocator: not enough free blocks; nothing changed */
    PA_ERR_BAD_INDEX = 4,    /* allocator: unknown sequence id or block id */
    PA_ERR_CUDA = 5,         /* a CUDA runtime call failed (no device, launch error) */
    PA_ERR_TOO_LARGE = 6     /* pa_decode_noalloc: the problem needs more scratch than */
                             /* the library's fixed buffer holds                      */
} pa_status;

typedef enum pa_dtype { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

/* Shapes shared by the GPU calls. */
typedef struct pa_dims {
    int32_t num_seqs;            /* S: sequences (one decode query each)             */
    int32_t num_q_heads;         /* Hq                                               */
    int32_t num_kv_heads;        /* Hkv; Hq % Hkv == 0, query head h reads KV head   */
                                 /*      h / (Hq / Hkv)                              */
    int32_t head_dim;            /* D                                                */
    int32_t block_size;          /* B: token slots per physical block                */
    int32_t num_blocks;          /* N: physical blocks in the pool                   */
    int32_t max_blocks_per_seq;  /* columns of block_tables                          */
    int32_t partition_size;      /* context tokens per split-K partition; a multiple */
                                 /* of B, at most 256 * B.  0 chooses by batch: with */
                                 /* W = num_seqs * num_kv_heads / 4 (work items per  */
                                 /* partition), 512 if W >= 256, 256 if W >= 32,     */
                                 /* else 128 (smaller partitions give a small batch  */
                                 /* enough parallel work); pa_chunk_attention takes  */
                                 /* four times that, at most 2048                    */
    int32_t kv_dtype;            /* pa_dtype of q, k, v, k_cache and v_cache         */
} pa_dims;

/* Bits of the per-device error word (see pa_device_errors). */
#define PA_DEVERR_BAD_BLOCK 1u   /* block-table entry outside [0, N): block skipped   */
#define PA_DEVERR_BAD_LEN 2u     /* context length < 0 or > max_blocks_per_seq * B:  */
                                 /* clamped into range                               */
#define PA_DEVERR_BAD_SLOT 4u    /* pa_write_kv slot >= N * B: token skipped          */
#define PA_DEVERR_BAD_PAIR 8u    /* pa_copy_blocks id outside [0, N): pair skipped    */
#define PA_DEVERR_TIMEOUT 16u    /* a bounded in-kernel wait gave up; outputs of the  */
                                 /* affected work item were not written              */

/* ------------------------------------------------------------------ GPU calls */

/*
 * pa_decode_workspace_bytes -- bytes of device scratch pa_decode needs: a
 * work list (S * P * 4 ints after a 256-byte header), plus, when one sequence
 * can span several partitions (P > 1), the split-K partials: S * Hq * P *
 * (D + 2) floats; P = ceil(max_blocks_per_seq * B / partition_size).  Each part
 * is rounded up to 256 bytes.  Returns 0 for S == 0 and for invalid dims.
 */
PA_API size_t pa_decode_workspace_bytes(const pa_dims *dims);

/*
 * pa_decode -- PagedAttention decode: for every sequence s and query head h,
 *
 *     out[s, h, :] = softmax(scale * q[s, h, :] . K_s^T) . V_s
 *
 * where K_s, V_s are the context_lens[s] keys/values of s read through its
 * block table, in token order, without building a contiguous copy.
 * ("Paged Attention and vLLM", "Block Table and Logical-to-Physical Mapping",
 * the a_t equation; section "Paged Attention CUDA Kernel" for the per-partition
 * (m_b, l_b, v_b^acc) terms and their log-sum-exp merge, used here as split-K
 * over context partitions of partition_size tokens.)
 *
 *   q             [S, Hq, D] kv_dtype, device
 *   k_cache,
 *   v_cache       [N, Hkv, B, D] kv_dtype, device
 *   block_tables  int32 [S, max_blocks_per_seq], device; entries past
 *                 ceil(context_lens[s] / B) are never read
 *   context_lens  int32 [S], device; 0 gives an all-zero output row
 *   scale         logit scale (1/sqrt(D) for standard attention)
 *   out           float32 [S, Hq, D], device, written
 *   workspace     device scratch of >= pa_decode_workspace_bytes(dims) bytes,
 *                 256-byte aligned; its contents need no initialisation (the
 *                 call resets what it uses) and are garbage afterwards;
 *                 concurrent calls need separate workspaces
 * Returns PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED or PA_ERR_CUDA.
 */
PA_API int32_t pa_decode(const pa_dims *dims, const void *q, const void *k_cache,
                  const void *v_cache, const int32_t *block_tables,
                  const int32_t *context_lens, float scale, float *out,
                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart to this call.
 *
 * Some callers cannot provide the split-K workspace: code running inside a
 * memory pool or arena that forbids further device allocations, plugin hosts
 * that own every allocation, or code paths where a cudaMalloc would
 * synchronise the device at a bad moment.  This call computes exactly what
 * pa_decode computes, with the same arguments except the workspace: its
 * scratch is a fixed buffer of PA_NOALLOC_SCRATCH_BYTES bytes built into the
 * library, held on every GPU that loads the library until the process exits.
 * It allocates nothing.
 *
 *  - The first call on each device looks up that buffer's device address
 *    (cudaGetSymbolAddress, with the device current) and caches it together
 *    with the id of the current CUDA context; make that first call before any
 *    stream capture on the device.  After a device reset the new context has
 *    a new id, and the next call looks the address up again.
 *  - Like every GPU call here, it works on the current device: the pointers
 *    and the stream must belong to it.
 *  - Returns PA_ERR_TOO_LARGE, doing nothing, when pa_decode_workspace_bytes
 *    (dims) exceeds PA_NOALLOC_SCRATCH_BYTES; use pa_decode with a workspace
 *    then.  Other statuses as for pa_decode.
 *  - All calls share the one buffer.  Calls whose GPU work overlaps (different
 *    streams, or different host threads, without ordering between them) race
 *    on it and give wrong results; order them on one stream.  Nothing carries
 *    over between calls: each call initialises what it reads.
 */
#define PA_NOALLOC_SCRATCH_BYTES (64u << 20) /* 64 MiB */
PA_API int32_t pa_decode_noalloc(const pa_dims *dims, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 const int32_t *context_lens, float scale, float *out, void *stream);

/*
 * pa_chunk_attention -- paged attention for several query tokens per sequence
 * (a prefill chunk, or drafted tokens being verified), over the same cache:
 * the n_s = query_start[s+1] - query_start[s] query rows of sequence s are its
 * last n_s positions, whose keys and values are already in the cache
 * (pa_write_kv), and the query at position pos = context_lens[s] - n_s + t
 * attends to positions 0 .. pos only:
 *
 *     out[i, h, :] = softmax(scale * q[i, h, :] . K_s[0..pos]^T) . V_s[0..pos],
 *     i = query_start[s] + t
 *
 * -- the result of decoding those tokens one at a time.  ("Paged Attention and
 * vLLM", "KV Cache Fundamentals": the cache of a sequence at length t holds
 * tokens 1..t; "Block Table and Logical-to-Physical Mapping" for the paged
 * read; "Paged Attention CUDA Kernel" for the per-partition terms and their
 * merge.  "KV Cache Optimization and Management", "Common misconception":
 * paging changes neither the scores nor the softmax.)
 *
 *   q             [T, Hq, D] kv_dtype, device; T = num_tokens
 *   query_start   int32 [S + 1], device: non-decreasing, query_start[0] >= 0,
 *                 query_start[S] <= T; rows outside every range are not written
 *   max_query_len an upper bound on every n_s (host-known; sizes the work split)
 *   out           float32 [T, Hq, D], device, written for the rows of valid
 *                 sequences
 *   other arguments as for pa_decode; kv_dtype must be PA_F16 or PA_BF16
 *                 (PA_ERR_UNSUPPORTED for PA_F32)
 * A sequence with n_s > context_lens[s] or n_s > max_query_len is skipped and
 * PA_DEVERR_BAD_LEN is set; a query_start that is not non-decreasing within
 * [0, T] skips every sequence and sets PA_DEVERR_BAD_LEN.
 *
 * Two kernels serve it: while max_query_len * Hq / Hkv (query rows per KV
 * head) is below 64, a persistent mma.sync kernel over context partitions
 * with a split-K merge; from 64 rows on, a persistent tcgen05 kernel with
 * 128-row tiles whose accumulators live in tensor memory, one CTA per SM
 * taking work items (tiles, KV head, sequence) longest first, each walking
 * its tiles' whole context (no partitions, no merge).
 *
 * pa_chunk_workspace_bytes -- the scratch it needs: a work list of S * P * R
 * int4 entries after a 256-byte header, T ints (the partitions each query
 * row sees), and, on the mma.sync path with P > 1, the split-K partials
 * T * Hq * P * (D + 2) floats, each part rounded up to 256 bytes; P as for
 * pa_decode, with the partition size chosen as for pa_chunk_attention,
 * R = ceil(ceil(max_query_len * Hq / Hkv / 16) / W), W = 2 if max_query_len *
 * Hq / Hkv > 16, else 1.  Returns 0 for invalid arguments.
 */
PA_API size_t pa_chunk_workspace_bytes(const pa_dims *dims, int32_t num_tokens, int32_t max_query_len);
PA_API int32_t pa_chunk_attention(const pa_dims *dims, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, const int32_t *query_start,
                                  int32_t num_tokens, int32_t max_query_len, float scale, float *out,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_write_kv -- the KV write (reshape-and-cache): store each new token's key
 * and value rows in its slot, for every KV head:
 *
 *     k_cache[slot / B, h, slot % B, :] = k[t, h, :]   (and the same for v)
 *
 * ("PagedAttention: Virtual Memory for the KV Cache", "Sharing a prefix and
 * copying a partial block": the engine writes the new entry into the block the
 * table now points at.)  The copy is bit-exact.
 *
 *   k, v          [num_tokens, Hkv, D] kv_dtype, device
 *   slot_mapping  int64 [num_tokens], device; slot = physical block * B +
 *                 offset; a negative slot skips the token (padding)
 *   k_cache,
 *   v_cache       [N, Hkv, B, D] kv_dtype, device, updated in place
 * Distinct tokens must have distinct slots.  Only num_kv_heads, head_dim,
 * block_size, num_blocks and kv_dtype of dims are used.
 */
PA_API int32_t pa_write_kv(const pa_dims *dims, const void *k, const void *v,
                    const int64_t *slot_mapping, int32_t num_tokens,
                    void *k_cache, void *v_cache, void *stream);

/*
 * pa_copy_blocks -- copy-on-write block copy: for each pair (src, dst) copy
 * the whole physical block src -> dst (all Hkv heads, all B slots, keys and
 * values), bit-exact.  ("PagedAttention: Virtual Memory for the KV Cache",
 * "Sharing a prefix and copying a partial block"; "Paged Attention and vLLM",
 * "Continuous Batching and Scheduler", the copy-on-write rule.)
 *
 *   src_dst_pairs  int64 [num_pairs, 2], device
 * Precondition: every dst is distinct and no dst is also a src (the allocator
 * only emits such pairs); otherwise the result is unspecified.  Only
 * num_kv_heads, head_dim, block_size, num_blocks and kv_dtype of dims are used.
 */
PA_API int32_t pa_copy_blocks(const pa_dims *dims, void *k_cache, void *v_cache,
                       const int64_t *src_dst_pairs, int32_t num_pairs, void *stream);

/*
 * pa_copy_blocks_layers -- pa_copy_blocks for num_layers caches at once: layer
 * l's caches start layer_stride_bytes * l after k_caches / v_caches (a
 * multi-layer pool [L, N, Hkv, B, D]; the block manager's ids are the same in
 * every layer).  layer_stride_bytes must be a multiple of 16 and at least one
 * pool (N * Hkv * B * D elements) when num_layers > 1.  One launch for all
 * layers, so num_layers is at most 32767 (PA_ERR_INVALID above).  Same
 * preconditions and errors as pa_copy_blocks.
 */
PA_API int32_t pa_copy_blocks_layers(const pa_dims *dims, void *k_caches, void *v_caches, int32_t num_layers,
                                     int64_t layer_stride_bytes, const int64_t *src_dst_pairs, int32_t num_pairs,
                                     void *stream);

/*
 * Step graph -- one decode step over num_layers layers, captured once into a
 * CUDA graph: for l = 0 .. L-1, pa_write_kv then pa_decode of layer l (the
 * decode work list, which depends only on the shared tables and lengths, is
 * built once per launch rather than per layer).  Every
 * pointer is a fixed device buffer read at each launch (update the buffers,
 * then launch); layer l uses
 *     k_caches + l * cache_layer_stride      (and v_caches)
 *     q        + l * q_layer_stride          [S, Hq, D]
 *     k_new    + l * kv_new_layer_stride     [num_tokens, Hkv, D] (and v_new)
 *     out      + l * out_layer_stride        [S, Hq, D] fp32
 * (strides in bytes; out_layer_stride a multiple of 16; with num_layers > 1
 * each stride at least one layer's tensor, so that layers do not overlap,
 * else PA_ERR_INVALID); slot_mapping, block_tables, context_lens and the
 * workspace are shared by all layers (layers run in order).  Arguments are
 * validated as by the two calls; on failure NULL is returned and *status
 * (nullable) holds the pa_status.  Copy-on-write copies, which are rare and
 * vary in number, are not in the graph: run pa_copy_blocks_layers first.
 * Launch with pa_step_graph_launch (asynchronous on `stream`); destroy with
 * pa_step_graph_destroy.  Creation must not overlap a capture on the calling
 * thread.
 */
typedef struct pa_step_graph pa_step_graph;
PA_API pa_step_graph *pa_step_graph_create(const pa_dims *dims, int32_t num_layers, void *k_caches,
                                           void *v_caches, int64_t cache_layer_stride, const void *q,
                                           int64_t q_layer_stride, const void *k_new, const void *v_new,
                                           int64_t kv_new_layer_stride, const int64_t *slot_mapping,
                                           int32_t num_tokens, const int32_t *block_tables,
                                           const int32_t *context_lens, float scale, float *out,
                                           int64_t out_layer_stride, void *workspace, size_t workspace_bytes,
                                           int32_t *status);
PA_API int32_t pa_step_graph_launch(pa_step_graph *graph, void *stream);
PA_API void pa_step_graph_destroy(pa_step_graph *graph);

/*
 * pa_swap_blocks -- block-granular swap between the device pools and a host
 * pool, for preempting a sequence (its blocks move to host memory, the device
 * blocks are reused) and resuming it later.  ("Paged Attention and vLLM",
 * "Continuous Batching and Scheduler": evict a sequence's physical blocks to
 * CPU, swap them back on resume, paying only for those blocks.)
 *
 *   host_k, host_v    [num_layers][num_host_blocks, Hkv, B, D] kv_dtype in host
 *                     memory the GPU can access directly (pinned or registered,
 *                     e.g. cudaHostAlloc); anything else gives PA_ERR_INVALID
 *   pairs             int64 [num_pairs, 2], device: PA_SWAP_OUT copies device
 *                     block pairs[i][0] to host block pairs[i][1]; PA_SWAP_IN
 *                     copies host block pairs[i][0] to device block pairs[i][1]
 *   strides           bytes between layers (used when num_layers > 1)
 *   num_layers        at most 32767 (PA_ERR_INVALID above)
 * One kernel moves every pair of every layer, K and V, with the GPU reading
 * and writing host memory directly; bit-exact.  Ids outside the pools are
 * skipped and flagged (PA_DEVERR_BAD_PAIR).  Destinations must be distinct.
 * pa_seq_swap_out / pa_seq_swap_in produce the pairs.
 */
#define PA_SWAP_OUT 0
#define PA_SWAP_IN 1
PA_API int32_t pa_swap_blocks(const pa_dims *dims, void *k_cache, void *v_cache, void *host_k, void *host_v,
                              int32_t num_host_blocks, int32_t num_layers, int64_t dev_layer_stride_bytes,
                              int64_t host_layer_stride_bytes, const int64_t *pairs, int32_t num_pairs,
                              int32_t direction, void *stream);

/*
 * pa_copy_to_device / pa_copy_to_host -- one asynchronous copy of `bytes`
 * bytes between host memory and device memory of the current device, on
 * `stream` (cudaMemcpyAsync).  The pages have no counterpart: this is the hop
 * a serving step makes to bring its inputs (queries, new K/V rows, slots,
 * block tables, lengths, copy pairs) to the GPU and its output back, offered
 * here so that a caller holding only host buffers needs nothing but this
 * library.  The copy overlaps kernels on other streams only when the host
 * buffer is pinned (page-locked, e.g. cudaHostAlloc); pageable memory makes
 * it synchronous.  bytes == 0 does nothing.  Returns PA_OK, PA_ERR_INVALID
 * (a null pointer with bytes > 0) or PA_ERR_CUDA.
 */
PA_API int32_t pa_copy_to_device(void *dst_device, const void *src_host, size_t bytes, void *stream);
PA_API int32_t pa_copy_to_host(void *dst_host, const void *src_device, size_t bytes, void *stream);

/*
 * pa_device_errors -- read (and, if clear != 0, reset) the sticky PA_DEVERR_*
 * bits of the current device.  Synchronises with the device.
 */
PA_API int32_t pa_device_errors(uint32_t *flags, int32_t clear);

/* Library version string, e.g. "pa 0.1.0 sm_103a". */
PA_API const char *pa_version(void);

/*
 * pa_selftest_bounded_wait -- a check of the kernels' failure path; the pages
 * have no counterpart.  Every wait of the library's kernels on an mbarrier
 * gives up after a bounded number of polls, records PA_DEVERR_TIMEOUT and
 * returns.  This runs that wait, `limit` polls (1 .. 2^20), on an mbarrier
 * nothing ever arrives at, in one kernel on `stream`, and writes the outcome
 * to *status (device uint32): PA_DEVERR_TIMEOUT when the wait gave up, 0 if
 * it was satisfied.  No fault and no hang: each poll is bounded in time by the
 * hardware.  Returns PA_OK, PA_ERR_INVALID (null status, limit out of range)
 * or PA_ERR_CUDA (launch error).
 */
PA_API int32_t pa_selftest_bounded_wait(uint32_t limit, uint32_t *status, void *stream);

/* ------------------------------------------------------- host block allocator
 *
 * A pool of N physical blocks of B slots with a FIFO free list, a reference
 * count per block, per-sequence block tables, prefix sharing by fork and
 * copy-on-write of a partially filled shared last block.  ("PagedAttention:
 * Virtual Memory for the KV Cache", sections "Growing a request" and "Sharing a
 * prefix and copying a partial block"; "KV Cache Optimization and Management",
 * "PagedAttention: borrowing virtual memory" and answer A6.)
 */
typedef struct pa_pool pa_pool;

typedef struct pa_pool_stats {
    int32_t num_blocks;
    int32_t block_size;
    int32_t free_blocks;
    int32_t used_blocks;      /* refcount >= 1                                   */
    int32_t shared_blocks;    /* refcount >= 2                                   */
    int32_t live_seqs;
    int64_t cow_copies;       /* copy-on-write pairs emitted since creation      */
    int64_t tokens;           /* sum of live sequence lengths                    */
    int64_t table_slots;      /* B * sum of live table lengths (per-seq view)    */
    int64_t padded_slots;     /* table_slots - tokens                            */
} pa_pool_stats;

/*
 * Create a pool of num_blocks blocks of block_size slots.  free_order (host,
 * nullable) is a permutation of 0..num_blocks-1 giving the order in which free
 * blocks are handed out; NULL means ascending ids.  Returns NULL on bad
 * arguments.  Destroy with pa_pool_destroy.
 */
PA_API pa_pool *pa_pool_create(int32_t num_blocks, int32_t block_size, const int32_t *free_order);
PA_API void pa_pool_destroy(pa_pool *pool);

/* New empty sequence; returns its id (>= 0; ids are never reused) or -PA_ERR_INVALID. */
PA_API int32_t pa_seq_create(pa_pool *pool);

/*
 * Fork: a new sequence sharing all of parent's blocks (each block's refcount
 * + 1) and its length.  Sharing is only valid when the prefix was computed
 * from the same model state, positions and inputs; the library does not check
 * that.  Returns the new id or -PA_ERR_BAD_INDEX.
 */
PA_API int32_t pa_seq_fork(pa_pool *pool, int32_t parent);

/*
 * Append n_tokens tokens to sequence seq and return their slots.
 *  - If the next token falls in a partially filled last block that is shared
 *    (refcount > 1), that block is first copied: a fresh block p' is taken,
 *    the pair (p, p') is written to cow_pairs_out[0..1], p's count drops by
 *    one and the table now points at p'.  *n_cow is set to 1, else 0.  The
 *    caller must run pa_copy_blocks on the pair before writing the new tokens.
 *    A full shared block is never copied: growth takes a new private block.
 *  - A new block is taken from the free list whenever a token starts a block.
 *  - slots_out[i] = table[pos / B] * B + pos % B for pos = len .. len+n-1.
 *  The call is atomic: when the blocks it needs (copy plus growth) are not all
 *  available it returns PA_ERR_OOM and changes nothing.  Within one call the
 *  copy block is taken before the growth blocks.
 *  slots_out: host int64[n_tokens] (may be NULL if n_tokens == 0);
 *  cow_pairs_out: host int64[2]; n_cow: host int32.
 */
PA_API int32_t pa_seq_append(pa_pool *pool, int32_t seq, int32_t n_tokens, int64_t *slots_out,
                      int64_t *cow_pairs_out, int32_t *n_cow);

/*
 * Batched append: append tokens_each tokens to each of n distinct sequences
 * seqs[0..n-1], in that order, with the same rules as pa_seq_append.
 * slots_out: int64[n * tokens_each] (row i for seqs[i]); cow_pairs_out:
 * int64[2 * n]; *n_cow receives the number of pairs written.  All-or-nothing:
 * PA_ERR_OOM leaves the pool unchanged.  Duplicate ids give PA_ERR_INVALID.
 */
PA_API int32_t pa_seq_append_batch(pa_pool *pool, const int32_t *seqs, int32_t n, int32_t tokens_each,
                            int64_t *slots_out, int64_t *cow_pairs_out, int32_t *n_cow);

/*
 * pa_copy_pairs_check -- host check of copy-on-write pairs before they go to
 * pa_copy_blocks, which reads its pairs on the device and cannot check them.
 * A copy-on-write copy goes to a fresh block ("PagedAttention: Virtual Memory
 * for the KV Cache", "Sharing a prefix and copying a partial block"), so a
 * valid list has every id in [0, num_blocks), no destination twice, and no
 * destination that is also a source (several pairs may share a source).
 *   pairs  host int64 [num_pairs, 2] (src, dst); may be NULL if num_pairs == 0
 * Returns PA_OK, PA_ERR_BAD_INDEX (an id out of range) or PA_ERR_INVALID (a
 * repeated destination, a destination that is a source, num_pairs < 0,
 * num_blocks <= 0, NULL pairs).  The pairs pa_seq_append and
 * pa_seq_append_batch emit always pass.
 */
PA_API int32_t pa_copy_pairs_check(const int64_t *pairs, int32_t num_pairs, int32_t num_blocks);

/* Release a sequence: each of its blocks' counts drops by one; blocks reaching
 * zero go to the back of the free list, in table order. */
PA_API int32_t pa_seq_free(pa_pool *pool, int32_t seq);

/* Copy up to cap table entries of seq into out; returns the table length or
 * -PA_ERR_BAD_INDEX. */
PA_API int32_t pa_seq_table(const pa_pool *pool, int32_t seq, int32_t *out, int32_t cap);

/* Length (stored tokens) of seq, or -PA_ERR_BAD_INDEX. */
PA_API int32_t pa_seq_len(const pa_pool *pool, int32_t seq);

/*
 * Export device-ready tables for n sequences: tables_out int32[n, max_blocks]
 * (row i = table of seqs[i], padded with `pad`) and lens_out int32[n].
 * PA_ERR_INVALID if a table is longer than max_blocks.
 */
PA_API int32_t pa_pool_export(const pa_pool *pool, const int32_t *seqs, int32_t n, int32_t max_blocks,
                       int32_t pad, int32_t *tables_out, int32_t *lens_out);

PA_API int32_t pa_pool_num_free(const pa_pool *pool);
PA_API int32_t pa_block_refcount(const pa_pool *pool, int32_t block);   /* -PA_ERR_BAD_INDEX if bad id */
PA_API int32_t pa_pool_get_stats(const pa_pool *pool, pa_pool_stats *out);

/*
 * Swap a sequence out of the device pool `dev` into the host-slot pool `host`
 * (a second pa_pool of the same block size whose block ids index the host
 * KV pool).  Every block of the sequence gets a private host block (shared
 * prefix blocks are duplicated on the host, not shared there); the pairs
 * (device block, host block) are written to pairs_out[2 * n] in table order;
 * the device sequence is then freed (blocks other sequences still use stay).
 * *host_seq receives the sequence's id in `host`.  Run pa_swap_blocks
 * (PA_SWAP_OUT) on the pairs before any kernel writes to a freed device block.
 * All-or-nothing: PA_ERR_OOM if the host pool is short, nothing changed.
 */
PA_API int32_t pa_seq_swap_out(pa_pool *dev, pa_pool *host, int32_t seq, int32_t *host_seq, int64_t *pairs_out,
                               int32_t *n_pairs);

/*
 * Swap a host sequence back in: fresh private device blocks, pairs (host
 * block, device block) in table order, the host sequence freed; *dev_seq gets
 * the new device id.  Run pa_swap_blocks (PA_SWAP_IN) before the sequence's
 * next decode.  All-or-nothing: PA_ERR_OOM if the device pool is short.
 */
PA_API int32_t pa_seq_swap_in(pa_pool *dev, pa_pool *host, int32_t host_seq, int32_t *dev_seq, int64_t *pairs_out,
                              int32_t *n_pairs);

/* ------------------------------------------------------- prefix cache
 *
 * A radix tree of cached token sequences over the pool's blocks, for reusing
 * the K/V of shared prompt prefixes across requests.  ("KV Cache Optimization
 * and Management", "RadixAttention: caching, not just packing, the prefix":
 * match a new request's tokens against the tree, reuse every matched token's
 * blocks, evict least-recently-used leaves when memory runs low, and let
 * reference counts protect what running requests still use.)  Only whole
 * blocks are cached and reused.  The cache holds one pool reference on every
 * block it keeps.  Exact rules:
 *  - pa_prefix_match returns the blocks of the longest cached block-aligned
 *    prefix of tokens (writing at most cap of them; the return value is the
 *    full count) and marks them as just used;
 *  - pa_prefix_insert caches the first min(n_blocks, n_tokens / B) blocks of a
 *    sequence under its tokens; prefixes already cached keep their blocks; the
 *    return value counts newly cached blocks.  A block is cached under one
 *    prefix at most: if a block to be newly cached is cached already, or occurs
 *    twice among them, it returns -PA_ERR_INVALID and changes nothing; a block
 *    id out of range or not allocated gives -PA_ERR_BAD_INDEX;
 *  - pa_prefix_evict drops, one block at a time, a cached prefix with no cached
 *    extension whose block no sequence uses (pool refcount 1), least recently
 *    used first (ties: lower block id), until n_blocks blocks have been freed
 *    or nothing qualifies; returns the number freed.
 * Token ids are int32.  Negative returns are -pa_status.
 */
typedef struct pa_prefix_cache pa_prefix_cache;
PA_API pa_prefix_cache *pa_prefix_cache_create(pa_pool *pool);
PA_API void pa_prefix_cache_destroy(pa_prefix_cache *cache);  /* drops its block references */
PA_API int32_t pa_prefix_match(pa_prefix_cache *cache, const int32_t *tokens, int32_t n_tokens,
                               int32_t *blocks_out, int32_t cap);
PA_API int32_t pa_prefix_insert(pa_prefix_cache *cache, const int32_t *tokens, int32_t n_tokens,
                                const int32_t *blocks, int32_t n_blocks);
PA_API int32_t pa_prefix_evict(pa_prefix_cache *cache, int32_t n_blocks);
PA_API int32_t pa_prefix_cached_blocks(const pa_prefix_cache *cache);

/*
 * A new sequence whose table starts with n_blocks existing blocks (each gains
 * a reference; e.g. the blocks pa_prefix_match returned) and whose length is
 * n_blocks * B; append the rest of its tokens with pa_seq_append.  Returns the
 * id or -pa_status.
 */
PA_API int32_t pa_seq_create_from_prefix(pa_pool *pool, const int32_t *blocks, int32_t n_blocks);

/*
 * Fault injection for tests: let only n more block allocations succeed; any
 * operation needing more fails with PA_ERR_OOM and changes nothing.  n < 0
 * removes the limit.
 */
PA_API int32_t pa_pool_set_fail_after(pa_pool *pool, int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */

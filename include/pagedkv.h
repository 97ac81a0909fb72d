/*
 * pagedkv.h — C ABI of libpagedkv.so: paged KV-cache attention for sm_103a.
 *
 * The cache is a pool of fixed-size physical blocks.  A sequence reaches its
 * tokens through a block table: the token at logical position p lives in
 * physical block table[p / B_p] at offset p mod B_p, i.e. at slot
 * table[p / B_p] * B_p + p mod B_p.
 *
 * Sources (page title, section) cited below:
 *   P1 = "03｜PagedAttention 与 KV Cache 内存系统" (llm-infra-atlas.github.io)
 *   P2 = "KV Cache：容量、布局与生命周期" (wineandchord.com)
 *   P3 = "PagedAttention 的原理是什么？它如何降低 KV Cache 的内存浪费？" (offer.aigcbaba.com)
 *   P4 = "vLLM学习笔记-显存管理之PagedAttention" (amentiraz.github.io)
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns every buffer.  Device pointers must stay valid
 *    until the work enqueued on `stream` has finished.  Nothing here allocates
 *    device memory at run time; scratch space is passed in (pa_decode's
 *    workspace), except for pa_decode_noalloc, whose scratch is a 16 MiB
 *    static array in the library's device image.
 *  - Asynchrony: device entry points only enqueue kernels on `stream` (NULL =
 *    the legacy default stream) and return; there is no internal sync.
 *    Ordering between calls (copy-on-write copy before the write that follows
 *    it, P2 "引用计数与尾块 COW") is the caller's stream order.
 *  - Errors: argument errors found on the host are returned at once and
 *    nothing is enqueued.  Data-dependent errors found on the device (a slot
 *    or block id outside the pool, a negative id) skip the offending row or
 *    page and store the first error code into *d_err (a device int32 the
 *    caller zeroes and reads after synchronising; NULL disables reporting).
 *    The kernels never trap or assert.  A bounded device-side wait that runs
 *    out stores PA_ERR_TIMEOUT.
 *  - Launch failures are returned as PA_ERR_CUDA (cudaGetLastError after the
 *    launch); the CUDA error string is available from pa_last_cuda_error().
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,    /* bad size, shape, dtype, null pointer, block size <= 0, pos < 0 */
    PA_ERR_OUT_OF_RANGE = 2,   /* logical block not allocated; slot or block id outside the pool */
    PA_ERR_NEGATIVE_BLOCK = 3, /* a block table names a negative physical id */
    PA_ERR_NO_FREE_BLOCK = 4,  /* allocator: free list empty */
    PA_ERR_REFCOUNT = 5,       /* allocator: release of a block nobody holds */
    PA_ERR_UNSUPPORTED = 6,    /* valid arguments outside what the kernels implement */
    PA_ERR_CUDA = 7,           /* a CUDA runtime call or kernel launch failed */
    PA_ERR_TIMEOUT = 8         /* a bounded device-side wait ran out (reported via d_err) */
} pa_status;

typedef enum {
    PA_DTYPE_F32 = 0,          /* IEEE float32 storage and operands */
    PA_DTYPE_BF16 = 1,         /* bfloat16 storage and operands, float32 accumulation */
    PA_DTYPE_FP8_E4M3 = 2      /* FP8 E4M3 pages with one float32 scale per (token, kv-head)
                                  row; new rows arrive as bf16, attention accumulates in
                                  float32 (operand precision: see pa_decode) */
} pa_dtype;

/*
 * A block pool (P1 §3, §3.1; P2 "物理布局").  K and V are separate device
 * arrays, each laid out [num_blocks][num_kv_heads][block_size][head_dim],
 * row-major: one (block, kv-head) page of one of them is block_size*head_dim
 * contiguous elements, one token row is head_dim contiguous elements.  The
 * in-block head-major order is a layout choice the pages leave open; slot
 * semantics are exactly the pages' (slot / B_p, slot mod B_p).
 *
 * FP8 pages (dtype PA_DTYPE_FP8_E4M3; the pages leave the format of quantised
 * pages open -- "KV Cache：容量、布局与生命周期" counts bytes per element in
 * the page budget): k_pool / v_pool hold E4M3 codes (OCP 8-bit float: sign,
 * 4 exponent bits with bias 7, 3 mantissa bits, max 448), and k_scale /
 * v_scale hold float32 [num_blocks][num_kv_heads][block_size], one per row.
 * A row x of D values is stored as code_d = E4M3(x_d * (448 / amax)) (float32
 * product, round to nearest even, saturating) with scale = amax / 448, amax =
 * max |x_d| (an all-zero row stores zeros and scale 0); its value is
 * decode(code_d) * scale.  k_scale / v_scale are ignored for other dtypes.
 */
typedef struct {
    void* k_pool;
    void* v_pool;
    int32_t num_blocks;
    int32_t block_size;        /* B_p, tokens per block */
    int32_t num_kv_heads;      /* H_kv */
    int32_t head_dim;          /* D */
    int32_t dtype;             /* pa_dtype */
    void* k_scale;             /* FP8 only: float32 [num_blocks][num_kv_heads][block_size] */
    void* v_scale;
} pa_kv_pool;

/* Human-readable name of a status code (static string). */
const char* pa_status_str(int32_t status);
/* Text of the last CUDA error seen by this library on the calling thread. */
const char* pa_last_cuda_error(void);
/* ABI version of this header: 2 (pa_kv_pool gained k_scale / v_scale). */
int32_t pa_abi_version(void);

/*
 * Bytes of one block for one layer, K and V together:
 * 2 * block_size * num_kv_heads * head_dim * dtype_bytes (P1 §3.1, P4
 * "获取显存块的数量"), plus 2 * block_size * num_kv_heads * 4 bytes of row
 * scales for FP8 pages.  Host only.
 */
pa_status pa_page_size_bytes(const pa_kv_pool* pool, int64_t* bytes);

/*
 * Slot of one token position (P2 "Page-table 寻址", P1 §3).  Host only.
 * table: host int32[n_entries], the sequence's logical -> physical block ids.
 * Errors: block_size <= 0 or pos < 0 -> INVALID_ARG; pos / block_size >=
 * n_entries -> OUT_OF_RANGE; a negative id -> NEGATIVE_BLOCK.  *slot is only
 * written on success.
 */
pa_status pa_physical_slot(const int32_t* table, int32_t n_entries, int32_t block_size,
                           int64_t pos, int64_t* slot);

/*
 * pa_physical_slot for `count` positions at once (the scheduler-side
 * slot_mapping of P1 §4.1).  Host only.  positions: host int64[count];
 * slots: host int64[count] out.  Stops at the first failing position and
 * returns its error; earlier entries are written.
 */
pa_status pa_slot_mapping(const int32_t* table, int32_t n_entries, int32_t block_size,
                          const int64_t* positions, int64_t count, int64_t* slots);

/*
 * Scatter write of new K/V rows into the pool (P1 §4.1, reshape_and_cache):
 * for t < num_tokens, k_new[t] and v_new[t] ([num_kv_heads][head_dim] each)
 * go to block slot_mapping[t] / B_p at offset slot_mapping[t] mod B_p, every
 * KV head.  The count is num_tokens = the length of slot_mapping, never a
 * padded K/V length.
 *   k_new, v_new: device [num_tokens][num_kv_heads][head_dim], pool dtype.
 *   slot_mapping: device int64[num_tokens].
 * A slot outside [0, num_blocks * block_size) skips that token and sets
 * *d_err = PA_ERR_OUT_OF_RANGE.  Two tokens naming the same slot race.
 * Bit-exact copy of the input bits.  num_tokens == 0 enqueues nothing.
 * Requires head_dim * dtype_bytes to be a multiple of 16 (else UNSUPPORTED).
 * FP8 pools: k_new / v_new are bf16 rows; each (token, kv-head) row is
 * quantised as the pool description states (codes and its scale written
 * together; bit-exact against that definition); head_dim must be 128.
 * The write is a dependent launch: it waits for the previous kernel in the
 * stream before touching the pool, its launch overlapping that kernel's end.
 */
pa_status pa_write_kv(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                      const int64_t* slot_mapping, int32_t num_tokens, int32_t* d_err,
                      pa_stream_t stream);

/*
 * Whole-block copy for copy-on-write of a shared, partially filled tail block
 * (P1 §5, P2 "引用计数与尾块 COW", P3 §四): for i < n, block dst[i] of both the
 * K and the V pool becomes a copy of block src[i], all heads and offsets.
 *   src, dst: device int32[n].
 * An id outside [0, num_blocks) skips that pair and sets *d_err =
 * PA_ERR_OUT_OF_RANGE.  A dst that is also a src or another dst races.
 * Bit-exact; for FP8 pools the blocks' row scales are copied with the codes.
 * n == 0 enqueues nothing.  Enqueue it before the write that follows the
 * copy-on-write decision, on the same stream.
 */
pa_status pa_copy_blocks(const pa_kv_pool* pool, const int32_t* src, const int32_t* dst,
                         int32_t n, int32_t* d_err, pa_stream_t stream);

/*
 * Split-KV decode plan.  A sequence's context is cut into partitions of
 * *partition_tokens positions (a multiple of 16); each (sequence, kv-head,
 * partition) is one unit of work whose partial softmax state is merged
 * afterwards (P1 §4: split-KV for long decode contexts).  This returns the
 * automatic choice for a batch shape on the current device.  Host only.
 */
pa_status pa_decode_partition_tokens(const pa_kv_pool* pool, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t max_context,
                                     int32_t* partition_tokens);

/*
 * Workspace bytes pa_decode needs for this shape and partition size
 * (partition_tokens 0 = the automatic choice).  The workspace holds, per
 * (sequence, q-head, partition), the running max, the exp-sum and the
 * weighted value sum (D floats).  Host only.
 */
pa_status pa_decode_workspace_bytes(const pa_kv_pool* pool, int32_t num_seqs,
                                    int32_t num_q_heads, int32_t max_context,
                                    int32_t partition_tokens, size_t* bytes);

/*
 * Paged decode attention (P1 §4 pseudo-kernel and backend rules; P3 §三).
 * One query token per sequence.  For sequence s and q-head g, with kv-head
 * h = g / (num_q_heads / num_kv_heads) and n = context_lens[s]:
 *   out[s][g] = sum_i softmax_i(scale * q[s][g] . K_i) V_i   over i < n,
 * where K_i, V_i are read through block_tables[s] (the lookup is fused into
 * the kernel).  Contexts are split into partitions whose (max, exp_sum,
 * weighted V) states are merged by a second kernel.
 *   q:            device [num_seqs][num_q_heads][head_dim], pool dtype.
 *   block_tables: device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                 ceil(n / B_p) are never read.
 *   context_lens: device int32 [num_seqs], tokens to attend to including the
 *                 new one (1 <= n <= max_context; 0 leaves out[s] untouched).
 *   max_context:  host upper bound of context_lens (sizes the plan); a
 *                 longer context is cut to its first max_context positions
 *                 and sets *d_err = PA_ERR_OUT_OF_RANGE.
 *   out:          device float32 [num_seqs][num_q_heads][head_dim].
 *   workspace:    device, >= pa_decode_workspace_bytes(...) bytes, 16-byte
 *                 aligned; may be NULL when that size is 0.
 * Implemented: head_dim * dtype_bytes == 256 (bf16 D=128, f32 D=64) or FP8
 * pages with D=128 and block size >= 4 (q is then bf16), block size a power of
 * two, num_q_heads / num_kv_heads in {1, 2, 4, 8}; other valid shapes return
 * UNSUPPORTED.  A table entry outside the pool skips its
 * tokens and sets *d_err.
 * Arithmetic: bf16 pools with D = 128, pages of >= 16 tokens and 2, 4 or 8
 * q-heads per kv-head run the score and P V products on tensor cores
 * (bf16 operands, float32 accumulation; the probabilities enter P V as a
 * bf16 high part plus a bf16 low part, about 16 significant bits).  FP8
 * pools with pages of >= 16 tokens and 8 q-heads per kv-head run them on
 * tensor cores with f16 operands: the E4M3 codes convert exactly, the query
 * is rounded to f16 once (exact for bf16 components of magnitude 2^-14 to
 * 65280; smaller ones keep an absolute precision of 2^-24; a component of
 * magnitude 65536 or more overflows and makes that row's output non-finite,
 * unflagged), the probabilities enter P V as an f16 high + low pair, and
 * accumulation is float32.  All other shapes run them in float32 on CUDA
 * cores.
 */
pa_status pa_decode(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t num_seqs, int32_t max_context,
                    float scale, int32_t partition_tokens, float* out, void* workspace,
                    size_t workspace_bytes, int32_t* d_err, pa_stream_t stream);

/*
 * The two phases of pa_decode, for callers that schedule or time them
 * separately.  pa_decode_partial takes pa_decode's arguments and runs only
 * the per-partition kernel: sequences that fit in one partition get their
 * final output in `out`, the others leave (max, exp_sum, weighted V) partials
 * in the workspace.  pa_decode_merge then combines those partials into `out`
 * (P1 §4: merge of softmax states); it must see the same pool shape,
 * num_seqs, num_q_heads, max_context and partition_tokens, and enqueues
 * nothing when every sequence fits in one partition.
 */
pa_status pa_decode_partial(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t num_seqs, int32_t max_context,
                            float scale, int32_t partition_tokens, float* out, void* workspace,
                            size_t workspace_bytes, int32_t* d_err, pa_stream_t stream);
pa_status pa_decode_merge(const pa_kv_pool* pool, int32_t num_q_heads,
                          const int32_t* context_lens, int32_t num_seqs, int32_t max_context,
                          int32_t partition_tokens, float* out, void* workspace,
                          size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode without a caller-provided workspace, for callers that cannot
 * allocate device memory when they run decode: plugin or custom-op hosts that
 * hand over raw device pointers but no allocator, and serving processes that
 * give all spare HBM to the block pool and keep no allocator headroom.  The
 * pages have no counterpart to this entry point.
 * Same arguments, kernels, partition plan and results as pa_decode minus
 * workspace/workspace_bytes.  The split-KV partials live in a static device
 * array of 16 MiB that the library's device image carries (every GPU that
 * loads the library's kernels holds it until the process exits).  A shape
 * whose pa_decode_workspace_bytes exceeds 16 MiB returns PA_ERR_UNSUPPORTED
 * and enqueues nothing.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 * Set-up: the first call in each CUDA context (the device's context, current
 * on the calling thread) looks up the array's address and caches it under
 * the context's unique id (a context created again after cudaDeviceReset is
 * looked up afresh); make the first call on each device before any stream
 * capture.  All calls share the array: calls that may overlap on the GPU
 * (unordered streams) race.  After *d_err = PA_ERR_TIMEOUT the output may
 * hold partials of an earlier call and must be discarded.
 */
pa_status pa_decode_noalloc(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t num_seqs, int32_t max_context,
                            float scale, int32_t partition_tokens, float* out, int32_t* d_err,
                            pa_stream_t stream);

/*
 * Sliding-window decode ("03｜PagedAttention 与 KV Cache 内存系统" §1.1 and §7:
 * a sliding/local-attention layer uses only the tokens of its window, and the
 * window of the token at position p is [p - w + 1, p]).  As pa_decode, but the
 * query of sequence s (position n - 1, n = context_lens[s]) attends only to
 * positions max(0, n - window) .. n - 1; pages before the window are not read.
 * window must be >= 1 (else PA_ERR_INVALID_ARG).  The workspace size depends on
 * the window: pa_decode_window_workspace_bytes.  Other arguments, limits and
 * errors as pa_decode.
 */
pa_status pa_decode_window_workspace_bytes(const pa_kv_pool* pool, int32_t num_seqs,
                                           int32_t num_q_heads, int32_t max_context,
                                           int32_t window, int32_t partition_tokens,
                                           size_t* bytes);
pa_status pa_decode_window(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t num_seqs, int32_t max_context,
                           int32_t window, float scale, int32_t partition_tokens, float* out,
                           void* workspace, size_t workspace_bytes, int32_t* d_err,
                           pa_stream_t stream);

/*
 * Shared-prefix-aware decode ("03｜PagedAttention 与 KV Cache 内存系统" §5:
 * sequences forked from one prefix hold the same physical blocks, and only a
 * partially filled shared tail is copied before a write; "PagedAttention 的原
 * 理是什么？…" §四: two requests with a common prefix point at the same
 * physical block, refcount 2).  Same result as pa_decode (the same float32
 * definition for every sequence), but a declared pair's shared pages are
 * read from HBM once for both members: one unit of work scores each shared
 * page against the q-heads of both sequences.
 *   partner:      device int32 [num_seqs]: the other member of s's pair, or -1.
 *   shared_lens:  device int32 [num_seqs]: tokens on the pair's shared
 *                 leading pages (the tables of both members hold the same
 *                 ids for the first shared_lens / block_size entries).
 * A declaration is used only if it is mutual (partner[partner[s]] == s, equal
 * shared_lens on both sides), shared_lens is a positive multiple of the block
 * size and of 16, and no longer than either member's context; otherwise
 * *d_err = PA_ERR_INVALID_ARG and both members are decoded on their own
 * (still correct).  Tables that differ over declared shared pages set
 * *d_err = PA_ERR_INVALID_ARG and leave that pair's outputs undefined.
 * Implemented: bf16 pools, head_dim 128, power-of-two block size >= 16,
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}; no sliding window.  The
 * workspace (pa_decode_shared_workspace_bytes, one partition slot per
 * sequence more than pa_decode's) holds the partials.  Other arguments,
 * limits and errors as pa_decode.
 */
pa_status pa_decode_shared_workspace_bytes(const pa_kv_pool* pool, int32_t num_seqs,
                                           int32_t num_q_heads, int32_t max_context,
                                           int32_t partition_tokens, size_t* bytes);
pa_status pa_decode_shared(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t num_seqs, int32_t max_context,
                           const int32_t* partner, const int32_t* shared_lens, float scale,
                           int32_t partition_tokens, float* out, void* workspace,
                           size_t workspace_bytes, int32_t* d_err, pa_stream_t stream);

/*
 * One decode step in a single launch: the fused form of pa_write_kv of one
 * new token per sequence followed by pa_decode (P1 §4.1: the new K/V go to
 * their slots, then attention reads them through the table; P1 §4: split-KV
 * partitions and the merge of their softmax states).  For every (sequence s,
 * kv-head h) the partition that holds position n - 1 (n = context_lens[s])
 * first writes k_new[s][h] and v_new[s][h] into slot slot_mapping[s], then
 * all partitions attend exactly as in pa_decode, and the last partition of
 * (s, h) to finish merges the group's partials into `out`.
 *   k_new, v_new:  device [num_seqs][num_kv_heads][head_dim], pool dtype,
 *                  16-byte aligned.
 *   slot_mapping:  device int64 [num_seqs]: the slot of position n - 1 under
 *                  block_tables[s] (any copy-on-write of that block must be
 *                  enqueued before).  Another slot inside the pool sets
 *                  *d_err = PA_ERR_INVALID_ARG, one outside it
 *                  PA_ERR_OUT_OF_RANGE; the row is then not written.
 *   workspace:     >= pa_decode_step_workspace_bytes(...) bytes, 16-byte
 *                  aligned (may be NULL when that size is 0), and ZERO-FILLED
 *                  before its first use (one cudaMemsetAsync after
 *                  allocation).  It holds the partials and one int32
 *                  semaphore per (sequence, kv-head); every call returns the
 *                  semaphores to zero, so the same workspace serves all later
 *                  calls of the same shape, including replays of a captured
 *                  CUDA graph.  Calls that share a workspace must be ordered
 *                  on one stream.
 * Other arguments, limits, arithmetic and errors as pa_decode (bf16 pools
 * with D = 128, pages of >= 16 tokens and 2, 4 or 8 q-heads per kv-head run
 * on tensor cores).  Allocates nothing and enqueues one kernel.
 */
pa_status pa_decode_step_workspace_bytes(const pa_kv_pool* pool, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t max_context,
                                         int32_t partition_tokens, size_t* bytes);
pa_status pa_decode_step(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, const void* q, int32_t num_q_heads,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t num_seqs, int32_t max_context,
                         float scale, int32_t partition_tokens, float* out, void* workspace,
                         size_t workspace_bytes, int32_t* d_err, pa_stream_t stream);

/*
 * Paged chunked-prefill attention on tensor cores (P1 §4: prefill reuses a
 * flash-style tiled kernel fed the paged table; paging and IO-aware tiling
 * are orthogonal).  Sequence s has new query tokens
 * q[cu_seqlens_q[s] .. cu_seqlens_q[s+1]) and context_lens[s] cache tokens
 * including those new ones (already written with pa_write_kv); new token i
 * sits at position context_lens[s] - n_new + i.  With causal != 0 it attends
 * to positions 0..its own; otherwise to all context_lens[s] positions.
 *   q:            device bf16 [total_q][num_q_heads][head_dim];
 *                 total_q = cu_seqlens_q[num_seqs] (bounds the tiled loads).
 *   cu_seqlens_q: device int32 [num_seqs + 1].
 *   context_lens: device int32 [num_seqs].
 *   block_tables: device int32 [num_seqs][max_blocks_per_seq].
 *   max_q_len:    host upper bound of the per-sequence query counts (grid).
 *   max_context:  host upper bound of context_lens (checked >= 0; the grid
 *                 depends only on max_q_len, so the kernel does not use it).
 *   out:          device float32 [total_q][num_q_heads][head_dim].
 * Implemented: bf16, head_dim 128, block size a power of two in [8, 128],
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}, pool and q 16-byte aligned.
 * A table entry outside the pool is read as block 0 and sets *d_err; a
 * sequence with context_lens < its query count sets PA_ERR_INVALID_ARG.
 * Precision: Q K^T runs on the bf16 operands; P V runs on fp16 operands (the
 * probabilities and the V values rounded to fp16, to nearest even), both
 * with float32 accumulation.  So the V values must lie within the fp16
 * range: |v| <= 65504 is exact apart from magnitudes below 2^-14, which are
 * fp16 subnormals (absolute rounding error <= 2^-25).  A V value of
 * magnitude >= 65536 (the next bf16 above 65504) or an infinity is
 * saturated to +-65504 and sets *d_err = PA_ERR_UNSUPPORTED; the output is
 * then the attention over the saturated values.
 */
pa_status pa_prefill(const pa_kv_pool* pool, const void* q, int32_t total_q,
                     int32_t num_q_heads, const int32_t* cu_seqlens_q,
                     const int32_t* context_lens, const int32_t* block_tables,
                     int32_t max_blocks_per_seq, int32_t num_seqs, int32_t max_q_len,
                     int32_t max_context, float scale, int32_t causal, float* out,
                     int32_t* d_err, pa_stream_t stream);

/*
 * Host block allocator: refcounts, free list, fork and copy-on-write tail
 * (P2 "引用计数与尾块 COW" and "生命周期与所有权"; P1 §5).  A handle is not
 * thread-safe.  Tables are caller-owned host int32 arrays; *n is their
 * current length and `capacity` their room.
 *
 * pa_alloc_create: pool of num_blocks ids, all free.  free_order (nullable,
 *   host int32[num_blocks], a permutation) gives the free list; allocation
 *   pops from its end.  NULL means ids 0..num_blocks-1 in order.
 */
pa_status pa_alloc_create(int32_t num_blocks, const int32_t* free_order, void** handle);
void pa_alloc_destroy(void* handle);
/* Pop a free block onto the end of the table, refcount 1.  NO_FREE_BLOCK,
 * INVALID_ARG if *n == capacity. */
pa_status pa_alloc_append(void* handle, int32_t* table, int32_t* n, int32_t capacity);
/* A fork: one more holder for every block of table[0..n).  The child table
 * is the caller's copy of the same ids. */
pa_status pa_alloc_fork(void* handle, const int32_t* table, int32_t n);
/*
 * Where the token at logical position `logical_length` may be written.
 * offset 0: a fresh block is appended (*n must equal logical_length /
 * block_size, else INVALID_ARG).  offset != 0 and the block has more than
 * one holder: it is replaced by a fresh exclusive block, *cow_src gets the
 * old id (the caller copies it with pa_copy_blocks before the write) and the
 * old block loses a holder.  Otherwise *cow_src = -1.  Outputs *block,
 * *offset.  OUT_OF_RANGE if the logical block is not allocated.
 */
pa_status pa_alloc_writable_tail(void* handle, int32_t* table, int32_t* n, int32_t capacity,
                                 int64_t logical_length, int32_t block_size, int32_t* block,
                                 int32_t* offset, int32_t* cow_src);
/*
 * Reserve `count` consecutive positions starting at logical_length: runs
 * pa_alloc_writable_tail for each position in order and writes the slot of
 * position logical_length + i to slots[i] (host int64[count]) — the
 * scheduler-side slot_mapping of P1 §4.1.  Every copy-on-write decision
 * appends (old, new) to cow_src/cow_dst (host int32[cow_capacity]); *n_cow
 * is the number of pairs already in them (in/out).  The caller enqueues
 * pa_copy_blocks for those pairs before pa_write_kv of the tokens.  Stops at
 * the first error (INVALID_ARG also when cow_capacity is exceeded).
 */
pa_status pa_alloc_reserve(void* handle, int32_t* table, int32_t* n, int32_t capacity,
                           int64_t logical_length, int64_t count, int32_t block_size,
                           int64_t* slots, int32_t* cow_src, int32_t* cow_dst,
                           int32_t cow_capacity, int32_t* n_cow);
/* Drop one holder from each block of table[0..n); blocks reaching 0 go back
 * on the end of the free list.  REFCOUNT on underflow (nothing changed). */
pa_status pa_alloc_release(void* handle, const int32_t* table, int32_t n);
/* Holders of one block (>= 0), or -1 for an id outside the pool. */
int32_t pa_alloc_refcount(void* handle, int32_t block);
/* Blocks on the free list. */
int32_t pa_alloc_num_free(void* handle);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */

/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged KV-cache attention library
 * (libpagedattn.so).
 *
 * The library implements the composition a model layer performs on its KV
 * cache: a slot-mapped write of each new token's K and V into a pool of
 * 16-token pages, then grouped-query causal softmax attention that reads the
 * pool back through a per-request block table, for full prefill, suffix
 * (chunked) prefill and single-query decode.
 *
 * Sources (web pages; cited by title and section):
 *   [C] "test(rocm): ReshapeAndCache->PagedAttention composition at real dims"
 *       -- What changed; maintainer review and rework (slot mapping derived
 *       from the block table, anti-vacuity guard).
 *   [R] "fix(rocm): stabilize direct paged CK attention for bitwise R/R"
 *       -- intro and Changes (fixed arithmetic schedule, real maximum query
 *       length, no implicit FMA contraction, tail-page sanitising, 64-bit
 *       addressing, one query per decode row, graph-cache identity including
 *       the KV scheduling bound); Additional checks (bitwise matrix).
 *
 * Conventions shared by every entry point:
 *   - All device buffers are owned by the caller.  The library never
 *     allocates device memory, never synchronises the stream (except
 *     pa_check_errors) and never reads device memory on the host, so calls
 *     are asynchronous on `stream` and can be captured in a CUDA graph.
 *   - Element types: q, key, value, caches and out are BF16 (passed as
 *     void*); slot_mapping is int64; block tables, lengths and
 *     query_start_loc are int32; lse is fp32.
 *   - Strides are in ELEMENTS; the head dimension is always contiguous.
 *   - Arguments are validated on the host before anything is launched; a
 *     failing check returns a status and launches nothing.  There is no
 *     fallback path: an unsupported shape is an error.
 *   - Device-side metadata errors (a block id outside [0, num_blocks), a slot
 *     past the pool, seq_len < query length, a length above its bound, a
 *     query_start_loc that decreases) never fault: the affected rows are
 *     written as NaN (attention) or skipped (cache write), other rows are
 *     untouched, and the first error is latched in a device flag read by
 *     pa_check_errors.  A request whose query range is inverted
 *     (query_start_loc[b+1] < query_start_loc[b]) owns no rows; its
 *     neighbours are checked against the bounds with the ranges they read.
 *   - `stream` is a cudaStream_t (0 = legacy default stream).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

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

typedef struct CUstream_st *pa_stream_t; /* same type as cudaStream_t */

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, bad stride */
    PA_ERR_UNSUPPORTED = 2,  /* shape outside the supported set (see below) */
    PA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    PA_ERR_BAD_METADATA = 4, /* device-side metadata error (pa_check_errors) */
    PA_ERR_TIMEOUT = 5,      /* an in-kernel wait ran past its limit */
    PA_ERR_CUDA = 6          /* a CUDA runtime call failed */
} pa_status;

/*
 * One paged KV cache: a K view and a V view with one shared set of strides.
 * Element (block, token-in-block, kv-head, d) of K is at
 *   k + block*block_stride + token*token_stride + head*head_stride + d.
 * The pages' pools map onto it as follows ([R] Additional checks names the
 * "separate", "interleaved" and ">2 GB" layouts):
 *   separate    : K and V are two [num_blocks, 16, Hkv, Dh] tensors;
 *   interleaved : one [num_blocks, 2, 16, Hkv, Dh] tensor, K = [:,0], V = [:,1]
 *                 (block_stride = 2*16*Hkv*Dh).
 * Offsets are computed in 64 bits, so a view may exceed 2**31 elements.
 * Requirements: block_size == 16; head_dim in {128, 256, 512}; k and v
 * 16-byte aligned; every stride a multiple of 8 elements (16 bytes).
 * kv_tile selects the KV tile of the attention's fixed arithmetic ("fix(rocm):
 * stabilize direct paged CK attention for bitwise R/R", Changes: fixed tile
 * 128, tile 64 also supported; Additional checks: each tile passes the bitwise
 * matrix on its own).  0 means 128 at head dims 128 and 256 and 64 at 512;
 * head dim 128 also takes 64.  Results are bitwise reproducible within one
 * tile (prefill, suffix and decode agree); the two tiles round differently.
 * Another value returns PA_ERR_INVALID_ARG, a tile the head dim lacks
 * PA_ERR_UNSUPPORTED.  The cache write and the gather ignore it.
 */
typedef struct {
    void *k;
    void *v;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t kv_tile;  /* attention KV tile: 0 = the head dim's default (see below) */
    int64_t block_stride;
    int64_t token_stride;
    int64_t head_stride;
} pa_kv_cache;

/*
 * Sets kernel attributes (dynamic shared memory) for the current device.
 * Called implicitly by the first launch on a device; call it explicitly
 * before capturing a CUDA graph ([R] Changes: warm before graph capture).
 */
PA_API pa_status pa_init(void);

/*
 * ReshapeAndCache ([C] What changed and review rework).  For every token i
 * in [0, num_tokens) with slot = slot_mapping[i] >= 0, copies the Dh BF16
 * values of each KV head h from key[i][h][:] and value[i][h][:] into block
 * slot/16, offset slot%16, head h of the K and V views.  A negative slot
 * marks a padding token and is skipped.  A slot >= num_blocks*16 is not
 * written and latches PA_ERR_BAD_METADATA with first_bad_index = i.
 *   key, value        : [num_tokens, Hkv, Dh] BF16, token stride
 *                       key_tok_stride / value_tok_stride (elements, >= Hkv*Dh,
 *                       multiple of 8), heads contiguous; 16-byte aligned.
 *   slot_mapping      : [num_tokens] int64 on the device.
 *   cache             : host struct describing the device pool (read only).
 * Duplicate non-negative slots are undefined (the pages' mapping never makes
 * them).  num_tokens == 0 launches nothing.
 */
PA_API pa_status pa_reshape_and_cache(const void *key, int64_t key_tok_stride, const void *value,
                               int64_t value_tok_stride, int64_t num_tokens,
                               const pa_kv_cache *cache, const int64_t *slot_mapping,
                               pa_stream_t stream);

/*
 * Bytes of scratch that pa_paged_attention needs for these bounds (split-KV
 * partial states and arrival counters).  The same bounds must be passed to
 * pa_paged_attention.  Returns 0 for invalid arguments.
 */
PA_API size_t pa_paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t max_query_len, int32_t max_seq_len);

/*
 * PagedAttention ([C] What changed; [R] Changes and Additional checks).
 * For request b (0 <= b < num_seqs) with q_b = query_start_loc[b+1] -
 * query_start_loc[b] new tokens and L_b = seq_lens[b] cached tokens (the new
 * tokens included, already written by pa_reshape_and_cache), query i of the
 * request sits at position p = L_b - q_b + i and attends causally to keys
 * 0..p.  Query head h uses KV head h / (Hq/Hkv).  Key j of request b lives
 * in block block_tables[b*max_blocks_per_seq + j/16] at offset j%16; table
 * columns at or past ceil(L_b/16) are never read.
 *   out[t][h][:] = softmax_j(scale * q[t][h].K_j) . V_j   (BF16, RNE)
 *   lse[t][h]    = ln(sum_j exp(scale * q[t][h].K_j))     (fp32, may be NULL)
 * Decode is query_start_loc = {0, 1, ..., num_seqs} ([R] Changes: one query
 * per row of metadata).
 *
 *   q                 : [num_q_tokens, Hq, Dh] BF16, token stride q_tok_stride
 *                       (elements, >= Hq*Dh, multiple of 8), heads contiguous.
 *   out               : [num_q_tokens, Hq, Dh] BF16, contiguous.  Rows of
 *                       tokens owned by no request are left untouched.
 *   lse               : [num_q_tokens, Hq] fp32, contiguous, or NULL.
 *                       out and lse may be device memory or page-locked host
 *                       memory mapped into the device's address space (the
 *                       kernels write them with plain stores).
 *   block_tables      : [num_seqs, max_blocks_per_seq] int32.
 *   seq_lens          : [num_seqs] int32.  query_start_loc: [num_seqs+1] int32,
 *                       non-decreasing, last entry <= num_q_tokens.
 *   max_query_len, max_seq_len : host-side upper bounds of q_b and L_b.  They
 *                       size the grid and the workspace only; any valid bound
 *                       gives bitwise-identical results ([R] Changes: real
 *                       maximum query length; KV scheduling bound in the graph
 *                       identity).  A request exceeding them latches
 *                       PA_ERR_BAD_METADATA.
 *   scale             : softmax scale, finite and > 0 (typically 1/sqrt(Dh)).
 *   workspace         : device scratch of at least
 *                       pa_paged_attention_workspace_size(...) bytes, 256-byte
 *                       aligned, zero-filled before its first use; the library
 *                       leaves it ready for the next call (after a call that
 *                       reports PA_ERR_TIMEOUT, zero-fill it again).  One
 *                       workspace must not be used by two calls that may run
 *                       concurrently.
 * Supported: head_dim in {128, 256, 512}; Hq % Hkv == 0; Hq/Hkv <= 128.
 *
 * Arithmetic is fixed ([R] intro: one schedule for strict agreement): every
 * (token, head) row is computed by the same sequence of operations whatever
 * the batch, the other requests, the query length or the bounds, so a
 * token's output and lse are bitwise identical in full prefill, suffix
 * prefill and decode.
 */
PA_API pa_status pa_paged_attention(const void *q, int64_t num_q_tokens, int64_t q_tok_stride,
                             int32_t num_q_heads, const pa_kv_cache *cache,
                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                             const int32_t *seq_lens, const int32_t *query_start_loc,
                             int32_t num_seqs, int32_t max_query_len, int32_t max_seq_len,
                             float scale, void *out, float *lse, void *workspace,
                             size_t workspace_bytes, pa_stream_t stream);

/*
 * Copies `bytes` bytes from `src` to device memory `dst` with a kernel on
 * `stream`, for step inputs that arrive in host memory.  `src` is page-locked
 * host memory mapped into the device's address space (cudaHostAlloc, or
 * cudaHostRegister with cudaHostRegisterMapped) or device memory; the kernel
 * reads it directly (on a coherent CPU-GPU link, one round trip instead of a
 * copy-engine transfer).
 *   - The paper (the source pages) has no counterpart to this entry point.
 *   - Launched with programmatic stream serialization: it waits for the
 *     preceding grid of the stream to complete before it writes dst (and,
 *     unless src_ready, before it reads src), and lets the next kernel of the
 *     stream (for instance the cache write of pa_reshape_and_paged_attention,
 *     which waits for it in turn) be scheduled meanwhile.
 *   - src_ready != 0 is the caller's statement that no kernel in flight on
 *     the GPU writes src (for instance host memory filled by the host before
 *     the call): the kernel then reads src at once, while the preceding grid
 *     may still run.
 *   - dst and src 16-byte aligned, not overlapping; otherwise
 *     PA_ERR_INVALID_ARG and nothing is launched.  bytes == 0 launches nothing.
 * The attention calls may likewise be given `out` and `lse` in page-locked,
 * mapped host memory: their kernels write the results there directly.
 */
PA_API pa_status pa_copy_to_device(void *dst, const void *src, size_t bytes, int32_t src_ready,
                                   pa_stream_t stream);

/*
 * PagedAttention for callers that cannot allocate device memory.
 *
 * Some callers cannot call cudaMalloc at all: code that runs while a CUDA
 * graph is being captured (allocation is not a capturable operation), or an
 * engine whose device memory is entirely reserved by its own pool allocator
 * and that therefore has no buffer to hand over as the workspace that
 * pa_paged_attention wants.  This variant takes the same arguments minus the
 * workspace and uses instead a scratch array built into the library: a
 * file-scope device array of PA_NOALLOC_SCRATCH_BYTES bytes that every GPU
 * which loads the library holds until the process exits.
 *   - The paper (the source pages) has no counterpart to this entry point.
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library
 *     routine.  It clears the scratch's arrival counters with
 *     cudaMemsetAsync on `stream`, then launches the same kernel as
 *     pa_paged_attention with the scratch as its workspace.
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - If the bounds need more scratch than PA_NOALLOC_SCRATCH_BYTES (see
 *     pa_paged_attention_workspace_size), it returns PA_ERR_WORKSPACE and
 *     launches nothing.
 *   - Every call on a device shares the one array: calls that may overlap on
 *     the GPU (different streams without ordering) race on it.
 */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
PA_API pa_status pa_paged_attention_noalloc(const void *q, int64_t num_q_tokens, int64_t q_tok_stride,
                                            int32_t num_q_heads, const pa_kv_cache *cache,
                                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                                            const int32_t *seq_lens, const int32_t *query_start_loc,
                                            int32_t num_seqs, int32_t max_query_len, int32_t max_seq_len,
                                            float scale, void *out, float *lse, pa_stream_t stream);

/*
 * The whole composition of [C] What changed in one call: ReshapeAndCache of
 * the num_new_tokens new tokens, then PagedAttention over the updated pool.
 * The arguments and results are those of pa_reshape_and_cache followed by
 * pa_paged_attention on `stream` (same meaning, layout and ownership); the
 * outputs are bitwise identical to that pair of calls.
 *   - Both argument sets are validated before anything is launched.
 *   - What it adds: the attention grid is scheduled while the cache write
 *     still runs.  It reads the metadata, the block tables and q and sets up
 *     its pipeline at once; only its K/V copies wait until the cache write
 *     has completed and its stores are visible.
 *   - For that reason q, block_tables, seq_lens and query_start_loc must not
 *     share bytes with the pool, and out, lse and the workspace must share
 *     none with the pool, key, value or slot_mapping.  An overlap returns
 *     PA_ERR_INVALID_ARG and launches nothing.
 *   - num_new_tokens == 0 launches only the attention, which then waits for
 *     whatever precedes it on the stream like pa_paged_attention.  An empty
 *     attention batch launches only the cache write.
 *   - Head dim 512 always waits at entry (no early reads).
 */
PA_API pa_status pa_reshape_and_paged_attention(
    const void *key, int64_t key_tok_stride, const void *value, int64_t value_tok_stride,
    int64_t num_new_tokens, const int64_t *slot_mapping, const void *q, int64_t num_q_tokens,
    int64_t q_tok_stride, int32_t num_q_heads, const pa_kv_cache *cache, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
    int32_t max_query_len, int32_t max_seq_len, float scale, void *out, float *lse, void *workspace,
    size_t workspace_bytes, pa_stream_t stream);

/*
 * Compact active-block gather of one KV head ("ROCm: harden compact
 * peer-local KV prefill for Gemma-4", Scope and Required hardening: the
 * block-table-selected pages of one K/V head packed for transfer, with
 * shuffled and sparse blocks, page boundaries, invalid metadata and byte
 * budgets).  Request b with L_b = seq_lens[b] tokens selects the
 * n_b = ceil(L_b / 16) pages block_tables[b][0..n_b-1].  With
 * off_b = n_0 + ... + n_{b-1} and total = off_{num_seqs}:
 *   packed_k[off_b + p][t][:] = K[block_tables[b][p]][t][kv_head][:]
 *   packed_v[off_b + p][t][:] = V[block_tables[b][p]][t][kv_head][:]
 *   compact_tables[b][p]      = off_b + p for p < n_b, -1 for p >= n_b
 *   compact_offsets[b]        = off_b, compact_offsets[num_seqs] = total
 * Whole pages are copied (a partial last page carries its tail rows as they
 * are in the pool).  The packed buffers form a pool of their own with one KV
 * head ({k, v, capacity_pages, 16, 1, Dh, 0, 16*Dh, Dh, Dh}); attention over
 * it with compact_tables and the group's query heads gives the same bits as
 * attention over the full pool.
 *   cache             : the pool (read only).  kv_head in [0, Hkv).
 *   block_tables      : [num_seqs, max_blocks_per_seq] int32, seq_lens
 *                       [num_seqs] int32, both on the device.
 *   packed_k, packed_v: [capacity_pages, 16, Dh] BF16 each, contiguous,
 *                       16-byte aligned, caller-owned (may be NULL when
 *                       capacity_pages == 0).
 *   compact_tables    : [num_seqs, max_blocks_per_seq] int32 (written).
 *   compact_offsets   : [num_seqs + 1] int32 (written).
 * Errors latched on the device and read with pa_check_errors:
 *   - a length outside [0, max_blocks_per_seq*16]: that request gets no
 *     pages; PA_ERR_BAD_METADATA, index = the request;
 *   - a block id outside [0, num_blocks): that packed page is NaN;
 *     PA_ERR_BAD_METADATA, index = the request;
 *   - total > capacity_pages: only compact_offsets is written (so the caller
 *     learns the size it needs); PA_ERR_WORKSPACE, index = total.
 * Host errors: PA_ERR_INVALID_ARG (bad head, sizes or pointers, or an
 * output that shares bytes with the pool, block_tables, seq_lens or another
 * output),
 * PA_ERR_UNSUPPORTED (num_seqs > 512 or num_seqs*max_blocks_per_seq >
 * INT32_MAX).  num_seqs == 0 launches nothing.  The launch waits for the
 * work before it on the stream (it may be launched early with programmatic
 * stream serialization and waits in the kernel).
 */
PA_API pa_status pa_gather_kv_head(const pa_kv_cache *cache, int32_t kv_head, const int32_t *block_tables,
                                   int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                                   void *packed_k, void *packed_v, int64_t capacity_pages,
                                   int32_t *compact_tables, int32_t *compact_offsets, pa_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * flag.  Returns PA_OK, PA_ERR_BAD_METADATA or PA_ERR_TIMEOUT (or
 * PA_ERR_CUDA if the synchronisation failed).  *first_bad_index (may be
 * NULL) receives the token index (cache write) or request index (attention)
 * of the first recorded error, else -1.
 */
PA_API pa_status pa_check_errors(pa_stream_t stream, int64_t *first_bad_index);

/*
 * Sets the time limit of the one wait in the split-KV fold that depends on
 * other CTAs (the folders of a (request, KV head) group waiting until every
 * CTA of the group has published its chunk state) and returns the previous
 * limit.  The default is 2 s.  It exists to exercise the timeout path ("ROCm:
 * harden compact peer-local KV prefill for Gemma-4", Required hardening:
 * bounded waits, fatal after submit, no retry): with 0 the waiting CTAs give
 * up at once, latch PA_ERR_TIMEOUT and leave their share of the rows
 * unwritten; the kernel still ends normally.  While nothing is copied or
 * computed at that point, no other wait is affected.  The value is read at
 * each launch (a captured CUDA graph keeps the value of its capture) and is
 * process-wide.  After a call that reported PA_ERR_TIMEOUT, zero-fill the
 * workspace before reusing it.
 */
PA_API uint64_t pa_set_fold_wait_limit_ns(uint64_t limit_ns);

/* Static, human-readable name of a status code. */
PA_API const char *pa_status_string(pa_status status);

/*
 * Copies a one-line description of the calling thread's most recent launch
 * (schedule, grid, chunk count, KV tile) into buf (NUL-terminated,
 * truncated to n bytes) -- the "selected entrypoint" breadcrumb of
 * [R] Changes.
 */
PA_API void pa_last_launch_info(char *buf, size_t n);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */

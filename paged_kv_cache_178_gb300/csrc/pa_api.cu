// C-ABI front end of libpagedattn.so: argument validation, the cache write
// kernel (K1), the device error latch and launch breadcrumbs.  The attention
// kernel lives in pa_attn.cu.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/pagedattn.h"
#include "pa_internal.h"

namespace pa {

// One error latch per device (each device that loads the module has its own
// copy); host code reaches it through cudaGetSymbolAddress.
__device__ ErrState g_err_state;

constexpr int kMaxDevices = 64;
static std::mutex g_mu;
static ErrState *g_err_ptr[kMaxDevices];
static bool g_attr_done[kMaxDevices];
static thread_local char g_last_info[256] = "none";

static pa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

// Per-device one-time set-up: resolve the error latch address and set kernel
// attributes.  Must run with the device current.
static pa_status device_setup(ErrState **err_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_attr_done[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_err_state) != cudaSuccess)
            return PA_ERR_CUDA;
        if (init_attention_attributes() != cudaSuccess)
            return PA_ERR_CUDA;
        g_err_ptr[dev] = static_cast<ErrState *>(ptr);
        g_attr_done[dev] = true;
    }
    if (err_out)
        *err_out = g_err_ptr[dev];
    return PA_OK;
}

CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, cuuint32_t rank, void *base,
                      const cuuint64_t *dims, const cuuint64_t *strides_bytes, const cuuint32_t *box,
                      CUtensorMapSwizzle swizzle)
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn)
        return CUDA_ERROR_NOT_FOUND;
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    return fn(map, dtype, rank, base, dims, strides_bytes, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// K1: slot-mapped cache write.  One thread per 16-byte vector of one
// (token, kv head, K-or-V) row.  Offsets are 64-bit.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4 *__restrict__ key, int64_t key_tok_stride, const uint4 *__restrict__ value,
    int64_t value_tok_stride, int64_t num_tokens, int32_t num_kv_heads, int32_t vecs_per_row,
    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, int64_t num_slots, int64_t block_stride,
    int64_t token_stride, int64_t head_stride, const int64_t *__restrict__ slot_mapping, ErrState *err)
{
    // Launched with programmatic stream serialization: wait for the preceding
    // grid of the stream (it may have produced key, value or slot_mapping),
    // then let the dependent grid be scheduled.  The attention that usually
    // follows may read its metadata and q from here on -- the grids before
    // this one have completed -- and waits for this grid before touching the
    // cache.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // strides arrive in 16-byte units
    const int64_t total = num_tokens * num_kv_heads * 2 * vecs_per_row;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int vec = (int)(idx % vecs_per_row);
        int64_t rest = idx / vecs_per_row;
        const int which = (int)(rest % 2);
        rest /= 2;
        const int h = (int)(rest % num_kv_heads);
        const int64_t i = rest / num_kv_heads;
        // the source vector does not depend on the slot: both loads are in
        // flight together (token i's row exists whatever its slot says)
        const uint4 src = which == 0 ? __ldg(key + i * key_tok_stride + (int64_t)h * vecs_per_row + vec)
                                     : __ldg(value + i * value_tok_stride + (int64_t)h * vecs_per_row + vec);
        const int64_t slot = __ldg(slot_mapping + i);
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            if (vec == 0 && which == 0 && h == 0)
                record_error(err, kErrBadMetadata, i);
            continue;
        }
        const int64_t dst = (slot >> 4) * block_stride + (slot & 15) * token_stride + h * head_stride + vec;
        (which == 0 ? k_cache : v_cache)[dst] = src;
    }
}

// Staging copy (pa_copy_to_device): 16-byte vectors, up to four per thread
// per pass with every load issued before the stores, so a source in host
// memory costs one round trip over the CPU-GPU link per pass; the bytes past
// the last whole vector go one by one.  With src_ready the first pass reads
// before the wait for the preceding grid (no grid in flight writes src);
// every store still waits for it (it may read dst).
__global__ void __launch_bounds__(256) copy_to_device_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                                             int64_t n16, uint8_t *__restrict__ dst_tail,
                                                             const uint8_t *__restrict__ src_tail, int tail,
                                                             int src_ready)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint4 v[4];
    uint8_t t8 = 0;
    const bool tail_thread = blockIdx.x == 0 && (int)threadIdx.x < tail;
    if (src_ready) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (base + i * stride < n16)
                v[i] = src[base + i * stride];
        if (tail_thread)
            t8 = src_tail[threadIdx.x];
    }
    // programmatic stream serialization: the preceding grid may still read
    // dst (and, without src_ready, write src) until it has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (bool first = true; base < n16; base += 4 * stride, first = false) {
        if (!first || !src_ready) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (base + i * stride < n16)
                    v[i] = src[base + i * stride];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (base + i * stride < n16)
                dst[base + i * stride] = v[i];
    }
    if (tail_thread)
        dst_tail[threadIdx.x] = src_ready ? t8 : src_tail[threadIdx.x];
}

}  // namespace pa

using namespace pa;

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The attention's KV tile: 0 (the head dim's default), or a tile that head
// dim has -- 64 or 128 at head dim 128, 128 at 256, 64 at 512.
static pa_status check_kv_tile(const pa_kv_cache *c)
{
    const int t = c->kv_tile;
    if (t == 0)
        return PA_OK;
    if (t != 64 && t != 128)
        return PA_ERR_INVALID_ARG;
    const bool ok = c->head_dim == 128 || (c->head_dim == 256 && t == 128) || (c->head_dim == 512 && t == 64);
    return ok ? PA_OK : PA_ERR_UNSUPPORTED;
}

static pa_status check_cache(const pa_kv_cache *c)
{
    if (!c || !c->k || !c->v)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(c->k) || !aligned16(c->v))
        return PA_ERR_INVALID_ARG;
    if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (c->block_size != 16)
        return PA_ERR_UNSUPPORTED;
    if (c->head_dim != 128 && c->head_dim != 256 && c->head_dim != 512)
        return PA_ERR_UNSUPPORTED;
    if (c->block_stride <= 0 || c->token_stride <= 0 || c->head_stride <= 0)
        return PA_ERR_INVALID_ARG;
    if ((c->block_stride | c->token_stride | c->head_stride) & 7)
        return PA_ERR_INVALID_ARG;
    if (c->head_stride < c->head_dim || c->num_blocks > (int64_t)1 << 31)
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

extern "C" {

const char *pa_status_string(pa_status s)
{
    switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_BAD_METADATA: return "PA_ERR_BAD_METADATA";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    }
    return "PA_ERR_UNKNOWN";
}

void pa_last_launch_info(char *buf, size_t n)
{
    if (!buf || !n)
        return;
    snprintf(buf, n, "%s", g_last_info);
}

pa_status pa_init(void) { return device_setup(nullptr); }

// Cache-write arguments after validation.
struct ReshapeCall {
    const void *key, *value;
    int64_t key_tok_stride, value_tok_stride, num_tokens;
    const pa_kv_cache *cache;
    const int64_t *slot_mapping;
};

static pa_status reshape_check(const ReshapeCall &c)
{
    pa_status st = check_cache(c.cache);
    if (st != PA_OK)
        return st;
    if (c.num_tokens < 0)
        return PA_ERR_INVALID_ARG;
    if (c.num_tokens == 0)
        return PA_OK;
    const int64_t row = (int64_t)c.cache->num_kv_heads * c.cache->head_dim;
    if (!c.key || !c.value || !c.slot_mapping || !aligned16(c.key) || !aligned16(c.value))
        return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(c.slot_mapping) & 7u) != 0)
        return PA_ERR_INVALID_ARG;
    if (c.key_tok_stride < row || c.value_tok_stride < row || (c.key_tok_stride & 7) || (c.value_tok_stride & 7))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

static pa_status reshape_launch(const ReshapeCall &c, ErrState *err, cudaStream_t stream, char *info,
                                size_t info_len)
{
    if (c.num_tokens == 0) {
        snprintf(info, info_len, "reshape_and_cache tokens=0 (nothing launched)");
        return PA_OK;
    }
    const pa_kv_cache *cache = c.cache;
    const int vecs = cache->head_dim / 8;
    const int64_t total = c.num_tokens * cache->num_kv_heads * 2 * vecs;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16)
        blocks = 152 * 16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, reshape_and_cache_kernel, static_cast<const uint4 *>(c.key), (int64_t)(c.key_tok_stride / 8),
        static_cast<const uint4 *>(c.value), (int64_t)(c.value_tok_stride / 8), c.num_tokens,
        (int32_t)cache->num_kv_heads, (int32_t)vecs, static_cast<uint4 *>(cache->k), static_cast<uint4 *>(cache->v),
        (int64_t)(cache->num_blocks * 16), (int64_t)(cache->block_stride / 8), (int64_t)(cache->token_stride / 8),
        (int64_t)(cache->head_stride / 8), c.slot_mapping, err);
    snprintf(info, info_len, "reshape_and_cache tokens=%lld grid=%lld block=256", (long long)c.num_tokens,
             (long long)blocks);
    return cuda_status(e);
}

// Validates an attention call and fills the kernel arguments and the plan.
// *empty is set when there is nothing to launch.
static pa_status attention_check(const void *q, int64_t num_q_tokens, int64_t q_tok_stride, int32_t num_q_heads,
                                 const pa_kv_cache *cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                                 int32_t max_query_len, int32_t max_seq_len, float scale, void *out, float *lse,
                                 void *workspace, size_t workspace_bytes, AttnArgs *a, AttnPlan *pl, bool *empty)
{
    *empty = false;
    pa_status st = check_cache(cache);
    if (st != PA_OK)
        return st;
    if ((st = check_kv_tile(cache)) != PA_OK)
        return st;
    if (num_q_heads <= 0 || num_seqs < 0 || max_query_len < 0 || max_seq_len < 0 || num_q_tokens < 0 ||
        max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % cache->num_kv_heads != 0 || num_q_heads / cache->num_kv_heads > 128)
        return PA_ERR_UNSUPPORTED;
    if (!(scale > 0.f) || scale == INFINITY)  // also rejects NaN
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_q_tokens == 0 || max_query_len == 0) {
        *empty = true;
        return PA_OK;
    }
    const int64_t row = (int64_t)num_q_heads * cache->head_dim;
    if (!q || !out || !block_tables || !seq_lens || !query_start_loc || !aligned16(q) || !aligned16(out))
        return PA_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return PA_ERR_INVALID_ARG;
    if (q_tok_stride < row || (q_tok_stride & 7) || num_q_tokens > ((int64_t)1 << 31) - 1)
        return PA_ERR_INVALID_ARG;
    if (max_blocks_per_seq == 0)
        return PA_ERR_INVALID_ARG;
    if (!plan_attention(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim, max_query_len, max_seq_len,
                        pl))
        return PA_ERR_UNSUPPORTED;
    if (cache->kv_tile != 0)
        pl->kt = cache->kv_tile;
    if (pl->ws_bytes > 0) {
        if (!workspace || workspace_bytes < pl->ws_bytes)
            return PA_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return PA_ERR_INVALID_ARG;
    }
    a->q = q;
    a->num_q_tokens = num_q_tokens;
    a->q_tok_stride = q_tok_stride;
    a->num_q_heads = num_q_heads;
    a->k = cache->k;
    a->v = cache->v;
    a->num_blocks = cache->num_blocks;
    a->num_kv_heads = cache->num_kv_heads;
    a->head_dim = cache->head_dim;
    a->block_stride = cache->block_stride;
    a->token_stride = cache->token_stride;
    a->head_stride = cache->head_stride;
    a->block_tables = block_tables;
    a->max_blocks_per_seq = max_blocks_per_seq;
    a->seq_lens = seq_lens;
    a->query_start_loc = query_start_loc;
    a->num_seqs = num_seqs;
    a->max_query_len = max_query_len;
    a->max_seq_len = max_seq_len;
    a->scale = scale;
    a->out = out;
    a->lse = lse;
    a->workspace = workspace;
    a->workspace_bytes = workspace_bytes;
    a->early_reads = false;
    return PA_OK;
}

static pa_status attention_launch(const AttnArgs &a, const AttnPlan &pl, ErrState *err, cudaStream_t stream,
                                  char *info, size_t info_len)
{
    cudaError_t e = launch_attention(a, pl, err, stream, info, info_len);
    if (e == cudaErrorNotSupported)
        return PA_ERR_UNSUPPORTED;
    return cuda_status(e);
}

// Half-open byte range [lo, hi) of a device buffer.
struct Span {
    uintptr_t lo, hi;
};

static Span span(const void *p, int64_t bytes)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Span{lo, lo + (uintptr_t)(bytes > 0 ? bytes : 0)};
}

static bool overlaps(const Span &x, const Span &y) { return x.lo < y.hi && y.lo < x.hi; }

// Bytes spanned by one view of the pool (K or V).
static int64_t pool_view_bytes(const pa_kv_cache *c)
{
    return ((c->num_blocks - 1) * c->block_stride + 15 * c->token_stride +
            (int64_t)(c->num_kv_heads - 1) * c->head_stride + c->head_dim) *
           2;
}

pa_status pa_reshape_and_cache(const void *key, int64_t key_tok_stride, const void *value,
                               int64_t value_tok_stride, int64_t num_tokens, const pa_kv_cache *cache,
                               const int64_t *slot_mapping, pa_stream_t stream)
{
    const ReshapeCall c{key, value, key_tok_stride, value_tok_stride, num_tokens, cache, slot_mapping};
    pa_status st = reshape_check(c);
    if (st != PA_OK)
        return st;
    ErrState *err = nullptr;
    if (num_tokens > 0 && (st = device_setup(&err)) != PA_OK)
        return st;
    return reshape_launch(c, err, reinterpret_cast<cudaStream_t>(stream), g_last_info, sizeof g_last_info);
}

pa_status pa_copy_to_device(void *dst, const void *src, size_t bytes, int32_t src_ready, pa_stream_t stream)
{
    if (bytes == 0)
        return PA_OK;
    if (!dst || !src)
        return PA_ERR_INVALID_ARG;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    if (d < s + bytes && s < d + bytes)
        return PA_ERR_INVALID_ARG;  // overlapping ranges
    if ((d | s) & 15u)
        return PA_ERR_INVALID_ARG;  // both 16-byte aligned
    ErrState *err = nullptr;
    pa_status st = device_setup(&err);
    if (st != PA_OK)
        return st;
    const int64_t n16 = (int64_t)(bytes / 16);
    const int tail = (int)(bytes % 16);
    int64_t blocks = (n16 + 4 * 256 - 1) / (4 * 256);
    if (blocks < 1)
        blocks = 1;
    if (blocks > 152 * 8)
        blocks = 152 * 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e =
        cudaLaunchKernelEx(&cfg, copy_to_device_kernel, static_cast<uint4 *>(dst), static_cast<const uint4 *>(src),
                           n16, static_cast<uint8_t *>(dst) + n16 * 16, static_cast<const uint8_t *>(src) + n16 * 16,
                           tail, src_ready ? 1 : 0);
    snprintf(g_last_info, sizeof g_last_info, "copy_to_device bytes=%zu grid=%lld block=256", bytes,
             (long long)blocks);
    return cuda_status(e);
}

size_t pa_paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t max_query_len, int32_t max_seq_len)
{
    AttnPlan pl{};
    if (!plan_attention(num_seqs, num_q_heads, num_kv_heads, head_dim, max_query_len, max_seq_len, &pl))
        return 0;
    return pl.ws_bytes;
}

pa_status pa_paged_attention(const void *q, int64_t num_q_tokens, int64_t q_tok_stride, int32_t num_q_heads,
                             const pa_kv_cache *cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                             const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                             int32_t max_query_len, int32_t max_seq_len, float scale, void *out, float *lse,
                             void *workspace, size_t workspace_bytes, pa_stream_t stream)
{
    AttnArgs a;
    AttnPlan pl{};
    bool empty = false;
    pa_status st = attention_check(q, num_q_tokens, q_tok_stride, num_q_heads, cache, block_tables,
                                   max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, max_query_len,
                                   max_seq_len, scale, out, lse, workspace, workspace_bytes, &a, &pl, &empty);
    if (st != PA_OK)
        return st;
    if (empty) {
        snprintf(g_last_info, sizeof g_last_info, "attention: empty batch (nothing launched)");
        return PA_OK;
    }
    ErrState *err = nullptr;
    if ((st = device_setup(&err)) != PA_OK)
        return st;
    return attention_launch(a, pl, err, reinterpret_cast<cudaStream_t>(stream), g_last_info, sizeof g_last_info);
}

pa_status pa_reshape_and_paged_attention(const void *key, int64_t key_tok_stride, const void *value,
                                         int64_t value_tok_stride, int64_t num_new_tokens,
                                         const int64_t *slot_mapping, const void *q, int64_t num_q_tokens,
                                         int64_t q_tok_stride, int32_t num_q_heads, const pa_kv_cache *cache,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *seq_lens, const int32_t *query_start_loc,
                                         int32_t num_seqs, int32_t max_query_len, int32_t max_seq_len,
                                         float scale, void *out, float *lse, void *workspace,
                                         size_t workspace_bytes, pa_stream_t stream)
{
    // Validate both calls before launching either.
    const ReshapeCall c{key, value, key_tok_stride, value_tok_stride, num_new_tokens, cache, slot_mapping};
    pa_status st = reshape_check(c);
    if (st != PA_OK)
        return st;
    AttnArgs a;
    AttnPlan pl{};
    bool empty = false;
    st = attention_check(q, num_q_tokens, q_tok_stride, num_q_heads, cache, block_tables, max_blocks_per_seq,
                         seq_lens, query_start_loc, num_seqs, max_query_len, max_seq_len, scale, out, lse,
                         workspace, workspace_bytes, &a, &pl, &empty);
    if (st != PA_OK)
        return st;
    if (!empty && num_new_tokens > 0) {
        // The attention grid reads q and the metadata, and writes out, lse
        // and the workspace, while the cache write may still run: none of
        // them may share bytes with what the cache write reads or writes.
        const int64_t kv_row = (int64_t)cache->num_kv_heads * cache->head_dim;
        const Span writes_of_write[2] = {span(cache->k, pool_view_bytes(cache)),
                                         span(cache->v, pool_view_bytes(cache))};
        const Span reads_of_write[3] = {span(key, ((num_new_tokens - 1) * key_tok_stride + kv_row) * 2),
                                        span(value, ((num_new_tokens - 1) * value_tok_stride + kv_row) * 2),
                                        span(slot_mapping, num_new_tokens * 8)};
        const Span early_reads[4] = {
            span(q, ((num_q_tokens - 1) * q_tok_stride + (int64_t)num_q_heads * cache->head_dim) * 2),
            span(block_tables, (int64_t)num_seqs * max_blocks_per_seq * 4), span(seq_lens, (int64_t)num_seqs * 4),
            span(query_start_loc, ((int64_t)num_seqs + 1) * 4)};
        const Span attn_writes[3] = {span(out, num_q_tokens * num_q_heads * (int64_t)cache->head_dim * 2),
                                     span(lse, lse ? num_q_tokens * num_q_heads * 4 : 0),
                                     span(workspace, (int64_t)pl.ws_bytes)};
        for (const Span &w : writes_of_write)
            for (const Span &r : early_reads)
                if (overlaps(w, r))
                    return PA_ERR_INVALID_ARG;
        for (const Span &w : attn_writes) {
            for (const Span &x : writes_of_write)
                if (overlaps(w, x))
                    return PA_ERR_INVALID_ARG;
            for (const Span &x : reads_of_write)
                if (overlaps(w, x))
                    return PA_ERR_INVALID_ARG;
        }
    }
    ErrState *err = nullptr;
    if ((st = device_setup(&err)) != PA_OK)
        return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char info_w[128], info_a[192];
    if ((st = reshape_launch(c, err, s, info_w, sizeof info_w)) != PA_OK)
        return st;
    if (empty) {
        snprintf(g_last_info, sizeof g_last_info, "%.80s; attention: empty batch (nothing launched)", info_w);
        return PA_OK;
    }
    // Only a cache write launched just before makes the early reads safe;
    // the head-dim 512 kernel always waits at entry.
    a.early_reads = num_new_tokens > 0 && cache->head_dim != 512;
    st = attention_launch(a, pl, err, s, info_a, sizeof info_a);
    snprintf(g_last_info, sizeof g_last_info, "%.80s; %.160s%s", info_w, info_a, a.early_reads ? " early_reads" : "");
    return st;
}

// Scratch for pa_paged_attention_noalloc: lives in the library image, so
// every device that loads the library holds it; nothing is allocated per call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];
static void *g_noalloc_ptr[kMaxDevices];

pa_status pa_paged_attention_noalloc(const void *q, int64_t num_q_tokens, int64_t q_tok_stride,
                                     int32_t num_q_heads, const pa_kv_cache *cache,
                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                     const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                                     int32_t max_query_len, int32_t max_seq_len, float scale, void *out,
                                     float *lse, pa_stream_t stream)
{
    // Every host check of pa_paged_attention runs first, against the
    // built-in array's size, before any CUDA call: a stand-in address (256,
    // aligned and never dereferenced) takes the scratch's place until the
    // call is known to be valid.  Bounds that need more scratch than the
    // array holds fail here with PA_ERR_WORKSPACE.
    AttnArgs a;
    AttnPlan pl{};
    bool empty = false;
    pa_status st = attention_check(q, num_q_tokens, q_tok_stride, num_q_heads, cache, block_tables,
                                   max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, max_query_len,
                                   max_seq_len, scale, out, lse, reinterpret_cast<void *>(uintptr_t{256}),
                                   PA_NOALLOC_SCRATCH_BYTES, &a, &pl, &empty);
    if (st != PA_OK)
        return st;
    if (empty) {
        snprintf(g_last_info, sizeof g_last_info, "attention: empty batch (nothing launched)");
        return PA_OK;
    }
    ErrState *err = nullptr;
    if ((st = device_setup(&err)) != PA_OK)
        return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PA_ERR_CUDA;
    void *scratch = nullptr;
    {
        // Host code cannot use the array's name as a device address: resolve
        // it once per device, with that device current.
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_noalloc_ptr[dev]) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
                return PA_ERR_CUDA;
            g_noalloc_ptr[dev] = ptr;
        }
        scratch = g_noalloc_ptr[dev];
    }
    a.workspace = scratch;
    a.workspace_bytes = PA_NOALLOC_SCRATCH_BYTES;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The arrival counters at the head of the scratch must start at zero; the
    // previous call (or an aborted one) may have left anything there.
    if (pl.ws_counter_bytes > 0 && cudaMemsetAsync(scratch, 0, pl.ws_counter_bytes, s) != cudaSuccess)
        return PA_ERR_CUDA;
    return attention_launch(a, pl, err, s, g_last_info, sizeof g_last_info);
}

uint64_t pa_set_fold_wait_limit_ns(uint64_t limit_ns) { return set_fold_wait_limit_ns(limit_ns); }

pa_status pa_check_errors(pa_stream_t stream, int64_t *first_bad_index)
{
    if (first_bad_index)
        *first_bad_index = -1;
    ErrState *err = nullptr;
    pa_status st = device_setup(&err);
    if (st != PA_OK)
        return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    ErrState h{};
    if (cudaMemcpy(&h, err, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PA_ERR_CUDA;
    if (h.code == 0)
        return PA_OK;
    const ErrState zero{};
    if (cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return PA_ERR_CUDA;
    if (first_bad_index)
        *first_bad_index = h.index;
    if (h.code == kErrBudget)
        return PA_ERR_WORKSPACE;
    return h.code == kErrTimeout ? PA_ERR_TIMEOUT : PA_ERR_BAD_METADATA;
}

pa_status pa_gather_kv_head(const pa_kv_cache *cache, int32_t kv_head, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                            void *packed_k, void *packed_v, int64_t capacity_pages, int32_t *compact_tables,
                            int32_t *compact_offsets, pa_stream_t stream)
{
    pa_status st = check_cache(cache);
    if (st != PA_OK)
        return st;
    if (kv_head < 0 || kv_head >= cache->num_kv_heads || num_seqs < 0 || max_blocks_per_seq <= 0 ||
        capacity_pages < 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs > kGatherMaxSeqsHost || (int64_t)num_seqs * max_blocks_per_seq > INT32_MAX)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) {
        snprintf(g_last_info, sizeof g_last_info, "gather_kv_head: empty batch (nothing launched)");
        return PA_OK;
    }
    if (!block_tables || !seq_lens || !compact_tables || !compact_offsets)
        return PA_ERR_INVALID_ARG;
    if (capacity_pages > 0 && (!packed_k || !packed_v || !aligned16(packed_k) || !aligned16(packed_v)))
        return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(compact_tables) | reinterpret_cast<uintptr_t>(compact_offsets) |
         reinterpret_cast<uintptr_t>(block_tables) | reinterpret_cast<uintptr_t>(seq_lens)) &
        3u)
        return PA_ERR_INVALID_ARG;
    {
        // the kernel writes its four outputs while it reads the pool and the
        // metadata: no output may share a byte with an input or another output
        const int64_t page_bytes = (int64_t)16 * cache->head_dim * 2;
        const int64_t table_bytes = (int64_t)num_seqs * max_blocks_per_seq * 4;
        const Span reads[4] = {span(cache->k, pool_view_bytes(cache)), span(cache->v, pool_view_bytes(cache)),
                               span(block_tables, table_bytes), span(seq_lens, (int64_t)num_seqs * 4)};
        const Span writes[4] = {span(packed_k, capacity_pages * page_bytes),
                                span(packed_v, capacity_pages * page_bytes), span(compact_tables, table_bytes),
                                span(compact_offsets, ((int64_t)num_seqs + 1) * 4)};
        for (int i = 0; i < 4; ++i) {
            for (const Span &r : reads)
                if (overlaps(writes[i], r))
                    return PA_ERR_INVALID_ARG;
            for (int j = i + 1; j < 4; ++j)
                if (overlaps(writes[i], writes[j]))
                    return PA_ERR_INVALID_ARG;
        }
    }
    ErrState *err = nullptr;
    if ((st = device_setup(&err)) != PA_OK)
        return st;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PA_ERR_CUDA;
    const cudaError_t e = launch_gather_kv_head(
        cache->k, cache->v, cache->num_blocks, cache->block_stride, cache->token_stride, cache->head_stride,
        kv_head, cache->head_dim, block_tables, max_blocks_per_seq, seq_lens, num_seqs, packed_k, packed_v,
        capacity_pages, compact_tables, compact_offsets, err, reinterpret_cast<cudaStream_t>(stream), nsm);
    snprintf(g_last_info, sizeof g_last_info, "gather_kv_head head=%d seqs=%d capacity_pages=%lld", kv_head,
             num_seqs, (long long)capacity_pages);
    return cuda_status(e);
}

}  // extern "C"

// Compact active-block gather: the pages that the block table selects for one
// KV head, packed into a contiguous buffer, with compact metadata
// ("ROCm: harden compact peer-local KV prefill for Gemma-4", Scope: compact
// active block-table-selected K/V head; Required hardening: shuffled and
// sparse blocks, page boundaries, invalid metadata, byte budgets).  Here the
// packed buffer stays on the same GPU: it is a pool of its own (one KV head,
// pages in request order) that the attention can read through the compact
// table.
//
// Request b with L_b tokens owns n_b = ceil(L_b / 16) pages, table columns
// 0..n_b-1.  Its packed pages start at off_b = n_0 + ... + n_{b-1}:
//   packed[off_b + p][t][:] = pool[table[b][p]][t][h][:]   (whole pages)
//   compact_table[b][p]     = off_b + p  (p < n_b), -1 beyond
//   compact_offsets[b]      = off_b, compact_offsets[num_seqs] = total pages
// K and V alike.  A block id outside the pool fills its packed page with NaN
// and latches PA_ERR_BAD_METADATA (index: the request); a length outside
// [0, max_blocks*16] latches it too and gives the request no pages.  When the
// pages do not fit in `capacity_pages`, only compact_offsets is written and
// PA_ERR_WORKSPACE is latched (index: the pages needed).
#include <cuda_bf16.h>

#include "pa_internal.h"

namespace pa {

constexpr int kGatherThreads = 512;
constexpr int kGatherMaxSeqs = kGatherThreads;  // one request per thread in the scan
constexpr int kGatherPagesPerPass = 4;          // pages in flight per CTA pass

// VPR: 16-byte vectors per K (or V) row of one head (head dim / 8), so the
// index arithmetic below is shifts and masks.
template <int VPR>
__global__ void __launch_bounds__(kGatherThreads, 3) gather_kv_head_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, int64_t num_blocks, int64_t block_stride,
    int64_t token_stride, int64_t head_off, const int32_t *__restrict__ block_tables,
    int32_t max_blocks, const int32_t *__restrict__ seq_lens, int32_t num_seqs, uint4 *__restrict__ packed_k,
    uint4 *__restrict__ packed_v, int64_t capacity_pages, int32_t *__restrict__ compact_tables,
    int32_t *__restrict__ compact_offsets, ErrState *err)
{
    // strides and head_off arrive in 16-byte units
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ int s_off[kGatherMaxSeqs + 1];
    __shared__ int s_warp[kGatherThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // pages per request (bad lengths: none, and the error is latched once)
    int n = 0;
    if (tid < num_seqs) {
        const int L = __ldg(seq_lens + tid);
        if (L < 0 || (int64_t)L > (int64_t)max_blocks * 16) {
            if (blockIdx.x == 0)
                record_error(err, kErrBadMetadata, tid);
        } else {
            n = (L + 15) / 16;
        }
    }
    // block-wide exclusive prefix sum
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += x;
    }
    if (lane == 31)
        s_warp[warp] = incl;
    __syncthreads();
    int wpre = 0, total = 0;
    for (int w = 0; w < kGatherThreads / 32; ++w) {
        if (w < warp)
            wpre += s_warp[w];
        total += s_warp[w];
    }
    if (tid < num_seqs)
        s_off[tid] = wpre + incl - n;
    if (tid == 0)
        s_off[num_seqs] = total;
    __syncthreads();
    if (blockIdx.x == 0)
        for (int b = tid; b <= num_seqs; b += blockDim.x)
            compact_offsets[b] = s_off[b];
    if ((int64_t)total > capacity_pages) {
        if (blockIdx.x == 0 && tid == 0)
            record_error(err, kErrBudget, total);
        return;
    }
    // compact table: the packed index of each selected page, -1 beyond
    const int64_t n_tab = (int64_t)num_seqs * max_blocks;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + tid; e < n_tab; e += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(e / max_blocks), p = (int)(e % max_blocks);
        const int nb = s_off[b + 1] - s_off[b];
        compact_tables[e] = p < nb ? s_off[b] + p : -1;
    }
    // pages: kGatherPagesPerPass per CTA pass, every vector loaded before any
    // is stored; the block ids of the next pass are read while this pass's
    // vectors are in flight
    constexpr int vecs_page = 16 * VPR;  // 16-byte vectors of one K (or V) page
    const uint4 qnan = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
    // block id of packed page c (raw, unchecked), and its request
    auto page_id = [&](int64_t c, int &req) -> int {
        // request of packed page c: the last b with s_off[b] <= c
        int lo = 0, hi = num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_off[mid] <= c)
                lo = mid;
            else
                hi = mid - 1;
        }
        req = lo;
        return __ldg(block_tables + (int64_t)lo * max_blocks + (c - s_off[lo]));
    };
    // lane j of every warp looks up page j of a pass; the others read it with
    // a shuffle
    const int64_t stride = (int64_t)gridDim.x * kGatherPagesPerPass;
    int64_t c0 = (int64_t)blockIdx.x * kGatherPagesPerPass;
    int next_id = 0, next_req = 0;
    if (lane < kGatherPagesPerPass && c0 + lane < total)
        next_id = page_id(c0 + lane, next_req);
    for (; c0 < total; c0 += stride) {
        int64_t src_page[kGatherPagesPerPass];
#pragma unroll
        for (int j = 0; j < kGatherPagesPerPass; ++j) {
            const int id = __shfl_sync(0xffffffffu, next_id, j);
            src_page[j] = -2;  // past the last page: nothing to do
            if (c0 + j < total) {
                if (id < 0 || (int64_t)id >= num_blocks) {
                    if (tid == j)
                        record_error(err, kErrBadMetadata, next_req);
                    src_page[j] = -1;  // NaN page
                } else {
                    src_page[j] = id;
                }
            }
        }
        const int64_t c1 = c0 + stride;
        if (lane < kGatherPagesPerPass && c1 + lane < total)
            next_id = page_id(c1 + lane, next_req);
        for (int e = tid; e < 2 * vecs_page; e += blockDim.x) {
            const int which = e / vecs_page, r = e % vecs_page;
            const int t = r / VPR, d = r % VPR;
            const uint4 *src = which ? v : k;
            uint4 *dst = which ? packed_v : packed_k;
            uint4 val[kGatherPagesPerPass];
#pragma unroll
            for (int j = 0; j < kGatherPagesPerPass; ++j)
                val[j] = src_page[j] >= 0
                             ? __ldg(src + src_page[j] * block_stride + t * token_stride + head_off + d)
                             : qnan;
#pragma unroll
            for (int j = 0; j < kGatherPagesPerPass; ++j)
                if (src_page[j] >= -1)
                    dst[(c0 + j) * vecs_page + r] = val[j];
        }
    }
}

cudaError_t launch_gather_kv_head(const void *k, const void *v, int64_t num_blocks, int64_t block_stride,
                                  int64_t token_stride, int64_t head_stride, int32_t kv_head, int32_t head_dim,
                                  const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens,
                                  int32_t num_seqs, void *packed_k, void *packed_v, int64_t capacity_pages,
                                  int32_t *compact_tables, int32_t *compact_offsets, ErrState *err,
                                  cudaStream_t stream, int num_sms)
{
    // pages of the largest batch the bounds allow, at most one wave of
    // resident CTAs (no tail wave)
    const int64_t max_pages = (int64_t)num_seqs * max_blocks;
    int64_t grid = (max_pages + kGatherPagesPerPass - 1) / kGatherPagesPerPass;
    void (*kern)(const uint4 *, const uint4 *, int64_t, int64_t, int64_t, int64_t, const int32_t *, int32_t,
                 const int32_t *, int32_t, uint4 *, uint4 *, int64_t, int32_t *, int32_t *, ErrState *) =
        head_dim == 128 ? gather_kv_head_kernel<16>
                        : (head_dim == 256 ? gather_kv_head_kernel<32> : gather_kv_head_kernel<64>);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGatherThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 152) * per_sm;
    if (grid > cap)
        grid = cap;
    if (grid < 1)
        grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kGatherThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint4 *>(k),
                              static_cast<const uint4 *>(v), num_blocks, block_stride / 8, token_stride / 8,
                              (int64_t)kv_head * head_stride / 8, block_tables,
                              max_blocks, seq_lens, num_seqs, static_cast<uint4 *>(packed_k),
                              static_cast<uint4 *>(packed_v), capacity_pages, compact_tables, compact_offsets,
                              err);
}

}  // namespace pa

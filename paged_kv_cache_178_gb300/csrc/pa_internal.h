// Internal interface between the C-ABI front end (pa_api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

// Device-side error latch: the first error code and the index it concerns.
struct ErrState {
    unsigned int code;
    unsigned int pad;
    long long index;
};

enum : unsigned int { kErrBadMetadata = 4u, kErrTimeout = 5u, kErrBudget = 3u };

__device__ __forceinline__ void record_error(ErrState *e, unsigned int code, long long index)
{
    if (atomicCAS(&e->code, 0u, code) == 0u)
        atomicExch(reinterpret_cast<unsigned long long *>(&e->index),
                   static_cast<unsigned long long>(index));
}

// Validated, host-side description of one attention call.
struct AttnArgs {
    const void *q;
    int64_t num_q_tokens;
    int64_t q_tok_stride;
    int32_t num_q_heads;
    const void *k;
    const void *v;
    int64_t num_blocks;
    int32_t num_kv_heads;
    int32_t head_dim;
    int64_t block_stride, token_stride, head_stride;
    const int32_t *block_tables;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    const int32_t *query_start_loc;
    int32_t num_seqs;
    int32_t max_query_len;
    int32_t max_seq_len;
    float scale;
    void *out;
    float *lse;
    void *workspace;
    size_t workspace_bytes;
    // The preceding kernel of the stream writes only the K/V pool: the
    // kernel may read everything else before that kernel has finished.
    bool early_reads;
};

// Work decomposition chosen from host scalars only.
struct AttnPlan {
    int head_dim;
    int group;          // Hq / Hkv
    int tokens_per_tile;  // query tokens per 128-row tile
    int qtiles;         // grid extent over query tiles
    int nch;            // grid extent over KV chunks (1 unless split)
    bool split;         // split-KV with partial states + in-kernel merge
    int cpu;            // split-KV: consecutive chunks per CTA (>= 1)
    int cl;             // CTAs per cluster (2: a CTA pair shares each MMA, in-CTA schedule)
    int ws_rows;        // rows per partial-state record
    size_t ws_counter_bytes;
    size_t ws_bytes;    // total workspace needed
    long long grid;     // CTAs (or clusters x 2 for Dh=512)
    int kt;             // keys per KV tile: the fixed arithmetic's tile (64 or 128)
};

bool plan_attention(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                    int32_t head_dim, int32_t max_query_len, int32_t max_seq_len, AttnPlan *plan);

// Launch the attention kernel for a validated call.  Returns a CUDA error
// code; *unsupported is set when the shape has no kernel.
cudaError_t launch_attention(const AttnArgs &a, const AttnPlan &plan, ErrState *err,
                             cudaStream_t stream, char *info, size_t info_len);

cudaError_t init_attention_attributes();

// Limit (ns) of the split-KV fold's cross-CTA wait; the setter returns the
// previous value.
uint64_t fold_wait_limit_ns();
uint64_t set_fold_wait_limit_ns(uint64_t ns);

// Head dim 512: two-CTA clusters (pa_attn512.cu).
cudaError_t init_attention512_attributes();
cudaError_t launch_attention512(const AttnArgs &a, const AttnPlan &plan, ErrState *err, cudaStream_t stream);

// Compact active-block gather of one KV head (pa_gather.cu).
cudaError_t launch_gather_kv_head(const void *k, const void *v, int64_t num_blocks, int64_t block_stride,
                                  int64_t token_stride, int64_t head_stride, int32_t kv_head, int32_t head_dim,
                                  const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens,
                                  int32_t num_seqs, void *packed_k, void *packed_v, int64_t capacity_pages,
                                  int32_t *compact_tables, int32_t *compact_offsets, ErrState *err,
                                  cudaStream_t stream, int num_sms);
constexpr int kGatherMaxSeqsHost = 512;

// Encodes a tiled tensor map (driver entry point fetched at run time).
CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, cuuint32_t rank, void *base,
                      const cuuint64_t *dims, const cuuint64_t *strides_bytes,
                      const cuuint32_t *box, CUtensorMapSwizzle swizzle);

}  // namespace pa

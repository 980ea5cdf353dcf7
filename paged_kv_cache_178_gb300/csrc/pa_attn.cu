// K2: paged grouped-query attention for sm_103a (head dims 128 and 256).
//
// One CTA owns a 128-row tile of (query token, query head) rows of one
// request and one KV head: rows r = t*G + hh are query token t of the tile
// and query head kvh*G + hh, so the G heads sharing a KV head share every
// K/V tile ("test(rocm): ReshapeAndCache->PagedAttention composition at real
// dims", What changed: Hq=8, Hkv=2).  Roles (256 threads):
//   warp 0     TMA producer: Q once, then per 128-key tile one 64-column box
//              per 16-token page for K and for V, block ids read from the
//              request's table; pages past the last needed key are not read
//              ("fix(rocm): stabilize direct paged CK attention for bitwise
//              R/R", Changes: tail-page padding and sanitising).
//   warp 1     tcgen05 issuer: S = Q.K^T into TMEM (double buffered), then
//              O += P.V into TMEM; zeroes V rows of keys past the last needed
//              key so a masked probability never meets a poisoned value.
//   warps 4-7  softmax / correction / epilogue, one thread per row.
//
// Fixed arithmetic (same page, intro and Changes: one schedule for every
// shape, no implicit FMA contraction): every row follows the same sequence
// of operations whatever the batch, query length, other rows or launch
// bounds, so prefill and decode agree bit for bit:
//   C1  KV tiles of 128 keys aligned to key 0; one MMA shape (M=128, K-steps
//       of 16 in ascending order, BF16 in, FP32 accumulate).
//   C2  s2 = S * (scale*log2 e) (one fp32 multiply, product formed on host).
//   C3  lazy online softmax over a chunk's tiles: the reference max m moves
//       only when a tile max exceeds m + 8 (then l and O are scaled by
//       exp2(m_old - m_new)); p = exp2(s2 - m) for allowed keys, exactly 0
//       otherwise; the tile's row sum is a fixed 8-way interleaved sum.
//   C4  P rounded to BF16 (RNE) before P.V.
//   C5  head dim 128: chunks of 256 keys aligned to key 0, each starting
//       fresh; chunk states fold left to right with one fold function
//       (in-CTA for prefill, by the last-arriving CTA for split decode).
//       Head dim 256: one chunk (no split).
//   C6  out = O * rcp_rn(l) -> BF16 RNE; lse = (m + log2 l) * ln 2.
#include <cuda_bf16.h>
#include <cstdio>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kRows = 128;          // M of every MMA: rows per tile
constexpr int kKeys = 128;          // keys per KV tile
constexpr float kTau = 8.0f;        // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kSplitCtaThreshold = 152;

template <int DH>
struct Cfg;
template <>
struct Cfg<128> {
    static constexpr int kStages = 2;      // K/V smem stages
    static constexpr int kPBufs = 2;       // P smem buffers
    static constexpr int kChunk = 256;     // keys per chunk (0 = one chunk)
    static constexpr int kOCol = 256;      // TMEM column of the chunk accumulator
    static constexpr int kAccCol = 384;    // TMEM column of the folded accumulator
};
template <>
struct Cfg<256> {
    static constexpr int kStages = 1;
    static constexpr int kPBufs = 1;
    static constexpr int kChunk = 0;
    static constexpr int kOCol = 256;
    static constexpr int kAccCol = -1;
};

template <int DH>
constexpr size_t smem_bytes()
{
    return 1024 /*align slack*/ + (size_t)(DH / 64) * 16384 * (1 + 2 * Cfg<DH>::kStages) +
           (size_t)Cfg<DH>::kPBufs * 32768 + 256 /*barriers and flags*/;
}

struct AttnParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    const int32_t *qsl;
    __nv_bfloat16 *out;
    float *lse;
    float *ws_part;
    uint32_t *ws_cnt;
    ErrState *err;
    int64_t num_q_tokens;
    int64_t num_blocks;
    int32_t max_blocks;
    int32_t num_seqs;
    int32_t hq, hkv, group, tq, qtiles, nch;
    int32_t max_query_len, max_seq_len;
    int32_t ws_rows;
    int32_t split;
    float scale_log2;
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Fold of two softmax states (m, l, O) -- C5.  A state with m = -inf holds
// no key: folding it in leaves the other side unchanged, and folding into it
// takes the other side verbatim.
struct Fold {
    float m, l, sa, sc;
    int mode;  // 0: keep a, 1: take c, 2: mix
};

__device__ __forceinline__ Fold fold_coef(float ma, float la, float mc, float lc)
{
    Fold f;
    if (mc == -INFINITY) {
        f.m = ma; f.l = la; f.sa = 1.f; f.sc = 0.f; f.mode = 0;
    } else if (ma == -INFINITY) {
        f.m = mc; f.l = lc; f.sa = 0.f; f.sc = 1.f; f.mode = 1;
    } else {
        f.m = fmaxf(ma, mc);
        f.sa = ex2(__fsub_rn(ma, f.m));
        f.sc = ex2(__fsub_rn(mc, f.m));
        f.l = __fadd_rn(__fmul_rn(la, f.sa), __fmul_rn(lc, f.sc));
        f.mode = 2;
    }
    return f;
}

__device__ __forceinline__ float fold_elem(float oa, float oc, const Fold &f)
{
    return f.mode == 0 ? oa : (f.mode == 1 ? oc : __fadd_rn(__fmul_rn(oa, f.sa), __fmul_rn(oc, f.sc)));
}

__device__ __forceinline__ float lse_of(float m, float l)
{
    return __fmul_rn(__fadd_rn(m, __log2f(l)), kLn2);
}

// Bounded mbarrier wait.  Gives up when another thread of the CTA already
// gave up (abort flag) or after kWaitLimitNs, latching PA_ERR_TIMEOUT.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      ErrState *err)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            record_error(err, kErrTimeout, -1);
            return false;
        }
    }
}

// Wait without the abort shortcut (used to drain in-flight work on exit).
__device__ __noinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    return true;
}

__device__ __forceinline__ void named_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Store 32 consecutive output values (fp32, already normalised) as BF16.
__device__ __forceinline__ void store_out32(__nv_bfloat16 *dst, const float (&v)[32])
{
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        d[i] = make_uint4(pack_bf16x2(v[8 * i + 0], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                          pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
}

template <int DH>
__device__ void write_nan_rows(const AttnParams &p, int64_t tok_first, int ntok, int kvh, int tid,
                               int nthreads)
{
    const __nv_bfloat16 qnan = __ushort_as_bfloat16(0x7FC0);
    const int G = p.group;
    const int64_t total = (int64_t)ntok * G * DH;
    for (int64_t e = tid; e < total; e += nthreads) {
        const int64_t row = e / DH;
        const int d = (int)(e % DH);
        const int64_t t = tok_first + row / G;
        const int h = kvh * G + (int)(row % G);
        p.out[(t * p.hq + h) * DH + d] = qnan;
        if (d == 0 && p.lse)
            p.lse[t * p.hq + h] = __int_as_float(0x7FC00000);
    }
}

// Last-arriving CTA of a split (request, KV head, query tile) folds the
// chunk partial states left to right and writes out / lse -- C5, C6.
template <int DH>
__device__ void merge_partials(const AttnParams &p, const float *part0, int64_t unit_stride,
                               int nchunks, int rows_valid, int64_t tok_first, int kvh, int tid,
                               int nthreads)
{
    const int R = p.ws_rows;
    const int G = p.group;
    for (int e = tid; e < rows_valid * DH; e += nthreads) {
        const int d = e / rows_valid;
        const int row = e % rows_valid;
        float ma = -INFINITY, la = 0.f, oa = 0.f;
        for (int c = 0; c < nchunks; ++c) {
            const float *pc = part0 + (int64_t)c * unit_stride;
            const float mc = __ldcg(pc + row);
            const float lc = __ldcg(pc + R + row);
            const float oc = __ldcg(pc + 2 * R + (int64_t)d * R + row);
            const Fold f = fold_coef(ma, la, mc, lc);
            oa = fold_elem(oa, oc, f);
            ma = f.m;
            la = f.l;
        }
        const int64_t t = tok_first + row / G;
        const int h = kvh * G + row % G;
        p.out[(t * p.hq + h) * DH + d] = __float2bfloat16_rn(__fmul_rn(oa, __frcp_rn(la)));
        if (d == 0 && p.lse)
            p.lse[t * p.hq + h] = lse_of(ma, la);
    }
}

template <int DH>
__device__ void arrive_and_maybe_merge(const AttnParams &p, int b, int kvh, int qt, int nchunks,
                                       int rows_valid, int64_t tok_first, int r, int *flag_last)
{
    __threadfence();
    named_sync(1, 128);
    const int64_t unit_q = ((int64_t)b * p.hkv + kvh) * p.qtiles + qt;
    if (r == 0) {
        const uint32_t old = atomicAdd(p.ws_cnt + unit_q, 1u);
        const int last = (old == (uint32_t)(nchunks - 1));
        if (last)
            p.ws_cnt[unit_q] = 0u;  // leave the workspace ready for the next call
        *flag_last = last;
    }
    named_sync(1, 128);
    if (*flag_last) {
        __threadfence();
        const int64_t unit_stride = (int64_t)p.ws_rows * (DH + 2);
        const float *part0 = p.ws_part + unit_q * p.nch * unit_stride;
        merge_partials<DH>(p, part0, unit_stride, nchunks, rows_valid, tok_first, kvh, r, 128);
    }
}

template <int DH>
__global__ void __launch_bounds__(256, 1) attn_kernel(const __grid_constant__ AttnParams p)
{
    using C = Cfg<DH>;
    constexpr int NKB = DH / 64;            // 64-column (128-byte) blocks of the head dim
    constexpr int TILE_BYTES = NKB * 16384;  // 128 rows (or keys) x DH BF16
    constexpr int NST = C::kStages;
    constexpr int NP = C::kPBufs;
    constexpr bool CHUNKED = C::kChunk > 0;
    constexpr int CHUNK_DIV = CHUNKED ? C::kChunk : 1;  // divisor used only when CHUNKED
    constexpr uint32_t ACC_COL = C::kAccCol < 0 ? 0u : (uint32_t)C::kAccCol;
    constexpr uint32_t ID_QK = idesc_bf16_f32(kRows, kKeys, false);
    constexpr uint32_t ID_PV = idesc_bf16_f32(kRows, DH, true);
    // barrier slots
    constexpr int B_Q = 0, B_KF = 1, B_VF = B_KF + NST, B_KE = B_VF + NST, B_VE = B_KE + NST;
    constexpr int B_SF = B_VE + NST, B_SE = B_SF + 2, B_PF = B_SE + 2, B_PV = B_PF + NP;
    constexpr int B_OF = B_PV + NP, B_DONE = B_OF + 1, NBARS = B_DONE + 1;
    static_assert(NBARS * 8 + 32 <= 256, "barrier area");

    // ---------------------------------------------------------- work unit --
    long long u = blockIdx.x;
    const int c_grid = (int)(u % p.nch);
    u /= p.nch;
    const int qt = (int)(u % p.qtiles);
    u /= p.qtiles;
    const int kvh = (int)(u % p.hkv);
    const int b = (int)(u / p.hkv);
    const int tid = threadIdx.x;
    if (b >= p.num_seqs)
        return;
    const int qs = p.qsl[b], qe = p.qsl[b + 1], L = p.seq_lens[b];
    const int qn = qe - qs;
    const bool rows_sane = qs >= 0 && qn >= 0 && (int64_t)qe <= p.num_q_tokens;
    const bool meta_ok = rows_sane && L >= qn && (int64_t)L <= (int64_t)p.max_blocks * 16 &&
                         qn <= p.max_query_len && L <= p.max_seq_len;
    const int tok0 = qt * p.tq;
    if (!meta_ok) {
        if (qt == 0 && c_grid == 0 && tid == 0)
            record_error(p.err, kErrBadMetadata, b);
        if (rows_sane && c_grid == 0 && tok0 < qn)
            write_nan_rows<DH>(p, (int64_t)qs + tok0, min(p.tq, qn - tok0), kvh, tid, blockDim.x);
        return;
    }
    if (tok0 >= qn)
        return;
    const int ntok = min(p.tq, qn - tok0);
    const int rows_valid = ntok * p.group;
    const int64_t tok_first = (int64_t)qs + tok0;
    const int kend = L - qn + tok0 + ntok;  // keys [0, kend) are needed by some row
    const int nchunks = CHUNKED ? (kend + CHUNK_DIV - 1) / CHUNK_DIV : 1;
    int kbeg = 0, kstop = kend;
    if (p.split) {
        if (c_grid >= nchunks)
            return;
        kbeg = c_grid * CHUNK_DIV;
        kstop = min(kbeg + CHUNK_DIV, kend);
    }
    const int t_begin = kbeg / kKeys;
    const int t_end = (kstop + kKeys - 1) / kKeys;
    const int n_it = t_end - t_begin;
    const int npages_need = (kend + 15) / 16;
    const int32_t *bt_row = p.block_tables + (int64_t)b * p.max_blocks;

    // Every block id this CTA will use must be inside the pool.
    int bad = 0;
    {
        const int pg_end = min(t_end * 8, npages_need);
        for (int pg = t_begin * 8 + tid; pg < pg_end; pg += blockDim.x) {
            const int id = bt_row[pg];
            bad |= (id < 0 || (int64_t)id >= p.num_blocks);
        }
    }
    bad = __syncthreads_or(bad);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem;
    uint8_t *sK = sQ + TILE_BYTES;
    uint8_t *sV = sK + NST * TILE_BYTES;
    uint8_t *sP = sV + NST * TILE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sP + NP * 32768);
    int *sflags = reinterpret_cast<int *>(bars + NBARS);  // [0] abort [1] tmem [2] last
    volatile int *abort_flag = sflags;
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    const int warp = tid / 32, lane = tid % 32;
    const int unit_stride_f = p.ws_rows * (DH + 2);

    if (bad) {
        if (tid == 0)
            record_error(p.err, kErrBadMetadata, b);
        if (!p.split) {
            write_nan_rows<DH>(p, tok_first, ntok, kvh, tid, blockDim.x);
            return;
        }
        if (warp < 4)
            return;
        const int r = tid - 128;
        const int64_t unit_q = ((int64_t)b * p.hkv + kvh) * p.qtiles + qt;
        float *part = p.ws_part + (unit_q * p.nch + c_grid) * unit_stride_f;
        if (r < rows_valid) {
            part[r] = 0.f;
            part[p.ws_rows + r] = __int_as_float(0x7FC00000);
            for (int d = 0; d < DH; ++d)
                part[2 * p.ws_rows + d * p.ws_rows + r] = __int_as_float(0x7FC00000);
        }
        arrive_and_maybe_merge<DH>(p, b, kvh, qt, nchunks, rows_valid, tok_first, r, &sflags[2]);
        return;
    }

    // -------------------------------------------------------------- setup --
    if (tid == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar(B_KF + s), 1);
            mbar_init(bar(B_VF + s), 1);
            mbar_init(bar(B_KE + s), 1);
            mbar_init(bar(B_VE + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_SF + i), 1);
            mbar_init(bar(B_SE + i), 4);
        }
        for (int i = 0; i < NP; ++i) {
            mbar_init(bar(B_PF + i), 4);
            mbar_init(bar(B_PV + i), 1);
        }
        mbar_init(bar(B_OF), 4);
        mbar_init(bar(B_DONE), 1);
        sflags[0] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&sflags[1]), 512);
        tmem_relinquish();
    }
    if (tid == 32 * 2) {
        prefetch_tensormap(&p.tm_q);
        prefetch_tensormap(&p.tm_k);
        prefetch_tensormap(&p.tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(sflags[1]);

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        bool ok = true;
        int last_k_use[NST], last_v_use[NST];
        for (int s = 0; s < NST; ++s) last_k_use[s] = last_v_use[s] = -1;
        if (lane == 0) {
            // Q box: 64 columns x G heads x tq tokens per 64-column block
            mbar_arrive_expect_tx(bar(B_Q), NKB * 128 * p.group * p.tq);
            for (int kb = 0; kb < NKB; ++kb)
                tma_load_3d(smem_addr(sQ + kb * 16384), &p.tm_q, bar(B_Q), kb * 64, kvh * p.group,
                            (int)tok_first);
        }
        int id_next = (lane < 8 && t_begin * 8 + lane < npages_need) ? bt_row[t_begin * 8 + lane] : 0;
        for (int it = 0; ok && it < n_it; ++it) {
            const int t = t_begin + it;
            const int id_cur = id_next;
            id_next = (it + 1 < n_it && lane < 8 && (t + 1) * 8 + lane < npages_need)
                          ? bt_row[(t + 1) * 8 + lane]
                          : 0;
            const int s = it % NST, use = it / NST;
            const int np = min(8, npages_need - t * 8);
            int ids[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) ids[i] = __shfl_sync(0xffffffffu, id_cur, i);
            if (lane == 0) {
                if (use >= 1)
                    ok = wait_bar(bar(B_KE + s), (use - 1) & 1, abort_flag, p.err);
                if (ok) {
                    mbar_arrive_expect_tx(bar(B_KF + s), np * NKB * 2048);
                    for (int i = 0; i < np; ++i)
                        for (int kb = 0; kb < NKB; ++kb)
                            tma_load_4d(smem_addr(sK + s * TILE_BYTES + kb * 16384 + i * 2048), &p.tm_k,
                                        bar(B_KF + s), kb * 64, kvh, 0, ids[i]);
                    last_k_use[s] = use;
                }
                if (ok && use >= 1)
                    ok = wait_bar(bar(B_VE + s), (use - 1) & 1, abort_flag, p.err);
                if (ok) {
                    mbar_arrive_expect_tx(bar(B_VF + s), np * NKB * 2048);
                    for (int i = 0; i < np; ++i)
                        for (int kb = 0; kb < NKB; ++kb)
                            tma_load_4d(smem_addr(sV + s * TILE_BYTES + kb * 16384 + i * 2048), &p.tm_v,
                                        bar(B_VF + s), kb * 64, kvh, 0, ids[i]);
                    last_v_use[s] = use;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        if (!ok && lane == 0) {
            // Let issued copies land before the CTA's shared memory goes away.
            for (int s = 0; s < NST; ++s) {
                if (last_k_use[s] >= 0)
                    wait_bar_drain(bar(B_KF + s), last_k_use[s] & 1);
                if (last_v_use[s] >= 0)
                    wait_bar_drain(bar(B_VF + s), last_v_use[s] & 1);
            }
            wait_bar_drain(bar(B_Q), 0);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer --
        bool ok = true;
        if (lane == 0)
            ok = wait_bar(bar(B_Q), 0, abort_flag, p.err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        auto issue_pv = [&](int j) -> bool {
            const int s = j % NST;
            const int t = t_begin + j;
            bool okj = wait_bar(bar(B_VF + s), (j / NST) & 1, abort_flag, p.err);
            okj = __all_sync(0xffffffffu, okj);
            if (!okj)
                return false;
            if ((t + 1) * kKeys > kend) {
                // keys >= kend: zero their V rows (stale or poisoned data)
                const int row0 = kend - t * kKeys;
                const int nz = (kKeys - row0) * NKB * 8;
                uint8_t *vs = sV + s * TILE_BYTES;
                for (int idx = lane; idx < nz; idx += 32) {
                    const int row = row0 + idx / (NKB * 8);
                    const int rem = idx % (NKB * 8);
                    *reinterpret_cast<uint4 *>(vs + (rem / 8) * 16384 + row * 128 + (rem % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) {
                okj = wait_bar(bar(B_PF + j % NP), (j / NP) & 1, abort_flag, p.err);
                const bool chunk_first = CHUNKED ? ((t * kKeys) % CHUNK_DIV == 0) : (j == 0);
                const int k = CHUNKED ? (t * kKeys - kbeg) / CHUNK_DIV : 0;
                if (okj && chunk_first && k > 0)
                    okj = wait_bar(bar(B_OF), (k - 1) & 1, abort_flag, p.err);
                if (okj) {
                    tc_fence_after();
                    const uint32_t pbase = smem_addr(sP + (j % NP) * 32768);
                    const uint32_t vbase = smem_addr(sV + s * TILE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk) {
                        const uint64_t a = sdesc_sw128(pbase + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(vbase + kk * 2048, 16384, 1024);
                        mma_bf16_ss(tmem + C::kOCol, a, bd, ID_PV, (kk > 0 || !chunk_first) ? 1u : 0u);
                    }
                    mma_commit(bar(B_VE + s));
                    mma_commit(bar(B_PV + j % NP));
                }
            }
            return __shfl_sync(0xffffffffu, okj, 0);
        };
        for (int it = 0; ok && it <= n_it; ++it) {
            if (it < n_it) {
                const int s = it % NST;
                if (lane == 0) {
                    ok = wait_bar(bar(B_KF + s), (it / NST) & 1, abort_flag, p.err);
                    if (ok && it >= 2)
                        ok = wait_bar(bar(B_SE + (it & 1)), ((it >> 1) - 1) & 1, abort_flag, p.err);
                    if (ok) {
                        tc_fence_after();
                        const uint32_t qbase = smem_addr(sQ);
                        const uint32_t kbase = smem_addr(sK + s * TILE_BYTES);
#pragma unroll
                        for (int kk = 0; kk < DH / 16; ++kk) {
                            const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                            mma_bf16_ss(tmem + (it & 1) * kKeys, sdesc_sw128(qbase + off, 16, 1024),
                                        sdesc_sw128(kbase + off, 16, 1024), ID_QK, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bar(B_KE + s));
                        mma_commit(bar(B_SF + (it & 1)));
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
            if (ok && it >= 1)
                ok = issue_pv(it - 1);
        }
        // all MMAs retired before TMEM is released
        if (lane == 0) {
            mma_commit(bar(B_DONE));
            wait_bar_drain(bar(B_DONE), 0);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------ softmax / epilogue WG --
        const int r = tid - 128;
        const int wq = warp - 4;
        const uint32_t lane_off = static_cast<uint32_t>(32 * wq) << 16;
        const bool row_valid = r < rows_valid;
        const bool warp_active = 32 * wq < rows_valid;
        const int G = p.group;
        const int pos = L - qn + tok0 + r / G;
        const int64_t tok = tok_first + r / G;
        const int head = kvh * G + r % G;
        float m = -INFINITY, l = 0.f, m_acc = -INFINITY, l_acc = 0.f;
        int nfold = 0;
        bool ok = true;
        for (int it = 0; ok && it < n_it; ++it) {
            const int t = t_begin + it;
            const int sb = it & 1, pb = it % NP;
            ok = wait_bar(bar(B_SF + sb), (it >> 1) & 1, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            float s[kKeys];
            if (warp_active) {
                uint32_t v[32];
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) {
                    tmem_ld32(tmem + lane_off + sb * kKeys + g4 * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[g4 * 32 + i] = __uint_as_float(v[i]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_SE + sb));
            float m_new = m, corr = 1.f, tsum = 0.f;
            bool need = false;
            if (warp_active) {
                const int nallow = row_valid ? max(0, min(kKeys, pos - t * kKeys + 1)) : 0;
                float tmax = -INFINITY;
#pragma unroll
                for (int c = 0; c < kKeys; ++c) {
                    s[c] = __fmul_rn(s[c], p.scale_log2);
                    tmax = (c < nallow) ? fmaxf(tmax, s[c]) : tmax;
                }
                if (tmax != -INFINITY) {
                    if (m == -INFINITY) {
                        m_new = tmax;
                    } else if (tmax > __fadd_rn(m, kTau)) {
                        m_new = tmax;
                        corr = ex2(__fsub_rn(m, m_new));
                        need = true;
                    }
                }
                float acc8[8];
#pragma unroll
                for (int c = 0; c < kKeys; ++c) {
                    const float e = (c < nallow) ? ex2(__fsub_rn(s[c], m_new)) : 0.f;
                    s[c] = e;
                    if (c < 8)
                        acc8[c] = e;
                    else
                        acc8[c & 7] = __fadd_rn(acc8[c & 7], e);
                }
                tsum = __fadd_rn(__fadd_rn(__fadd_rn(acc8[0], acc8[1]), __fadd_rn(acc8[2], acc8[3])),
                                 __fadd_rn(__fadd_rn(acc8[4], acc8[5]), __fadd_rn(acc8[6], acc8[7])));
            }
            // P buffer pb is free once PV(it - NP) has completed
            if (it >= NP) {
                ok = wait_bar(bar(B_PV + pb), ((it / NP) - 1) & 1, abort_flag, p.err);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            }
            if (warp_active) {
                uint8_t *prow = sP + pb * 32768 + r * 128;
#pragma unroll
                for (int c8 = 0; c8 < kKeys / 8; ++c8) {
                    const int kb = c8 / 8, ch = c8 % 8;
                    const uint4 w = make_uint4(pack_bf16x2(s[c8 * 8 + 0], s[c8 * 8 + 1]),
                                               pack_bf16x2(s[c8 * 8 + 2], s[c8 * 8 + 3]),
                                               pack_bf16x2(s[c8 * 8 + 4], s[c8 * 8 + 5]),
                                               pack_bf16x2(s[c8 * 8 + 6], s[c8 * 8 + 7]));
                    *reinterpret_cast<uint4 *>(prow + kb * 16384 + ((ch ^ (r & 7)) << 4)) = w;
                }
                fence_proxy_async_smem();
            }
            if (__any_sync(0xffffffffu, need)) {
                // O of this chunk must hold PV(it - 1) before it is rescaled
                ok = wait_bar(bar(B_PV + (it - 1) % NP), ((it - 1) / NP) & 1, abort_flag, p.err);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                const float f = need ? corr : 1.f;
#pragma unroll 1
                for (int g = 0; g < DH / 32; ++g) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + C::kOCol + g * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__fmul_rn(__uint_as_float(v[i]), f));
                    tmem_st32(tmem + lane_off + C::kOCol + g * 32, v);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_PF + pb));
            l = need ? __fadd_rn(__fmul_rn(l, corr), tsum) : __fadd_rn(l, tsum);
            m = m_new;

            const bool final_tile = (it == n_it - 1);
            const bool chunk_end = final_tile || (CHUNKED && ((t + 1) * kKeys) % CHUNK_DIV == 0);
            if (!chunk_end)
                continue;
            ok = wait_bar(bar(B_PV + pb), (it / NP) & 1, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            if (p.split) {
                // partial state of this CTA's chunk
                const int64_t unit_q = ((int64_t)b * p.hkv + kvh) * p.qtiles + qt;
                float *part = p.ws_part + (unit_q * p.nch + c_grid) * unit_stride_f;
                const int R = p.ws_rows;
                if (row_valid) {
                    part[r] = m;
                    part[R + r] = l;
                }
#pragma unroll 1
                for (int g = 0; g < DH / 32; ++g) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + C::kOCol + g * 32, v);
                    tmem_wait_ld();
                    if (row_valid) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            __stcg(part + 2 * R + (int64_t)(g * 32 + i) * R + r, __uint_as_float(v[i]));
                    }
                }
            } else if (final_tile) {
                // epilogue: out = fold(acc, chunk) / l
                const Fold f = (nfold == 0) ? fold_coef(-INFINITY, 0.f, m, l) : fold_coef(m_acc, l_acc, m, l);
                const float inv = __frcp_rn(f.l);
#pragma unroll 1
                for (int g = 0; g < DH / 32; ++g) {
                    uint32_t vc[32], va[32];
                    tmem_ld32(tmem + lane_off + C::kOCol + g * 32, vc);
                    if (nfold > 0)
                        tmem_ld32(tmem + lane_off + ACC_COL + g * 32, va);
                    tmem_wait_ld();
                    float o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float oa = (nfold > 0) ? __uint_as_float(va[i]) : 0.f;
                        o[i] = __fmul_rn(fold_elem(oa, __uint_as_float(vc[i]), f), inv);
                    }
                    if (row_valid)
                        store_out32(p.out + (tok * p.hq + head) * DH + g * 32, o);
                }
                if (row_valid && p.lse)
                    p.lse[tok * p.hq + head] = lse_of(f.m, f.l);
            } else {
                // fold this chunk into the running accumulator (TMEM)
                const Fold f = (nfold == 0) ? fold_coef(-INFINITY, 0.f, m, l) : fold_coef(m_acc, l_acc, m, l);
#pragma unroll 1
                for (int g = 0; g < DH / 32; ++g) {
                    uint32_t vc[32], va[32];
                    tmem_ld32(tmem + lane_off + C::kOCol + g * 32, vc);
                    if (nfold > 0)
                        tmem_ld32(tmem + lane_off + ACC_COL + g * 32, va);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float oa = (nfold > 0) ? __uint_as_float(va[i]) : 0.f;
                        va[i] = __float_as_uint(fold_elem(oa, __uint_as_float(vc[i]), f));
                    }
                    tmem_st32(tmem + lane_off + ACC_COL + g * 32, va);
                }
                tmem_wait_st();
                m_acc = f.m;
                l_acc = f.l;
                ++nfold;
            }
            tc_fence_before();
            __syncwarp();
            if (!final_tile && lane == 0)
                mbar_arrive(bar(B_OF));
            m = -INFINITY;
            l = 0.f;
        }
        if (p.split && ok)
            arrive_and_maybe_merge<DH>(p, b, kvh, qt, nchunks, rows_valid, tok_first, r, &sflags[2]);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host --

bool plan_attention(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t max_query_len, int32_t max_seq_len, AttnPlan *plan)
{
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads ||
        max_query_len < 0 || max_seq_len < 0)
        return false;
    const int G = num_q_heads / num_kv_heads;
    if (G > kRows)
        return false;
    if (head_dim != 128 && head_dim != 256 && head_dim != 512)
        return false;
    AttnPlan pl{};
    pl.head_dim = head_dim;
    pl.group = G;
    pl.tokens_per_tile = kRows / G;
    pl.qtiles = max_query_len > 0 ? (max_query_len + pl.tokens_per_tile - 1) / pl.tokens_per_tile : 0;
    const int chunk = head_dim == 128 ? Cfg<128>::kChunk : 0;
    const long long full_ctas = (long long)num_seqs * num_kv_heads * pl.qtiles;
    pl.split = chunk > 0 && max_seq_len > chunk && full_ctas < kSplitCtaThreshold;
    pl.nch = pl.split ? (max_seq_len + chunk - 1) / chunk : 1;
    pl.ws_rows = G * (max_query_len < pl.tokens_per_tile ? max_query_len : pl.tokens_per_tile);
    pl.ws_counter_bytes = 0;
    pl.ws_bytes = 0;
    if (pl.split) {
        const size_t units_q = (size_t)full_ctas;
        pl.ws_counter_bytes = ((units_q * 4 + 255) / 256) * 256;
        pl.ws_bytes = pl.ws_counter_bytes + units_q * pl.nch * (size_t)pl.ws_rows * (head_dim + 2) * 4;
    }
    pl.grid = full_ctas * pl.nch;
    *plan = pl;
    return true;
}

cudaError_t init_attention_attributes()
{
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<128>());
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(attn_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<256>());
}

template <int DH>
static cudaError_t launch_dh(const AttnArgs &a, const AttnPlan &pl, ErrState *err, cudaStream_t stream)
{
    AttnParams p;
    memset(&p, 0, sizeof(p));
    const int G = pl.group;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)DH, (cuuint64_t)a.num_q_heads, (cuuint64_t)a.num_q_tokens};
        const cuuint64_t strides[2] = {(cuuint64_t)DH * 2, (cuuint64_t)a.q_tok_stride * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)pl.tokens_per_tile};
        if (encode_tiled(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {(cuuint64_t)DH, (cuuint64_t)a.num_kv_heads, 16, (cuuint64_t)a.num_blocks};
        const cuuint64_t strides[3] = {(cuuint64_t)a.head_stride * 2, (cuuint64_t)a.token_stride * 2,
                                       (cuuint64_t)a.block_stride * 2};
        const cuuint32_t box[4] = {64, 1, 16, 1};
        if (encode_tiled(&p.tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(a.k), dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        if (encode_tiled(&p.tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(a.v), dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    p.block_tables = a.block_tables;
    p.seq_lens = a.seq_lens;
    p.qsl = a.query_start_loc;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    p.ws_cnt = static_cast<uint32_t *>(a.workspace);
    p.ws_part = pl.split ? reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) + pl.ws_counter_bytes)
                         : nullptr;
    p.err = err;
    p.num_q_tokens = a.num_q_tokens;
    p.num_blocks = a.num_blocks;
    p.max_blocks = a.max_blocks_per_seq;
    p.num_seqs = a.num_seqs;
    p.hq = a.num_q_heads;
    p.hkv = a.num_kv_heads;
    p.group = G;
    p.tq = pl.tokens_per_tile;
    p.qtiles = pl.qtiles;
    p.nch = pl.nch;
    p.max_query_len = a.max_query_len;
    p.max_seq_len = a.max_seq_len;
    p.ws_rows = pl.ws_rows;
    p.split = pl.split ? 1 : 0;
    // C2: scale * log2(e) formed once, in fp32, on the host
    p.scale_log2 = a.scale * 1.4426950408889634f;
    attn_kernel<DH><<<(unsigned)pl.grid, 256, smem_bytes<DH>(), stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_attention(const AttnArgs &a, const AttnPlan &pl, ErrState *err, cudaStream_t stream,
                             char *info, size_t info_len)
{
    if (info && info_len)
        snprintf(info, info_len, "attention dh=%d schedule=%s grid=%lld qtiles=%d chunks=%d kv_tile=%d chunk=%d",
                 pl.head_dim, pl.split ? "split-kv" : "in-cta", pl.grid, pl.qtiles, pl.nch, kKeys,
                 pl.head_dim == 128 ? Cfg<128>::kChunk : 0);
    if (pl.grid == 0)
        return cudaSuccess;
    switch (a.head_dim) {
    case 128: return launch_dh<128>(a, pl, err, stream);
    case 256: return launch_dh<256>(a, pl, err, stream);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace pa

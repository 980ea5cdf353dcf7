// Split-KV pieces of the attention kernels that split a request's keys over
// several CTAs: the partial-state record layout (pa_attn.cu and pa_decode.cu),
// and for the 128-row kernel (pa_attn.cu) the compacted unit schedule and the
// arrival + left-to-right fold of the chunk states (C5, C6).
#pragma once
#include "pa_attn_common.cuh"

namespace pa {

// Split-KV partial-state record of one chunk (fp32): m[R], l[R] padded to a
// multiple of 4 floats, then O[R][DH] row-major (unnormalised).
__host__ __device__ constexpr int64_t part_header_floats(int R) { return (2 * R + 3) / 4 * 4; }
__host__ __device__ constexpr int64_t part_record_floats(int R, int DH)
{
    return part_header_floats(R) + (int64_t)R * DH;
}

// Arrival on the (request, KV head, query tile) counter and the fold of the
// chunk partial states, left to right (C5, C6).  All threads of the CTA take
// part; `work` is shared memory the pipeline no longer uses.
//
// With `multi` (every unit of the grid is resident at once: units <= SMs, one
// CTA per SM) the last kMergers CTAs to arrive share the fold: CTA m of them
// folds columns [m*DH/K, (m+1)*DH/K) of every row.  Each first waits (bounded)
// until the whole group has arrived; they are the only CTAs that wait, and
// every CTA they wait for already holds an SM.  Otherwise the last CTA to
// arrive folds every column.  The fold is staged: a segment of records is
// copied to shared memory in one pass, the per-row coefficient chain
// (fold_coef) runs once per row, then every element applies fold_elem in
// chunk order -- the same operations, in the same order, as the in-CTA fold.
constexpr int kMergers = 4;

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *ptr)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

template <int DH>
__device__ __forceinline__ void split_arrive_and_merge(const AttnParams &p, int64_t unit_q, int nchunks,
                                       int narrive, int rv, int64_t tok_first, int kvh, float *work,
                                       int work_floats, int *flag_merger, bool multi)
{
    // narrive: CTAs of the group (each brings ceil-divided consecutive
    // chunks); nchunks: chunk records to fold
    const int tid = threadIdx.x, nth = blockDim.x;
    const int K = (multi && narrive >= kMergers) ? kMergers : 1;
    if (tid == 0) {
        // acquire-release at GPU scope: releases this CTA's partial record
        // (written before the CTA barrier that precedes this call) and, for
        // the last arrival, acquires every other CTA's
        uint32_t old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(old)
                     : "l"(p.ws_cnt + unit_q)
                     : "memory");
        int merger = (int)old - (narrive - K);  // < 0: not one of the last K
        if (merger >= K)
            merger = -1;  // a counter left over by a failed call: fold nothing
        if (merger >= 0 && K > 1) {
            // wait for the rest of the group: once the counter reaches
            // narrive every partial record is visible (the acquire reads the
            // end of the release sequence formed by the arrivals)
            if (merger < K - 1) {
                // bounded by p.fold_wait_ns; a limit of 0 gives up without
                // polling (nothing is in flight here: no copy, no MMA)
                const uint64_t t0 = global_timer_ns();
                while (p.fold_wait_ns == 0 || ld_acquire_u32(p.ws_cnt + unit_q) < (uint32_t)narrive) {
                    if (p.fold_wait_ns == 0 || global_timer_ns() - t0 > p.fold_wait_ns) {
                        record_error(p.err, kErrTimeout, ((long long)blockIdx.x << 8) | 0xFF);
                        merger = -1;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            // leave: the last of the K to pass its wait returns the counter
            // to zero for the next call (no CTA reads it after that)
            if (merger >= 0) {
                const uint32_t left = atomicAdd(p.ws_cnt + unit_q, 1u);
                if (left == (uint32_t)(narrive + K - 1))
                    atomicExch(p.ws_cnt + unit_q, 0u);
            }
        } else if (merger >= 0) {
            p.ws_cnt[unit_q] = 0u;  // leave the workspace ready for the next call
        }
        *flag_merger = merger;
    }
    __syncthreads();
    const int merger = *flag_merger;
    if (merger < 0)
        return;
    constexpr int kColsAll = DH;
    const int ncol = kColsAll / K;   // columns this CTA folds
    const int col0 = merger * ncol;
    const int R = p.ws_rows;
    const int64_t hdr = part_header_floats(R);
    const int64_t ustride = part_record_floats(R, DH);
    const float *part0 = p.ws_part + unit_q * p.nch * ustride;
    const int run_f = (2 * rv + 3) / 4 * 4;
    float *s_acc = work;                 // [rv][ncol] running O (this CTA's columns)
    float *s_run = s_acc + rv * ncol;    // [rv][2] running (m, l)
    float *s_run2 = s_run + run_f;       // [rv][2] (m, l) after the current segment
    float *s_seg = s_run2 + run_f;
    const int per_chunk = rv * (ncol + 5) + 8;
    const int seg = max(1, (work_floats - rv * ncol - 2 * run_f) / per_chunk);
    for (int e = tid; e < rv * ncol; e += nth)
        s_acc[e] = 0.f;
    for (int r = tid; r < rv; r += nth) {
        s_run[2 * r] = -INFINITY;
        s_run[2 * r + 1] = 0.f;
    }
    for (int c0 = 0; c0 < nchunks; c0 += seg) {
        const int cn = min(seg, nchunks - c0);
        float *s_ml = s_seg;                             // [cn][rv][2]
        float *s_o = s_ml + (2 * cn * rv + 3) / 4 * 4;   // [cn][rv][ncol]
        float *s_cf = s_o + cn * rv * ncol;              // [cn][rv][2]
        int *s_md = reinterpret_cast<int *>(s_cf + 2 * cn * rv);  // [cn][rv]
        // (a) stage the segment's records: every copy in flight at once
        for (int i = tid; i < cn * rv * 2; i += nth) {
            const int c = i / (2 * rv), k = i % (2 * rv);
            const int which = k / rv, r = k % rv;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(s_ml + (c * rv + r) * 2 + which)),
                         "l"(part0 + (c0 + c) * ustride + which * R + r)
                         : "memory");
        }
        const int vec_per_row = ncol / 4;
        const int vec_per_chunk = rv * vec_per_row;
        for (int i = tid; i < cn * vec_per_chunk; i += nth) {
            const int c = i / vec_per_chunk, k = i % vec_per_chunk;
            const int r = k / vec_per_row, v4 = k % vec_per_row;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                             smem_addr(s_o + (c * rv + r) * ncol + 4 * v4)),
                         "l"(part0 + (c0 + c) * ustride + hdr + (int64_t)r * DH + col0 + 4 * v4)
                         : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
        // (b) fold coefficients of every (row, chunk).  The running max before
        //     chunk c is the max over the earlier chunks (fmaxf is exact and
        //     a chunk without keys holds -inf), so each (row, chunk) can be
        //     computed on its own; fold_coef's mixing factors depend only on
        //     that max and the chunk's own.
        //     The prefix maxima come from warp scans, one warp per row and
        //     32 chunks per step (max is exact: the grouping changes nothing).
        for (int r = tid / 32; r < rv; r += nth / 32) {
            const int ln = tid % 32;
            float run = s_run[2 * r];
            for (int cb = 0; cb < cn; cb += 32) {
                const int c = cb + ln;
                const float mc = c < cn ? s_ml[(c * rv + r) * 2] : -INFINITY;
                float inc = mc;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float x = __shfl_up_sync(0xffffffffu, inc, o);
                    if (ln >= o)
                        inc = fmaxf(inc, x);
                }
                float excl = __shfl_up_sync(0xffffffffu, inc, 1);
                if (ln == 0)
                    excl = -INFINITY;
                if (c < cn) {
                    const Fold f = fold_coef(fmaxf(run, excl), 0.f, mc, 0.f);
                    s_cf[(c * rv + r) * 2] = f.sa;
                    s_cf[(c * rv + r) * 2 + 1] = f.sc;
                    s_md[c * rv + r] = f.mode;
                }
                run = fmaxf(run, __shfl_sync(0xffffffffu, inc, 31));
            }
        }
        __syncthreads();
        // (c) the sequential parts, in chunk order -- the same operations
        //     fold_coef / fold_elem perform, with no branch inside a chain.
        //     The (m, l) chains run on the last warps, one row per thread;
        //     the O chains on the others, one element per thread and pass.
        //     Each loads the operands of seven chunks before their seven steps.
        const int n_ml = (rv + 31) / 32 * 32;
        const int n_o = nth - n_ml;
        if (tid >= n_o) {
            const int r = tid - n_o;
            if (r < rv) {
                float ma = s_run[2 * r], la = s_run[2 * r + 1];
                for (int cb = 0; cb < cn; cb += 7) {
                    int md7[7];
                    float2 ml7[7], cf7[7];
#pragma unroll
                    for (int k = 0; k < 7; ++k) {
                        const int c = min(cb + k, cn - 1);
                        md7[k] = cb + k < cn ? s_md[c * rv + r] : 0;  // past the last chunk: keep
                        ml7[k] = *reinterpret_cast<const float2 *>(s_ml + (c * rv + r) * 2);
                        cf7[k] = *reinterpret_cast<const float2 *>(s_cf + (c * rv + r) * 2);
                    }
#pragma unroll
                    for (int k = 0; k < 7; ++k) {
                        const float l2 = __fadd_rn(__fmul_rn(la, cf7[k].x), __fmul_rn(ml7[k].y, cf7[k].y));
                        const float m2 = fmaxf(ma, ml7[k].x);
                        la = md7[k] == 1 ? ml7[k].y : (md7[k] == 2 ? l2 : la);
                        ma = md7[k] == 1 ? ml7[k].x : (md7[k] == 2 ? m2 : ma);
                    }
                }
                s_run2[2 * r] = ma;
                s_run2[2 * r + 1] = la;
            }
        } else {
            for (int e = tid; e < rv * ncol; e += n_o) {
                const int r = e / ncol;
                float oa = s_acc[e];
                for (int cb = 0; cb < cn; cb += 7) {
                    float o7[7], a7[7], b7[7];
                    int m7[7];
#pragma unroll
                    for (int k = 0; k < 7; ++k) {
                        const int c = min(cb + k, cn - 1);
                        o7[k] = s_o[c * rv * ncol + e];
                        const float2 cf = *reinterpret_cast<const float2 *>(s_cf + (c * rv + r) * 2);
                        a7[k] = cf.x;
                        b7[k] = cf.y;
                        m7[k] = cb + k < cn ? s_md[c * rv + r] : 0;  // past the last chunk: keep
                    }
#pragma unroll
                    for (int k = 0; k < 7; ++k)
                        oa = fold_elem_sel(oa, o7[k], a7[k], b7[k], m7[k]);
                }
                s_acc[e] = oa;
            }
        }
        __syncthreads();
        for (int r = tid; r < rv; r += nth) {
            s_run[2 * r] = s_run2[2 * r];
            s_run[2 * r + 1] = s_run2[2 * r + 1];
        }
        __syncthreads();
    }
    // (d) epilogue
    const int G = p.group;
    for (int e = tid; e < rv * ncol; e += nth) {
        const int r = e / ncol, d = col0 + e % ncol;
        const float ma = s_run[2 * r], la = s_run[2 * r + 1];
        const int64_t t = tok_first + r / G;
        const int h = kvh * G + r % G;
        p.out[(t * p.hq + h) * DH + d] = __float2bfloat16_rn(__fmul_rn(s_acc[e], __frcp_rn(la)));
        if (d == 0 && p.lse)
            p.lse[t * p.hq + h] = lse_of(ma, la);
    }
}

// Number of chunks a query tile needs: keys [0, kend) with kend one past the
// tile's last query position.
__device__ __forceinline__ int tile_chunks(const ReqMeta &m, int qt, int tq, int chunk)
{
    const int kend = m.L - m.qn + min(m.qn, (qt + 1) * tq);
    return (kend + chunk - 1) / chunk;
}

struct Unit {
    int b, kvh, qt, c;
    int total;  // units in the whole grid (every CTA computes the same count)
    bool valid;  // false: this CTA has nothing to do
    ReqMeta meta;
};

// Split-KV schedule: CTA i takes the i-th non-empty (request, KV head, query
// tile, chunk) unit, so every CTA with work comes first in the grid.  A
// request whose lengths are inconsistent gets one unit per (KV head, query
// tile) that only writes NaN rows.  Uses all threads; scratch in `s_int`
// (>= 38 ints).
__device__ inline Unit split_unit(const AttnParams &p, int chunk, int *s_int)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int cnt = 0;
    if (tid < p.num_seqs) {
        const ReqMeta m = read_meta(p, tid);
        if (!m.sane) {
            if (blockIdx.x == 0)
                record_error(p.err, kErrBadMetadata, tid);
        } else {
            const int qtl = (m.qn + p.tq - 1) / p.tq;
            if (!m.ok) {
                cnt = qtl;
            } else {
                for (int qt = 0; qt < qtl; ++qt)
                    cnt += (tile_chunks(m, qt, p.tq, chunk) + p.cpu - 1) / p.cpu;
            }
            cnt *= p.hkv;
        }
    }
    // block-wide exclusive prefix sum of cnt
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        s_int[warp] = incl;
    if (tid == 0)
        s_int[32] = -1;
    __syncthreads();
    int total = 0;
    for (int w = 0; w < (int)(blockDim.x / 32); ++w)
        total += s_int[w];
    int wpre = 0;
    for (int w = 0; w < warp; ++w)
        wpre += s_int[w];
    const long long excl = (long long)wpre + incl - cnt;
    const long long target = blockIdx.x;
    if (cnt > 0 && target >= excl && target < excl + cnt) {
        const ReqMeta m = read_meta(p, tid);  // cached: this thread just read it
        s_int[32] = tid;
        s_int[33] = (int)(target - excl);
        s_int[34] = m.qs;
        s_int[35] = m.qn;
        s_int[36] = m.L;
        s_int[37] = (m.sane ? 1 : 0) | (m.ok ? 2 : 0);
    }
    __syncthreads();
    Unit u;
    u.valid = false;
    u.total = total;
    const int b = s_int[32];
    if (b < 0)
        return u;
    int r = s_int[33];
    ReqMeta m;
    m.qs = s_int[34];
    m.qn = s_int[35];
    m.L = s_int[36];
    m.sane = (s_int[37] & 1) != 0;
    m.ok = (s_int[37] & 2) != 0;
    u.meta = m;
    u.c = 0;
    const int qtl = (m.qn + p.tq - 1) / p.tq;
    u.b = b;
    u.valid = true;
    if (!m.ok) {
        u.kvh = r / qtl;
        u.qt = r % qtl;
        return u;
    }
    int per_kvh = 0;
    for (int qt = 0; qt < qtl; ++qt)
        per_kvh += (tile_chunks(m, qt, p.tq, chunk) + p.cpu - 1) / p.cpu;
    u.kvh = r / per_kvh;
    r %= per_kvh;
    for (int qt = 0; qt < qtl; ++qt) {
        const int n = (tile_chunks(m, qt, p.tq, chunk) + p.cpu - 1) / p.cpu;
        if (r < n) {
            u.qt = qt;
            u.c = r;
            break;
        }
        r -= n;
    }
    return u;
}

}  // namespace pa

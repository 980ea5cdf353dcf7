// K2d: paged decode attention for head dim 128 with the MMA operands swapped.
//
// A decode CTA owns few query rows -- G query heads of one or a few tokens of
// one request and KV head ("fix(rocm): stabilize direct paged CK attention for
// bitwise R/R", Changes: one query per decode row) -- but every KV tile it
// reads has 128 keys.  With the rows as the M dimension of the MMA, 124 of 128
// TMEM lanes hold nothing and the softmax of a tile runs on one SM
// sub-partition.  Here the keys are the M dimension instead:
//   S^T = K . Q^T    A = the K tile (128 keys, K-major), B = Q (NR rows),
//                    D = S^T in TMEM: lane = key, column = query row;
//   O^T += V^T . P^T A = the V tile read MN-major (M = the head dim),
//                    B = P^T (NR rows, K-major, written by the softmax),
//                    D = O^T in TMEM: lane = head-dim element, column = row.
// Every output element is still the same K-step-16 dot product in ascending
// order on the same tensor-core instruction family as in the prefill kernel
// (pa_attn.cu); a swapped product equals the unswapped one bit for bit (IEEE
// multiplication commutes and the accumulation order over K is unchanged).
// So the fixed arithmetic C1-C7 of pa_attn.cu holds here unchanged:
//   C1  KV tiles of 128 keys from key 0, K-steps of 16 ascending.
//   C2  tile max of the raw scores over allowed keys, times c = scale*log2 e.
//   C3  lazy online softmax (threshold 8); p = exp2(fma(S, c, -m)), 0 for
//       masked keys; tile row sum: for each half of the keys an 8-way
//       interleaved sum (accumulator k sums the half's keys k, k+8, .. in
//       order, then ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7))), then half0 + half1.
//   C4  P rounded to BF16 (RNE) before P.V.
//   C5  256-key chunks from key 0, each starting fresh; chunk states fold left
//       to right (in the CTA, or in the split-KV merge of pa_split.cuh).
//   C6  out = O * rcp_rn(l) -> BF16 RNE; lse = (m + log2 l) * ln 2.
//
// Roles (384 threads):
//   warp 0       TMA producer: each group's Q tile (double-buffered), then
//                per tile one 64-column box per 16-token page for K and V
//                (block ids range-checked).
//   warp 1       tcgen05 issuer (one thread).
//   warps 4-7    softmax: thread j = key j of the tile (TMEM lane j); row
//                maxima by warp butterflies, row sums in the fixed order from
//                a shared-memory copy of p, P^T written to shared memory; in
//                a group's last tile, the V rows past its last key zeroed.
//   warps 8-11   chunk epilogue: thread d = head-dim element d (TMEM lane d):
//                chunk records (split-KV) or the in-CTA fold and the output.
//   all          the request scan before; in the last-arriving CTA of a
//                split-KV group, the fold of the group's chunk records after.
// Split-KV: the chunks of all groups are dealt out as one wave of equal
// contiguous ranges, one per CTA.  For a group cut by a range boundary the
// epilogue warps arrive on the group's counter as soon as their chunk records
// are written; the last arrival folds (no CTA waits).
#include <cuda_bf16.h>

#include <cstdio>
#include <cstring>

#include "pa_attn_common.cuh"
#include "pa_split.cuh"

namespace pa {

namespace dec {

constexpr int kThreads = 384;
constexpr int DH = 128;
constexpr int kKeys = 128;                // C1
constexpr int kChunk = 256;               // C5 at head dim 128
constexpr int TPC = kChunk / kKeys;       // tiles per chunk
constexpr int NSK = 3;                    // K stages
// V stages: three where shared memory allows (up to 16 rows), so the copy of
// V(j) can start once P.V(j-3) has finished rather than P.V(j-2)
template <int R>
constexpr int nsv_of() { return R <= 16 ? 3 : 2; }
constexpr int KST = kKeys * DH * 2;       // one K (or V) stage: 32 KB
constexpr int KBLK = kKeys * 128;         // one 64-column block of a stage
constexpr uint32_t kSCol = 0;             // TMEM: S^T buffers at columns 0 and 32
constexpr uint32_t kOCol = 64;            // TMEM: O^T chunk accumulators at 64 and 96
constexpr int kTmemCols = 128;
// Split-KV runs for fewer than 152 (request, KV head) groups, so at most
// this many requests: their lengths and chunk prefix sit in shared memory.
constexpr int kMaxSplitSeqs = 152;
constexpr int kReqBytes = ((6 * kMaxSplitSeqs + 1) * 4 + 15) / 16 * 16;
constexpr int kFlagBytes = 64;
// Bad-block-id flags in flight between the producer and the epilogue: the
// producer finishes chunk k only after the epilogue has read chunk k - 5.
constexpr int kBadRing = 8;
constexpr int kSmallBytes = 512 /*barriers*/ + kFlagBytes + 4 * 32 * 4 /*row maxima*/ +
                            2 * 32 * 4 /*m, factor*/ + 3 * 32 * 2 * 4 /*chunk and folded (m, l)*/ + kReqBytes;

// R: query rows the CTA processes (4, 8, 16 or 32: the largest request's
// query tokens times G, rounded up); NR: the N of both swapped MMAs (at least 16).
template <int R>
constexpr int nr_of() { return R < 16 ? 16 : R; }

template <int R>
constexpr size_t smem_bytes()
{
    constexpr int NR = nr_of<R>();
    return 1024 + (size_t)NSK * KST + (size_t)nsv_of<R>() * KST + 2 * 2 * NR * 128 /*Q x2*/ + 2 * 2 * NR * 128 /*P^T x2*/ +
           (size_t)R * kKeys * 4 /*p, fp32*/ + kSmallBytes;
}

// One butterfly step of the row maxima: the lane keeps one half of its CNT*2
// row values and takes the partner's copy of that half.
template <int CNT, int R>
__device__ __forceinline__ void bfly_max_step(float (&w)[R], int lane)
{
    constexpr int O = 32 * CNT / R;
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < CNT; ++i) {
        const float keep = up ? w[CNT + i] : w[i];
        const float send = up ? w[i] : w[CNT + i];
        w[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, O));
    }
}

// Max over the warp's 32 keys of each of R rows.  Afterwards w[0] of lane l
// holds row l / (32 / R).
template <int R>
__device__ __forceinline__ void warp_row_max(float (&w)[R], int lane)
{
    if constexpr (R >= 32) bfly_max_step<16, R>(w, lane);
    if constexpr (R >= 16) bfly_max_step<8, R>(w, lane);
    if constexpr (R >= 8) bfly_max_step<4, R>(w, lane);
    bfly_max_step<2, R>(w, lane);
    bfly_max_step<1, R>(w, lane);
    // lanes that differ only in the low bits hold the same row: reduce them
#pragma unroll
    for (int o = 16 / R; o >= 1; o >>= 1)
        w[0] = fmaxf(w[0], __shfl_xor_sync(0xffffffffu, w[0], o));
}

template <int R>
__device__ __forceinline__ void tmem_ld_r(uint32_t taddr, uint32_t (&r)[R])
{
    if constexpr (R == 32)
        tmem_ld32(taddr, r);
    else if constexpr (R == 16)
        tmem_ld16(taddr, r);
    else if constexpr (R == 8)
        tmem_ld8(taddr, r);
    else
        tmem_ld4(taddr, r);
}

template <int R>
__device__ __forceinline__ void tmem_st_r(uint32_t taddr, const uint32_t (&r)[R])
{
    if constexpr (R == 32)
        tmem_st32(taddr, r);
    else if constexpr (R == 16)
        tmem_st16(taddr, r);
    else if constexpr (R == 8)
        tmem_st8(taddr, r);
    else
        tmem_st4(taddr, r);
}

}  // namespace dec

// Split-KV arrival, by the four epilogue warps (thread t = 0..127) right
// after they wrote this CTA's chunk records of the group: an acquire-release
// add on the (request, KV head) group's counter.  The last CTA of the group
// to arrive folds (dec_merge); the others go on, so no CTA ever waits for
// another.  True in thread 0 of the folding CTA.
__device__ __forceinline__ bool dec_arrive(const AttnParams &p, int64_t unit_q, int narrive)
{
    bool last = false;
    const int t = threadIdx.x - 256;
    named_sync(3, 128);  // every record of this CTA is written (each thread's stores precede the barrier)
    if (t == 0) {
        // releases this CTA's records and, for the last arrival, acquires
        // every other CTA's
        uint32_t old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.ws_cnt + unit_q) : "memory");
        last = old == (uint32_t)(narrive - 1);  // above: a counter left by a failed call, fold nothing
        if (last)
            p.ws_cnt[unit_q] = 0u;  // ready for the next call
    }
    return last;
}

// The fold of a group's chunk records, left to right (C5), and the output
// (C6), by every thread of the last-arriving CTA after the CTA barrier that
// follows dec_arrive (which orders the acquire before these loads).  It is the
// in-CTA fold's sequence of fold_coef / fold_elem steps, computed per segment
// of records staged in shared memory: first the factors and mode of every
// (chunk, row) from the running maximum before the chunk (fold_coef's m is
// max(m_acc, m_chunk) in every mode and max is exact, so a warp scan gives
// it), then the l chains (last warp, one row per thread) beside the O chains
// (the other warps, one warp per row, four consecutive elements per thread,
// four chunks' operands loaded ahead of their steps).
template <int R>
__device__ __forceinline__ void dec_merge(const AttnParams &p, int64_t unit_q, int nchunks, int rv, int64_t tok_first,
                                          int kvh, float *work, int work_floats)
{
    constexpr int DH = dec::DH;
    constexpr int NTH = dec::kThreads;
    const int tid = threadIdx.x, warp = tid / 32, ln = tid % 32;
    const int Rw = p.ws_rows;
    const int64_t hdr = part_header_floats(Rw);
    const int64_t ustride = part_record_floats(Rw, DH);
    const float *part0 = p.ws_part + unit_q * p.nch * ustride;
    // staging area after a fixed head: [32] running max per row, [64] final (m, l)
    float *s_carry = work, *s_fin = work + 32;
    float *stage = work + 96;
    // per segment: m[cn][rv], l[cn][rv] (each padded to 4 floats), O[cn][rv][DH],
    // factors {sa, sc}[cn][rv], mode[cn][rv]
    const int per_chunk = rv * (DH + 5);
    const int seg = max(1, (work_floats - 96 - 16) / per_chunk);
    if (tid < 32)
        s_carry[tid] = -INFINITY;
    // O chains: warp w (w < NOW) takes rows w, w + NOW, ..; lane l takes the
    // head-dim elements 4l .. 4l+3 of its row (one 16-byte load per chunk)
    constexpr int NOW = NTH / 32 - 1;             // O-chain warps (the last warp runs the l chains)
    constexpr int NPR = (R + NOW - 1) / NOW;      // rows per O-chain warp
    float4 ov[NPR];
#pragma unroll
    for (int q = 0; q < NPR; ++q)
        ov[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    float l_run = 0.f;
    for (int c0 = 0; c0 < nchunks; c0 += seg) {
        const int cn = min(seg, nchunks - c0);
        const int hdr4 = (cn * rv + 3) & ~3;
        float *s_m = stage, *s_l = s_m + hdr4, *s_o = s_l + hdr4;
        float2 *s_cf = reinterpret_cast<float2 *>(s_o + cn * rv * DH);
        int *s_md = reinterpret_cast<int *>(s_cf + cn * rv);
        // (a) stage the segment's records: every copy in flight at once
        for (int i = tid; i < cn * rv * 2; i += NTH) {
            const int c = i / (2 * rv), k = i % (2 * rv), which = k / rv, n = k % rv;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr((which ? s_l : s_m) + c * rv + n)),
                         "l"(part0 + (c0 + c) * ustride + which * Rw + n)
                         : "memory");
        }
        for (int i = tid; i < cn * rv * (DH / 4); i += NTH) {
            const int c = i / (rv * (DH / 4)), k = i % (rv * (DH / 4)), n = k / (DH / 4), v4 = k % (DH / 4);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(s_o + (c * rv + n) * DH + 4 * v4)),
                         "l"(part0 + (c0 + c) * ustride + hdr + (int64_t)n * DH + 4 * v4)
                         : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
        // (b) factors and mode of every (chunk, row), one warp per row, 32 chunks per step
        for (int n = warp; n < rv; n += NTH / 32) {
            float run = s_carry[n];
            for (int cb = 0; cb < cn; cb += 32) {
                const int c = cb + ln;
                const float mc = c < cn ? s_m[c * rv + n] : -INFINITY;
                float inc = mc;
#pragma unroll
                for (int o2 = 1; o2 < 32; o2 <<= 1) {
                    const float x = __shfl_up_sync(0xffffffffu, inc, o2);
                    if (ln >= o2)
                        inc = fmaxf(inc, x);
                }
                float excl = __shfl_up_sync(0xffffffffu, inc, 1);
                if (ln == 0)
                    excl = -INFINITY;
                if (c < cn) {
                    const Fold f = fold_coef(fmaxf(run, excl), 0.f, mc, 0.f);
                    s_cf[c * rv + n] = make_float2(f.sa, f.sc);
                    s_md[c * rv + n] = f.mode;
                }
                run = fmaxf(run, __shfl_sync(0xffffffffu, inc, 31));
            }
            __syncwarp();
            if (ln == 0)
                s_carry[n] = run;
        }
        __syncthreads();
        if (warp == NOW) {
            // (c) the l chain of row ln: fold_coef's l, in chunk order
            const int n = ln;
            if (n < rv) {
                for (int cb = 0; cb < cn; cb += 7) {
                    float lc[7];
                    float2 cf[7];
                    int md[7];
#pragma unroll
                    for (int k = 0; k < 7; ++k) {
                        const int i = min(cb + k, cn - 1) * rv + n;
                        lc[k] = s_l[i];
                        cf[k] = s_cf[i];
                        md[k] = cb + k < cn ? s_md[i] : 0;  // past the last chunk: keep
                    }
#pragma unroll
                    for (int k = 0; k < 7; ++k) {
                        const float l2 = __fadd_rn(__fmul_rn(l_run, cf[k].x), __fmul_rn(lc[k], cf[k].y));
                        l_run = md[k] == 1 ? lc[k] : (md[k] == 2 ? l2 : l_run);
                    }
                }
            }
        } else {
            // (d) the O chains: per chunk one 16-byte load of the row's four
            //     elements, the row's factors and mode (broadcast), four steps
#pragma unroll
            for (int q = 0; q < NPR; ++q) {
                const int n = warp + q * NOW;
                if (n < rv) {
                    float4 a = ov[q];
                    for (int cb = 0; cb < cn; cb += 4) {
                        float4 x[4];
                        float2 f[4];
                        int md[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int c = min(cb + k, cn - 1);
                            x[k] = reinterpret_cast<const float4 *>(s_o + (c * rv + n) * DH)[ln];
                            f[k] = s_cf[c * rv + n];
                            md[k] = cb + k < cn ? s_md[c * rv + n] : 0;  // past the last chunk: keep
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            a.x = fold_elem_sel(a.x, x[k].x, f[k].x, f[k].y, md[k]);
                            a.y = fold_elem_sel(a.y, x[k].y, f[k].x, f[k].y, md[k]);
                            a.z = fold_elem_sel(a.z, x[k].z, f[k].x, f[k].y, md[k]);
                            a.w = fold_elem_sel(a.w, x[k].w, f[k].x, f[k].y, md[k]);
                        }
                    }
                    ov[q] = a;
                }
            }
        }
        __syncthreads();  // the next segment reuses the staging area
    }
    // (e) epilogue (C6)
    if (warp == NOW && ln < rv) {
        s_fin[2 * ln] = s_carry[ln];
        s_fin[2 * ln + 1] = l_run;
    }
    __syncthreads();
    const int G = p.group;
    if (warp < NOW) {
#pragma unroll
        for (int q = 0; q < NPR; ++q) {
            const int n = warp + q * NOW;
            if (n < rv) {
                const int64_t tok = tok_first + n / G;
                const int head = kvh * G + n % G;
                const float ln_ = s_fin[2 * n + 1];
                const float r = __frcp_rn(ln_);
                const uint32_t lo = pack_bf16x2(__fmul_rn(ov[q].x, r), __fmul_rn(ov[q].y, r));
                const uint32_t hi = pack_bf16x2(__fmul_rn(ov[q].z, r), __fmul_rn(ov[q].w, r));
                *reinterpret_cast<uint2 *>(p.out + (tok * p.hq + head) * DH + 4 * ln) = make_uint2(lo, hi);
                if (ln == 0 && p.lse)
                    p.lse[tok * p.hq + head] = lse_of(s_fin[2 * n], ln_);
            }
        }
    }
}

// A chunk of the work: chunk lc of the (request b, KV head kvh) group, with
// the request's lengths.  Chunks are numbered request-major: request b's
// groups start at hkv * pre[b], group (b, kvh) at gs = hkv * pre[b] + kvh * nch.
struct DecChunk {
    int bi;        // index into the shared request arrays
    int b;         // request
    int kvh, lc;   // KV head, chunk within the group
    int nchb;      // chunks of each of the request's groups
    int nt;        // tiles of this chunk (1 or 2)
    int L, qs, qn;
    int64_t gs;    // the group's first chunk in the sequence
};

// Shared-memory view of the requests (split-KV: all of them; otherwise the
// CTA's one request at index 0, request number b_off).
struct DecReqs {
    const int *qs, *qn, *len, *nch, *pre;
    int n, hkv, b_off;
};

__device__ __forceinline__ void dec_set_request(DecChunk &c, const DecReqs &v, int bi)
{
    c.bi = bi;
    c.b = bi + v.b_off;
    c.qs = v.qs[bi];
    c.qn = v.qn[bi];
    c.L = v.len[bi];
    c.nchb = v.nch[bi];
}

__device__ __forceinline__ void dec_set_tiles(DecChunk &c)
{
    c.nt = min(dec::TPC, (c.L + dec::kKeys - 1) / dec::kKeys - c.lc * dec::TPC);
}

// floor(num / den) for 0 <= num, 0 < den: one 32-bit division when both
// fit (the usual case; the 64-bit one is a long instruction sequence)
__device__ __forceinline__ int64_t dec_div(uint64_t num, uint64_t den)
{
    if ((num | den) <= 0xffffffffull)
        return (int64_t)((uint32_t)num / (uint32_t)den);
    return (int64_t)(num / den);
}

// Chunk x of the sequence (0 <= x < hkv * pre[n]).
__device__ __forceinline__ DecChunk dec_chunk_at(const DecReqs &v, int64_t x)
{
    // the largest b0 with hkv * pre[b0] <= x: a request with chunks
    int b0 = 0, b1 = v.n;
    while (b1 - b0 > 1) {
        const int mid = (b0 + b1) >> 1;
        if ((int64_t)v.hkv * v.pre[mid] <= x)
            b0 = mid;
        else
            b1 = mid;
    }
    DecChunk c;
    dec_set_request(c, v, b0);
    const int64_t base = (int64_t)v.hkv * v.pre[b0];
    const int r = (int)(x - base);  // < hkv * nch of one request
    c.kvh = r / c.nchb;
    c.lc = r % c.nchb;
    c.gs = base + (int64_t)c.kvh * c.nchb;
    dec_set_tiles(c);
    return c;
}

// The chunk after c (the caller knows there is one).
__device__ __forceinline__ void dec_chunk_next(DecChunk &c, const DecReqs &v)
{
    if (++c.lc >= c.nchb) {
        c.lc = 0;
        c.gs += c.nchb;
        if (++c.kvh >= v.hkv) {
            c.kvh = 0;
            int bi = c.bi + 1;
            while (bi < v.n - 1 && v.nch[bi] == 0)
                ++bi;
            dec_set_request(c, v, bi);
        }
    }
    dec_set_tiles(c);
}

// R: query rows the CTA processes (a power of two >= the largest request's
// query tokens times G); NR = max(R, 16) is the N of both swapped MMAs.
// Rows are token-major: row n = t*G + hh is query token t of the request,
// head kvh*G + hh.
//
// Work: the chunks (C5) of all (request, KV head) groups in request-major
// order.  Split-KV: the sequence is dealt out as gridDim equal contiguous
// ranges, one per CTA, each streamed through one pipeline (a range may hold
// the end of one group, whole groups and the start of another).  A group
// wholly inside one range is folded in that CTA; a group cut by a range
// boundary is written as chunk records, and the last of its CTAs to arrive
// folds them (dec_merge).  Without split-KV each CTA takes one group.
template <int R>
__global__ void __launch_bounds__(dec::kThreads, 1) dec_kernel(const __grid_constant__ AttnParams p)
{
    using namespace dec;
    constexpr int NR = nr_of<R>();
    constexpr int NSV = nsv_of<R>();
    constexpr int PASSES = (R * 16 + 127) / 128;  // softmax passes over the row-sum chains
    constexpr int PPT = kKeys / 16;  // pages per tile
    constexpr int NKB = DH / 64;     // 64-column blocks of the head dim
    constexpr int QBLK = NR * 128;   // one 64-column block of a Q tile
    constexpr int QBUF = 2 * QBLK;   // one Q tile
    constexpr int PBLK = NR * 128;   // one 64-key block of a P^T buffer
    constexpr int PBUF = 2 * PBLK;   // one P^T buffer (128 keys)
    constexpr uint32_t ID_QK = idesc_bf16_f32_ab(128, NR, false, false);
    constexpr uint32_t ID_PV = idesc_bf16_f32_ab(128, NR, true, false);
    constexpr int B_QF = 0, B_QE = B_QF + 2, B_KF = B_QE + 2, B_KE = B_KF + NSK, B_VF = B_KE + NSK;
    constexpr int B_VE = B_VF + NSV, B_SF = B_VE + NSV, B_PF = B_SF + 2, B_PV = B_PF + 2;
    constexpr int B_CR = B_PV + 2, B_OF = B_CR + 2;
    constexpr int B_OD = B_OF + 2;    // a chunk's last P.V has completed (by chunk parity)
    constexpr int B_IDS = B_OD + 2;   // a chunk's block ids are checked (ring of kBadRing)
    constexpr int B_DONE = B_IDS + kBadRing, NBARS = B_DONE + 1;
    static_assert(NBARS * 8 <= 512, "barrier area");
    static_assert(R == 4 || R == 8 || R == 16 || R == 32, "rows per CTA");
    static_assert(dec::smem_bytes<R>() <= kMaxSmemPerBlock, "shared-memory layout");

    // Launched with programmatic stream serialization (see pa_attn.cu): by
    // default nothing reads global memory before the preceding grid has
    // completed; with early_reads only the K/V copies wait.
    if (!p.early_reads)
        griddep_wait();
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sK = smem;
    uint8_t *sV = sK + NSK * KST;
    uint8_t *sQ = sV + NSV * KST;                                // two Q tiles (by segment parity)
    uint8_t *sP = sQ + 2 * QBUF;                                 // two P^T buffers
    float *sPs = reinterpret_cast<float *>(sP + 2 * PBUF);      // [R][128] p of the tile (fp32)
    uint8_t *small = reinterpret_cast<uint8_t *>(sPs) + R * kKeys * 4;
    uint64_t *bars = reinterpret_cast<uint64_t *>(small);
    // [0] abort [1] tmem [2] groups to fold [3, 4] those groups [8 + k % 8] chunk k's bad ids
    int *sflags = reinterpret_cast<int *>(small + 512);
    float *s_xmax = reinterpret_cast<float *>(small + 512 + kFlagBytes);  // [4 warps][32 rows]; scan scratch first
    float *s_mcur = s_xmax + 4 * 32;                          // [32] reference max after this tile
    float *s_mcor = s_mcur + 32;                              // [32] O factor: 1 or exp2(m_old - m_new)
    float *s_ml = s_mcor + 32;                                // [2 chunk parities][32][2] chunk (m, l)
    float *s_accml = s_ml + 2 * 32 * 2;                       // [32][2] in-CTA folded (m, l)
    // the requests: query start, query tokens, length, chunks per group,
    // status (1: inconsistent lengths), and the exclusive prefix of chunks
    int *s_qs = reinterpret_cast<int *>(s_accml + 32 * 2);
    int *s_qn = s_qs + kMaxSplitSeqs, *s_len = s_qn + kMaxSplitSeqs, *s_nch = s_len + kMaxSplitSeqs;
    int *s_st = s_nch + kMaxSplitSeqs, *s_pre = s_st + kMaxSplitSeqs;  // s_pre: [n + 1]
    volatile int *abort_flag = sflags;
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    auto wb = [&](int i, uint32_t parity) { return wait_bar(bar(i), parity, abort_flag, p.err, i); };
    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    float *const merge_work = reinterpret_cast<float *>(sK);
    constexpr int kMergeWorkFloats = (NSK * KST + NSV * KST) / 4;
    static_assert(kMergeWorkFloats >= R * (DH + 5) + 96 + 16 + 8, "merge staging: one chunk of R rows");
    const int G = p.group, hkv = p.hkv;

    // ----------------------------------------------------------- the work --
    // This CTA's chunks: [lo, hi) of the sequence of T chunks.
    int64_t lo, hi, T;
    int G_eff = 1;
    DecReqs rq;
    rq.qs = s_qs;
    rq.qn = s_qn;
    rq.len = s_len;
    rq.nch = s_nch;
    rq.pre = s_pre;
    rq.hkv = hkv;
    if (p.split) {
        // The block ids a CTA reads first depend on the scan below; a table
        // of up to 1 MB is brought into L2 meanwhile, spread over the CTAs,
        // so that read hits L2 rather than DRAM.
        {
            const int64_t lines = ((int64_t)p.num_seqs * p.max_blocks * 4 + 127) / 128;
            const int64_t line = (int64_t)tid * gridDim.x + blockIdx.x;
            if (lines <= (1 << 13) && line < lines)
                prefetch_l2(reinterpret_cast<const char *>(p.block_tables) + line * 128);
        }
        rq.n = p.num_seqs;
        rq.b_off = 0;
        int nch = 0;
        if (tid < p.num_seqs) {
            const ReqMeta m = read_meta(p, tid);
            if (!m.sane && blockIdx.x == 0)
                record_error(p.err, kErrBadMetadata, tid);
            if (m.ok && m.qn > 0)
                nch = (m.L + kChunk - 1) / kChunk;
            s_qs[tid] = m.qs;
            s_qn[tid] = m.qn;
            s_len[tid] = m.L;
            s_nch[tid] = nch;
            s_st[tid] = (m.sane && !m.ok && m.qn > 0) ? 1 : 0;  // NaN rows to write
        }
        // block-wide exclusive prefix of the chunk counts
        int incl = nch;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        int *s_wsum = reinterpret_cast<int *>(s_xmax);
        if (lane == 31)
            s_wsum[warp] = incl;
        __syncthreads();
        int wpre = 0, tot = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const int s = s_wsum[w];
            wpre += w < warp ? s : 0;
            tot += s;
        }
        if (tid < p.num_seqs)
            s_pre[tid] = wpre + incl - nch;
        if (tid == 0)
            s_pre[p.num_seqs] = tot;
        __syncthreads();
        // a request with inconsistent lengths: NaN rows, from one CTA
        for (int b = blockIdx.x; b < p.num_seqs; b += gridDim.x) {
            if (s_st[b]) {
                if (tid == 0)
                    record_error(p.err, kErrBadMetadata, b);
                for (int k = 0; k < hkv; ++k)
                    write_nan_rows<DH>(p, (int64_t)s_qs[b], min(p.tq, s_qn[b]), k);
            }
        }
        T = (int64_t)hkv * tot;
        G_eff = (int)(T < (int64_t)gridDim.x ? T : (int64_t)gridDim.x);
        if ((int)blockIdx.x >= G_eff)
            return;
        lo = dec_div((uint64_t)blockIdx.x * T, G_eff);
        hi = dec_div((uint64_t)(blockIdx.x + 1) * T, G_eff);
    } else {
        const int b = (int)(blockIdx.x / hkv), kvh = (int)(blockIdx.x % hkv);
        const ReqMeta m = read_meta(p, b);
        if (!m.ok) {
            if (tid == 0)
                record_error(p.err, kErrBadMetadata, b);
            if (m.sane && m.qn > 0)
                write_nan_rows<DH>(p, (int64_t)m.qs, min(p.tq, m.qn), kvh);
            return;
        }
        if (m.qn <= 0)
            return;
        const int nch = (m.L + kChunk - 1) / kChunk;  // >= 1: L >= qn > 0
        rq.n = 1;
        rq.b_off = b;
        if (tid == 0) {
            s_qs[0] = m.qs;
            s_qn[0] = m.qn;
            s_len[0] = m.L;
            s_nch[0] = nch;
            s_pre[0] = 0;
            s_pre[1] = nch;
        }
        T = (int64_t)hkv * nch;
        lo = (int64_t)kvh * nch;
        hi = lo + nch;
        __syncthreads();
    }
    const int nck = (int)(hi - lo);  // >= 1
    // the CTA (of G_eff) whose range holds chunk x
    auto cta_of = [&](int64_t x) { return (int)dec_div((uint64_t)(x + 1) * G_eff + T - 1, T) - 1; };

    // block ids of a chunk's (up to) 16 pages, lanes 0..15
    auto chunk_ids = [&](const DecChunk &c) {
        const int npn = (c.L + 15) / 16;
        const int pg = c.lc * (kChunk / 16) + lane;
        return (lane < kChunk / 16 && pg < npn) ? __ldg(p.block_tables + (int64_t)c.b * p.max_blocks + pg) : 0;
    };
    DecChunk c0;
    int ids_cur = 0;
    if (warp == 0) {
        c0 = dec_chunk_at(rq, lo);
        ids_cur = chunk_ids(c0);
    }

    // -------------------------------------------------------------- setup --
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_QF + i), 1);
            mbar_init(bar(B_QE + i), 1);
            mbar_init(bar(B_SF + i), 1);
            mbar_init(bar(B_PF + i), 4);  // the four softmax warps
            mbar_init(bar(B_PV + i), 1);
            mbar_init(bar(B_CR + i), 4);  // the four softmax warps, at a chunk's end
            mbar_init(bar(B_OF + i), 4);  // the four epilogue warps have read the chunk's O^T
            mbar_init(bar(B_OD + i), 1);
        }
        for (int s = 0; s < NSK; ++s) {
            mbar_init(bar(B_KF + s), 1);
            mbar_init(bar(B_KE + s), 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(bar(B_VF + s), 1);
            mbar_init(bar(B_VE + s), 1);
        }
        for (int i = 0; i < kBadRing; ++i)
            mbar_init(bar(B_IDS + i), 1);
        mbar_init(bar(B_DONE), 1);
        sflags[0] = 0;
        sflags[2] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&sflags[1]), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 64) {
        prefetch_tensormap(&p.tm_q);
        prefetch_tensormap(&p.tm_k);
        prefetch_tensormap(&p.tm_v);
    }
    if (R < NR) {
        // the softmax writes P^T rows 0..R-1 each tile; rows R..NR-1 stay zero
        for (int i = tid; i < 2 * PBUF / 16; i += kThreads)
            reinterpret_cast<uint4 *>(sP)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(sflags[1]);

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        // Per segment (the chunks of one group in this range) the group's Q
        // tile, double-buffered; per tile one 64-column box per 16-token page
        // for K and V, block ids read one chunk ahead and range-checked; per
        // chunk its bad-id flag for the epilogue.
        bool ok = true;
        int last_k_use[NSK], last_v_use[NSV], last_q_use[2] = {-1, -1};
        for (int s = 0; s < NSK; ++s) last_k_use[s] = -1;
        for (int s = 0; s < NSV; ++s) last_v_use[s] = -1;
        bool waited = !p.early_reads;
        // K and V are read once: their lines go first, so the code, block
        // tables and request metadata stay in L2
        const uint64_t kv_policy = l2_policy_evict_first();
        DecChunk c = c0;
        int it = 0, seg = -1;
        for (int k = 0; ok && k < nck; ++k) {
            if (k > 0)
                dec_chunk_next(c, rq);
            int ids_next = 0;
            if (k + 1 < nck) {
                DecChunk cn = c;
                dec_chunk_next(cn, rq);
                ids_next = chunk_ids(cn);
            }
            if (k == 0 || c.lc == 0) {
                // a new segment: its Q tile (G heads x NR/G tokens per block)
                ++seg;
                const int qb = seg & 1, uq = seg >> 1;
                if (lane == 0) {
                    if (uq >= 1)
                        ok = wb(B_QE + qb, (uq - 1) & 1);
                    if (ok)
                        mbar_arrive_expect_tx(bar(B_QF + qb), NKB * 128 * G * (NR / G));
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok)
                    break;
                if (lane < NKB)
                    tma_load_3d(smem_addr(sQ + qb * QBUF + lane * QBLK), &p.tm_q, bar(B_QF + qb), lane * 64,
                                c.kvh * G, c.qs);
                last_q_use[qb] = uq;
            }
            if (!waited) {
                griddep_wait();  // the cache write has completed and is visible
                waited = true;
            }
            const int npn = (c.L + 15) / 16;
            bool any_bad = false;
            for (int tt = 0; tt < c.nt; ++tt, ++it) {
                const int t = c.lc * TPC + tt;
                const int np = min(PPT, npn - t * PPT);
                int id = __shfl_sync(0xffffffffu, ids_cur, tt * PPT + lane % PPT);
                const bool badl = lane < np && (id < 0 || (int64_t)id >= p.num_blocks);
                if (badl)
                    id = 0;  // keep the pipeline flowing; the rows become NaN
                any_bad |= __any_sync(0xffffffffu, badl);
                const int pg = lane / NKB, kb = lane % NKB;
                const int pid = __shfl_sync(0xffffffffu, id, pg % PPT);
                const bool issue = lane < PPT * NKB && pg < np;
                const int sk = it % NSK, uk = it / NSK;
                if (lane == 0) {
                    if (uk >= 1)
                        ok = wb(B_KE + sk, (uk - 1) & 1);
                    if (ok)
                        mbar_arrive_expect_tx(bar(B_KF + sk), np * NKB * 2048);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok)
                    break;
                if (issue)
                    tma_load_4d_hint(smem_addr(sK + sk * KST + kb * KBLK + pg * 2048), &p.tm_k, bar(B_KF + sk),
                                     kb * 64, c.kvh, 0, pid, kv_policy);
                last_k_use[sk] = uk;
                const int sv = it % NSV, uv = it / NSV;
                if (lane == 0) {
                    if (uv >= 1)
                        ok = wb(B_VE + sv, (uv - 1) & 1);
                    if (ok)
                        mbar_arrive_expect_tx(bar(B_VF + sv), np * NKB * 2048);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok)
                    break;
                if (issue)
                    tma_load_4d_hint(smem_addr(sV + sv * KST + kb * KBLK + pg * 2048), &p.tm_v, bar(B_VF + sv),
                                     kb * 64, c.kvh, 0, pid, kv_policy);
                last_v_use[sv] = uv;
            }
            if (!ok)
                break;
            // the chunk's bad-id flag, released to the epilogue by the arrival.
            // Ring of kBadRing: issuing chunk k's last tile needed the P.V of
            // the tile NSV (<= 3) tiles before, so chunk k-5 has been read
            // (chunk k'+2's first P.V waits for the epilogue to read chunk
            // k'); the epilogue has passed this slot's previous phase.
            if (lane == 0) {
                if (any_bad)
                    record_error(p.err, kErrBadMetadata, c.b);
                sflags[8 + (k % kBadRing)] = any_bad ? 1 : 0;
                mbar_arrive(bar(B_IDS + (k % kBadRing)));
            }
            __syncwarp();
            ids_cur = ids_next;
        }
        if (lane == 0 && !ok) {
            // let issued copies land before the CTA's shared memory goes away
            for (int s = 0; s < NSK; ++s)
                if (last_k_use[s] >= 0)
                    wait_bar_drain(bar(B_KF + s), last_k_use[s] & 1);
            for (int s = 0; s < NSV; ++s)
                if (last_v_use[s] >= 0)
                    wait_bar_drain(bar(B_VF + s), last_v_use[s] & 1);
            for (int q = 0; q < 2; ++q)
                if (last_q_use[q] >= 0)
                    wait_bar_drain(bar(B_QF + q), last_q_use[q] & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer --
        // QK(0), QK(1), then PV(j) followed by QK(j+2): QK(j+2) overwrites the
        // S^T buffer and, through its commit, tells the softmax that PV(j) --
        // the last reader of P^T buffer j % 2 -- has completed.  Two cursors
        // walk the tiles: the QKs two ahead of the P.Vs.
        if (lane == 0) {
            struct Cur {
                DecChunk c;
                int k, tt, it, seg;
            };
            auto advance = [&](Cur &u) {
                const bool seg_end = u.tt == u.c.nt - 1 && (u.k == nck - 1 || u.c.lc == u.c.nchb - 1);
                ++u.it;
                if (++u.tt >= u.c.nt) {
                    u.tt = 0;
                    if (++u.k < nck)
                        dec_chunk_next(u.c, rq);
                }
                u.seg += seg_end ? 1 : 0;
            };
            Cur cq, cv;
            cq.c = dec_chunk_at(rq, lo);
            cq.k = cq.tt = cq.it = cq.seg = 0;
            cv = cq;
            int kc = 0;  // chunk of the P.V cursor
            auto issue_qk = [&](const Cur &u) -> bool {
                const int qb = u.seg & 1;
                if (u.tt == 0 && (u.k == 0 || u.c.lc == 0) && !wb(B_QF + qb, (u.seg >> 1) & 1))
                    return false;
                const int sk = u.it % NSK;
                if (!wb(B_KF + sk, (u.it / NSK) & 1))
                    return false;
                const uint32_t k0 = smem_addr(sK + sk * KST), q0 = smem_addr(sQ + qb * QBUF);
                tc_fence_after();
                uint64_t ad[8], bd[8];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    ad[kk] = sdesc_sw128(k0 + (kk / 4) * KBLK + (kk % 4) * 32, 16, 1024);
                    bd[kk] = sdesc_sw128(q0 + (kk / 4) * QBLK + (kk % 4) * 32, 16, 1024);
                }
                mma8_ss<1>(tmem + kSCol + (uint32_t)(u.it & 1) * 32, ad, bd, ID_QK, 0u);
                mma_commit(bar(B_KE + sk));
                mma_commit(bar(B_SF + (u.it & 1)));
                // the segment's last QK: its Q tile may be replaced
                if (u.tt == u.c.nt - 1 && (u.k == nck - 1 || u.c.lc == u.c.nchb - 1))
                    mma_commit(bar(B_QE + qb));
                return true;
            };
            auto issue_pv = [&](const Cur &u) -> bool {
                const int j = u.it;
                const int sv = j % NSV;
                const bool chunk_first = u.tt == 0;
                // P ready also means a tile past the group's last key has had
                // those V rows zeroed (by the softmax)
                bool okj = wb(B_VF + sv, (j / NSV) & 1);
                if (okj)
                    okj = wb(B_PF + (j & 1), (j >> 1) & 1);
                if (okj && chunk_first && kc >= 2)
                    okj = wb(B_OF + (kc & 1), ((kc >> 1) - 1) & 1);  // chunk kc-2 has been read
                if (okj) {
                    tc_fence_after();
                    const uint32_t v0 = smem_addr(sV + sv * KST), p0 = smem_addr(sP + (j & 1) * PBUF);
                    uint64_t ad[8], bd[8];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        ad[kk] = sdesc_sw128(v0 + kk * 2048, KBLK, 1024);  // 16 keys per step, MN-major
                        bd[kk] = sdesc_sw128(p0 + (kk / 4) * PBLK + (kk % 4) * 32, 16, 1024);
                    }
                    mma8_ss<1>(tmem + kOCol + (uint32_t)(kc & 1) * 32, ad, bd, ID_PV, chunk_first ? 0u : 1u);
                    mma_commit(bar(B_VE + sv));
                    mma_commit(bar(B_PV + (j & 1)));
                    // the chunk's last tile: its O^T is complete.  One phase per
                    // chunk of this parity, and chunk kc + 2's first P.V waits for
                    // the epilogue to have read chunk kc, so the epilogue's wait
                    // is never two phases behind.
                    if (u.tt == u.c.nt - 1)
                        mma_commit(bar(B_OD + (kc & 1)));
                }
                return okj;
            };
            bool ok = true;
            for (int i = 0; ok && i < 2 && cq.k < nck; ++i) {
                ok = issue_qk(cq);
                advance(cq);
            }
            while (ok && cv.k < nck) {
                ok = issue_pv(cv);
                const bool chunk_end = cv.tt == cv.c.nt - 1;
                advance(cv);
                kc += chunk_end ? 1 : 0;
                if (ok && cq.k < nck) {
                    ok = issue_qk(cq);
                    advance(cq);
                }
            }
            mma_commit(bar(B_DONE));
            wait_bar_drain(bar(B_DONE), 0);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // -------------------------------------------------------- softmax --
        // Per tile: row maxima (warp butterflies, then the four warps'
        // maxima through shared memory), then every thread runs the same
        // lazy reference-max update for all R rows (identical inputs and
        // operations, so identical bits in every thread), p and P^T, one
        // barrier, the O^T rescale, the P-ready arrival, and only then the
        // fixed-order row sums (off the P.V path).  Row n's l lives in the
        // thread that finishes its sum chain.
        const int j = tid - 128;           // key of the tile = TMEM lane
        const int w4 = warp - 4;           // TMEM lane quadrant
        const uint32_t lane_off = static_cast<uint32_t>(32 * w4) << 16;
        float m_run[R];                    // reference max of every row (all threads)
#pragma unroll
        for (int n = 0; n < R; ++n)
            m_run[n] = -INFINITY;
        float l_own[PASSES];               // l of row (ps*128 + j)/16 when j % 16 == 0
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps)
            l_own[ps] = 0.f;
        bool failed = false;
        DecChunk c = dec_chunk_at(rq, lo);
        int it = 0;
        for (int kc = 0; kc < nck && !failed; ++kc) {
            if (kc > 0)
                dec_chunk_next(c, rq);
            const int rv = c.qn * G;      // valid rows: columns 0..rv-1 of S^T and O^T (rv <= R)
            const int pos0 = c.L - c.qn;  // position of query token 0; row n sits at pos0 + n/G
            for (int tt = 0; tt < c.nt; ++tt, ++it) {
                const int t = c.lc * TPC + tt;
                const int sb = it & 1;
                bool okw = !failed && wb(B_SF + sb, (it >> 1) & 1);
                // A tile past the group's last key: its V rows of keys >= L are
                // zeroed here once they have landed (stale or poisoned data never
                // meets P = 0).  The wait names the right phase: S(it) ready
                // means P.V(it-2) was issued, so this stage's previous tile has
                // landed, and its next tile needs P.V(it), after this arrival.
                const bool zt = (t + 1) * kKeys > c.L;
                if (okw && zt)
                    okw = wb(B_VF + it % NSV, (it / NSV) & 1);
                okw = __all_sync(0xffffffffu, okw);
                tc_fence_after();
                uint32_t sr[R];
                if (okw) {
                    tmem_ld_r<R>(tmem + lane_off + kSCol + sb * 32, sr);
                    tmem_wait_ld();
                }
                // rows [nlo, rv) may see key kabs (row n sits at pos0 + n/G)
                const int kabs = t * kKeys + j;
                const int nlo = kabs <= pos0 ? 0 : min(rv, (kabs - pos0) * G);
                float w[R];
#pragma unroll
                for (int n = 0; n < R; ++n)
                    w[n] = (okw && n >= nlo && n < rv) ? __uint_as_float(sr[n]) : -INFINITY;
                warp_row_max<R>(w, lane);
                if (lane % (32 / R) == 0)
                    s_xmax[w4 * 32 + lane / (32 / R)] = w[0];
                if (named_sync_or(2, 128, !okw)) {
                    failed = true;
                    break;
                }
                // C2 tile max and the lazy reference-max update (C3), every row
                float fac[R];  // O and l factor of each row: 1, or exp2(m_old - m_new)
                bool any_need = false;
#pragma unroll
                for (int n = 0; n < R; ++n) {
                    const float tmax = __fmul_rn(
                        fmaxf(fmaxf(s_xmax[n], s_xmax[32 + n]), fmaxf(s_xmax[64 + n], s_xmax[96 + n])), p.scale_log2);
                    float mn = m_run[n], f = 1.f;
                    if (n < rv && tmax != -INFINITY) {
                        if (mn == -INFINITY) {
                            mn = tmax;
                        } else if (tmax > __fadd_rn(m_run[n], kTau)) {
                            mn = tmax;
                            f = ex2(__fsub_rn(m_run[n], mn));
                            any_need = true;
                        }
                    }
                    m_run[n] = mn;
                    fac[n] = f;
                    if (n == j) {  // for the owner of the row's sum
                        s_mcur[n] = mn;
                        s_mcor[n] = f;
                    }
                }
                // p = exp2(fma(S, c, -m)) for allowed keys, exactly 0 otherwise
                float pv[R];
#pragma unroll
                for (int n = 0; n < R; ++n) {
                    pv[n] = (n >= nlo && n < rv) ? ex2(__fmaf_rn(__uint_as_float(sr[n]), p.scale_log2, -m_run[n]))
                                                 : 0.f;
                    if (n < rv)
                        sPs[n * kKeys + j] = pv[n];
                }
                // P^T (BF16, C4), K-major with 128-byte swizzle: keys j and j+1 of
                // a row share one 32-bit word; even lanes write rows 0..R/2-1, odd
                // lanes rows R/2..R-1
                {
                    const bool odd = (lane & 1) != 0;
                    const int key0 = j & ~1;
                    uint8_t *pb = sP + sb * PBUF + (key0 / 64) * PBLK;
                    const int chunk16 = ((key0 % 64) * 2) / 16, within = (key0 % 8) * 2;
#pragma unroll
                    for (int i = 0; i < R / 2; ++i) {
                        const float mine = odd ? pv[R / 2 + i] : pv[i];
                        const float send = odd ? pv[i] : pv[R / 2 + i];
                        const uint32_t mb = __bfloat16_as_ushort(__float2bfloat16_rn(mine));
                        const uint32_t sbits = __bfloat16_as_ushort(__float2bfloat16_rn(send));
                        const uint32_t got = __shfl_xor_sync(0xffffffffu, sbits, 1);
                        const int n = odd ? R / 2 + i : i;
                        const uint32_t word = odd ? (got | (mb << 16)) : (mb | (got << 16));
                        *reinterpret_cast<uint32_t *>(pb + n * 128 + ((chunk16 ^ (n & 7)) << 4) + within) = word;
                    }
                }
                if (zt) {
                    const int row0 = c.L - t * kKeys;
                    const int nz = (kKeys - row0) * NKB * 8;
                    uint8_t *vs = sV + (it % NSV) * KST;
                    for (int idx = j; idx < nz; idx += 128) {
                        const int row = row0 + idx / (NKB * 8);
                        const int rem = idx % (NKB * 8);
                        *reinterpret_cast<uint4 *>(vs + (rem / 8) * KBLK + row * 128 + (rem % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                named_sync(2, 128);  // P^T, p and zeroed V rows complete; every thread has read the row maxima
                // O^T of this chunk must hold PV(it - 1) before it is rescaled
                // (a rescale needs an earlier tile of the same chunk)
                if (any_need) {
                    const bool okr = __all_sync(0xffffffffu, wb(B_PV + ((it - 1) & 1), ((it - 1) >> 1) & 1));
                    if (!okr) {
                        failed = true;
                    } else {
                        tc_fence_after();
                        uint32_t o[R];
                        const uint32_t col = tmem + lane_off + kOCol + (uint32_t)(kc & 1) * 32;
                        tmem_ld_r<R>(col, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int n = 0; n < R; ++n)
                            o[n] = __float_as_uint(__fmul_rn(__uint_as_float(o[n]), fac[n]));
                        tmem_st_r<R>(col, o);
                        tmem_wait_st();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(B_PF + sb));
                // row sums in the fixed order: chain (n, h, k) sums keys 64h+k+8i,
                // i = 0..7; the lanes of one (n, h) hold k = 0..7, so the butterfly
                // over xor 1, 2, 4 is ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7)), and xor 8
                // adds the other half
                const bool chunk_end = tt == c.nt - 1;
#pragma unroll
                for (int ps = 0; ps < PASSES; ++ps) {
                    const int ci = ps * 128 + j;
                    const int n = ci >> 4, h = (ci >> 3) & 1, k = ci & 7;
                    float a = 0.f;
                    if (n < rv) {
                        const float *row = sPs + n * kKeys + 64 * h + k;
                        a = row[0];
#pragma unroll
                        for (int i = 1; i < 8; ++i)
                            a = __fadd_rn(a, row[8 * i]);
                    }
                    a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 1));
                    a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 2));
                    a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 4));
                    const float other = __shfl_xor_sync(0xffffffffu, a, 8);
                    if (n < rv && (ci & 15) == 0) {
                        // l = l * factor + tile sum (factor 1 when m did not move: the
                        // same bits as l + tile sum)
                        l_own[ps] = __fadd_rn(__fmul_rn(l_own[ps], s_mcor[n]), __fadd_rn(a, other));
                        if (chunk_end) {
                            // the slot was last read for chunk kc - 2 (before that chunk's O-free arrival)
                            if (kc >= 2 && !wb(B_OF + (kc & 1), ((kc >> 1) - 1) & 1))
                                failed = true;
                            s_ml[((kc & 1) * 32 + n) * 2] = s_mcur[n];
                            s_ml[((kc & 1) * 32 + n) * 2 + 1] = l_own[ps];
                            l_own[ps] = 0.f;
                        }
                    }
                }
                if (chunk_end) {
#pragma unroll
                    for (int n = 0; n < R; ++n)
                        m_run[n] = -INFINITY;
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(bar(B_CR + (kc & 1)));
                }
                // a failed wait above ends the loop for all four warps together at
                // the next tile's first barrier
            }
        }
    } else if (warp >= 8) {
        // --------------------------------------------------- chunk epilogue --
        // Per chunk: O^T into the in-CTA fold of a group wholly in this range
        // (the output after the group's last chunk), or to a split-KV record
        // (after the group's last chunk here, the arrival on its counter).
        const int d = tid - 256;  // head-dim element = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
        const int64_t rec_floats = part_record_floats(p.ws_rows, DH);
        const int64_t rec_hdr = part_header_floats(p.ws_rows);
        const float qnan = __int_as_float(0x7FC00000);
        float acc[R];   // in-CTA fold: the folded O^T column entries of element d
        bool gbad = false;  // a bad block id in the group so far (in-CTA fold)
        DecChunk c = dec_chunk_at(rq, lo);
        // CTAs arriving on the groups cut by this range's ends (computed
        // while the first chunk's data is still on its way)
        int narrive_first = 1, narrive_last = 1;
        int64_t gs_last = c.gs;
        if (p.split) {
            narrive_first = cta_of(c.gs + c.nchb - 1) - cta_of(c.gs) + 1;
            const DecChunk cl = dec_chunk_at(rq, hi - 1);
            gs_last = cl.gs;
            narrive_last = cta_of(cl.gs + cl.nchb - 1) - cta_of(cl.gs) + 1;
        }
        for (int k = 0; k < nck; ++k) {
            if (k > 0)
                dec_chunk_next(c, rq);
            const int rv = c.qn * G;
            const bool whole = !p.split || (c.gs >= lo && c.gs + c.nchb <= hi);
            bool ok = wb(B_CR + (k & 1), (k >> 1) & 1);
            if (ok)
                ok = wb(B_OD + (k & 1), (k >> 1) & 1);
            if (ok)
                ok = wb(B_IDS + (k % kBadRing), (k / kBadRing) & 1);
            ok = __all_sync(0xffffffffu, ok);
            // the four warps leave together; the barrier also orders the
            // previous chunk's writes of the folded (m, l) before this chunk's reads
            if (named_sync_or(3, 128, !ok))
                break;
            tc_fence_after();
            uint32_t o[R];
            tmem_ld_r<R>(tmem + lane_off + kOCol + (uint32_t)(k & 1) * 32, o);
            tmem_wait_ld();
            const float *ml = s_ml + (k & 1) * 64;  // the chunk's (m, l) per row
            const bool bad = sflags[8 + (k % kBadRing)] != 0;
            if (!whole) {
                // partial state of chunk lc of the group: m, l, then the O rows
                const int64_t unit_q = (int64_t)c.b * hkv + c.kvh;
                float *part = p.ws_part + (unit_q * p.nch + c.lc) * rec_floats;
                if (d < rv) {
                    part[d] = bad ? 0.f : ml[2 * d];
                    part[p.ws_rows + d] = bad ? qnan : ml[2 * d + 1];
                }
#pragma unroll
                for (int n = 0; n < R; ++n)
                    if (n < rv)
                        __stcg(part + rec_hdr + (int64_t)n * DH + d, bad ? qnan : __uint_as_float(o[n]));
            } else {
                if (c.lc == 0) {
                    // the group's first chunk: an empty fold
#pragma unroll
                    for (int n = 0; n < R; ++n)
                        acc[n] = 0.f;
                    gbad = false;
                    if (d < 32) {
                        s_accml[2 * d] = -INFINITY;  // the folded (m, l) of row d
                        s_accml[2 * d + 1] = 0.f;
                    }
                    named_sync(3, 128);
                }
                gbad |= bad;
                const bool final_chunk = c.lc == c.nchb - 1;
                const int64_t tok_first = c.qs;
                float fm_own = 0.f, fl_own = 0.f;  // row d's folded (m, l)
#pragma unroll
                for (int n = 0; n < R; ++n) {
                    if (n >= rv)
                        continue;
                    const Fold f = fold_coef(s_accml[2 * n], s_accml[2 * n + 1], ml[2 * n], ml[2 * n + 1]);
                    const float v = fold_elem(acc[n], __uint_as_float(o[n]), f);
                    if (final_chunk) {
                        const int64_t tok = tok_first + n / G;
                        const int head = c.kvh * G + n % G;
                        p.out[(tok * p.hq + head) * DH + d] =
                            gbad ? __ushort_as_bfloat16(0x7FC0) : __float2bfloat16_rn(__fmul_rn(v, __frcp_rn(f.l)));
                        if (d == n && p.lse)
                            p.lse[tok * p.hq + head] = gbad ? qnan : lse_of(f.m, f.l);
                    } else {
                        acc[n] = v;
                    }
                    if (d == n) {
                        fm_own = f.m;
                        fl_own = f.l;
                    }
                }
                named_sync(3, 128);  // every thread has read the folded (m, l)
                if (d < rv) {
                    s_accml[2 * d] = fm_own;
                    s_accml[2 * d + 1] = fl_own;
                }
            }
            tc_fence_before();
            __syncwarp();
            // this parity's O^T buffer and (m, l) slot are free for chunk k + 2
            if (lane == 0)
                mbar_arrive(bar(B_OF + (k & 1)));
            if (!whole && (k == nck - 1 || c.lc == c.nchb - 1)) {
                // the group's last chunk in this range: arrive on its counter
                const int narrive = c.gs == gs_last ? narrive_last : narrive_first;
                const int64_t unit_q = (int64_t)c.b * hkv + c.kvh;
                if (dec_arrive(p, unit_q, narrive)) {
                    const int nf = sflags[2];
                    sflags[3 + nf] = (int)unit_q;
                    sflags[2] = nf + 1;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // The groups this CTA arrived last on (at most two: those cut by the
    // range's ends), folded by every thread: all of this CTA's MMAs and
    // copies have completed, so the K/V stage area is free.
    const int nfold = sflags[2];
    for (int f = 0; f < nfold; ++f) {
        const int unit_q = sflags[3 + f];
        const int bi = unit_q / hkv, kvh = unit_q % hkv;
        dec_merge<R>(p, unit_q, s_nch[bi], s_qn[bi] * G, (int64_t)s_qs[bi], kvh, merge_work, kMergeWorkFloats);
        __syncthreads();
    }
}

// ------------------------------------------------------------------ host --

cudaError_t init_decode_attributes()
{
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(dec_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)dec::smem_bytes<4>())) != cudaSuccess ||
        (e = cudaFuncSetAttribute(dec_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)dec::smem_bytes<8>())) != cudaSuccess ||
        (e = cudaFuncSetAttribute(dec_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)dec::smem_bytes<16>())) != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(dec_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)dec::smem_bytes<32>());
}

int decode_rows(const AttnPlan &pl, int32_t max_query_len, int32_t num_seqs)
{
    if (pl.head_dim != 128 || pl.kt != 128 || pl.cl != 1 || pl.qtiles != 1)
        return 0;
    if (pl.split && num_seqs > dec::kMaxSplitSeqs)
        return 0;
    const long long rows = (long long)pl.group * max_query_len;
    for (int r = 4; r <= 32; r *= 2)
        if (rows <= r)
            return r;
    return 0;
}

long long decode_grid(const AttnPlan &pl, int32_t num_seqs, int32_t num_kv_heads, int num_sms)
{
    const long long groups = (long long)num_seqs * num_kv_heads;
    if (!pl.split)
        return groups;  // one CTA per (request, KV head)
    // split-KV: one wave, a contiguous range of chunks per CTA
    const long long chunks = groups * pl.nch;
    const long long sms = num_sms > 0 ? num_sms : 1;
    return chunks < sms ? chunks : sms;
}

cudaError_t launch_decode(const AttnArgs &a, const AttnPlan &pl, AttnParams &p, int rows, cudaStream_t stream)
{
    const int nr = rows < 16 ? 16 : rows;  // the MMAs' N: rows of the Q tile
    // Q box: 64 columns x G heads x (nr / G) tokens
    {
        const int G = pl.group;
        const cuuint64_t dims[3] = {128, (cuuint64_t)a.num_q_heads, (cuuint64_t)a.num_q_tokens};
        const cuuint64_t strides[2] = {(cuuint64_t)128 * 2, (cuuint64_t)a.q_tok_stride * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(nr / G)};
        if (encode_tiled(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    const long long grid = decode_grid(pl, a.num_seqs, a.num_kv_heads, p.num_sms);
    if (grid <= 0)
        return cudaSuccess;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(dec::kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (rows) {
    case 4: cfg.dynamicSmemBytes = dec::smem_bytes<4>(); return cudaLaunchKernelEx(&cfg, dec_kernel<4>, p);
    case 8: cfg.dynamicSmemBytes = dec::smem_bytes<8>(); return cudaLaunchKernelEx(&cfg, dec_kernel<8>, p);
    case 16: cfg.dynamicSmemBytes = dec::smem_bytes<16>(); return cudaLaunchKernelEx(&cfg, dec_kernel<16>, p);
    case 32: cfg.dynamicSmemBytes = dec::smem_bytes<32>(); return cudaLaunchKernelEx(&cfg, dec_kernel<32>, p);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace pa

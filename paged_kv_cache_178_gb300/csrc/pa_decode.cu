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
//   warp 0       TMA producer: Q once, then per tile one 64-column box per
//                16-token page for K and V (block ids range-checked), and the
//                zeroing of the last tile's V rows past the last needed key.
//   warp 1       tcgen05 issuer (one thread).
//   warps 4-7    softmax: thread j = key j of the tile (TMEM lane j); row
//                maxima by warp butterflies, row sums in the fixed order from
//                a shared-memory copy of p, P^T written to shared memory.
//   warps 8-11   chunk epilogue: thread d = head-dim element d (TMEM lane d):
//                chunk records (split-KV) or the in-CTA fold and the output.
//   all          the unit scan before; in the last-arriving CTA of a split-KV
//                group, the fold of the group's chunk records after.
// Split-KV: the epilogue warps arrive on the group's counter as soon as
// their chunk records are written; the last arrival folds (no CTA waits).
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
constexpr int kSmallBytes = 512 /*barriers*/ + 64 /*flags*/ + 4 * 32 * 4 /*row maxima*/ +
                            3 * 32 * 4 /*m, factor, sums*/ + 3 * 32 * 2 * 4 /*chunk and folded (m, l)*/;

// R: query rows the CTA processes (4, 8, 16 or 32: the request's query
// tokens times G, rounded up); NR: the N of both swapped MMAs (at least 16).
template <int R>
constexpr int nr_of() { return R < 16 ? 16 : R; }

template <int R>
constexpr size_t smem_bytes()
{
    constexpr int NR = nr_of<R>();
    return 1024 + (size_t)NSK * KST + (size_t)nsv_of<R>() * KST + 2 * NR * 128 /*Q*/ + 2 * 2 * NR * 128 /*P^T x2*/ +
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
// after they wrote this CTA's chunk records: an acquire-release add on the
// (request, KV head) group's counter.  The last CTA of the group to arrive
// folds (dec_merge); the others leave at once, so no CTA ever waits for
// another.  *s_flag = 1 in the folding CTA.
__device__ __forceinline__ void dec_arrive(const AttnParams &p, int64_t unit_q, int narrive, int *s_flag)
{
    const int t = threadIdx.x - 256;
    named_sync(3, 128);  // every record of this CTA is written (each thread's stores precede the barrier)
    if (t == 0) {
        // releases this CTA's records and, for the last arrival, acquires
        // every other CTA's
        uint32_t old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.ws_cnt + unit_q) : "memory");
        const bool last = old == (uint32_t)(narrive - 1);  // above: a counter left by a failed call, fold nothing
        if (last)
            p.ws_cnt[unit_q] = 0u;  // ready for the next call
        *s_flag = last ? 1 : 0;
    }
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

// R: query rows the CTA processes (a power of two >= the request's query
// tokens times G); NR = max(R, 16) is the N of both swapped MMAs.  Rows are
// token-major: row n = t*G + hh is query token t of the request, head kvh*G+hh.
template <int R>
__global__ void __launch_bounds__(dec::kThreads, 1) dec_kernel(const __grid_constant__ AttnParams p)
{
    using namespace dec;
    constexpr int NR = nr_of<R>();
    constexpr int NSV = nsv_of<R>();
    constexpr int PASSES = (R * 16 + 127) / 128;  // softmax passes over the row-sum chains
    constexpr int PPT = kKeys / 16;  // pages per tile
    constexpr int TPL = 16 / PPT;    // tiles whose block ids one 16-lane read covers
    constexpr int NKB = DH / 64;     // 64-column blocks of the head dim
    constexpr int QBLK = NR * 128;   // one 64-column block of the Q tile
    constexpr int PBLK = NR * 128;   // one 64-key block of a P^T buffer
    constexpr int PBUF = 2 * PBLK;   // one P^T buffer (128 keys)
    constexpr uint32_t ID_QK = idesc_bf16_f32_ab(128, NR, false, false);
    constexpr uint32_t ID_PV = idesc_bf16_f32_ab(128, NR, true, false);
    constexpr int B_Q = 0, B_KF = 1, B_KE = B_KF + NSK, B_VF = B_KE + NSK, B_VE = B_VF + NSV;
    constexpr int B_SF = B_VE + NSV, B_PF = B_SF + 2, B_PV = B_PF + 2, B_CR = B_PV + 2, B_OF = B_CR + 2;
    constexpr int B_OD = B_OF + 2;  // a chunk's last P.V has completed (by chunk parity)
    constexpr int B_PROD = B_OD + 2, B_DONE = B_PROD + 1, B_VZ = B_DONE + 1, NBARS = B_VZ + 1;
    static_assert(NBARS * 8 <= 512, "barrier area");
    static_assert(R == 4 || R == 8 || R == 16 || R == 32, "rows per CTA");

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
    uint8_t *sQ = sV + NSV * KST;
    uint8_t *sP = sQ + 2 * QBLK;                                // two P^T buffers
    float *sPs = reinterpret_cast<float *>(sP + 2 * PBUF);     // [R][128] p of the tile (fp32)
    uint8_t *small = reinterpret_cast<uint8_t *>(sPs) + R * kKeys * 4;
    uint64_t *bars = reinterpret_cast<uint64_t *>(small);
    int *sflags = reinterpret_cast<int *>(small + 512);  // [0] abort [1] tmem [2] merger [3] bad [4,5] rescale
    float *s_xmax = reinterpret_cast<float *>(small + 576);  // [4 warps][32 rows]; unit-scan scratch first
    float *s_mcur = s_xmax + 4 * 32;                          // [32] reference max after this tile
    float *s_mcor = s_mcur + 32;                              // [32] O factor: 1 or exp2(m_old - m_new)
    float *s_tsum = s_mcor + 32;                              // [32] tile row sums
    float *s_ml = s_tsum + 32;                                // [2 chunk parities][32][2] chunk (m, l)
    float *s_accml = s_ml + 2 * 32 * 2;                       // [32][2] in-CTA folded (m, l)
    volatile int *abort_flag = sflags;
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    auto wb = [&](int i, uint32_t parity) { return wait_bar(bar(i), parity, abort_flag, p.err, i); };
    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    float *const merge_work = reinterpret_cast<float *>(sK);
    constexpr int kMergeWorkFloats = (NSK * KST + NSV * KST) / 4;
    static_assert(kMergeWorkFloats >= R * (DH + 5) + 96 + 16 + 8, "merge staging: one chunk of R rows");

    // ---------------------------------------------------------- work unit --
    int b, kvh, c_grid = 0;
    ReqMeta meta;
    if (p.split) {
        const Unit un = split_unit(p, kChunk, reinterpret_cast<int *>(s_xmax));
        if (!un.valid)
            return;
        b = un.b;
        kvh = un.kvh;
        c_grid = un.c;
        meta = un.meta;
    } else {
        const long long u = blockIdx.x;
        kvh = (int)(u % p.hkv);
        b = (int)(u / p.hkv);
        meta = read_meta(p, b);
    }
    const int qs = meta.qs, qn = meta.qn, L = meta.L;
    if (!meta.ok) {
        if (tid == 0)
            record_error(p.err, kErrBadMetadata, b);
        if (meta.sane && qn > 0)
            write_nan_rows<DH>(p, (int64_t)qs, min(p.tq, qn), kvh);
        return;
    }
    if (qn <= 0)
        return;
    const int G = p.group;
    const int rv = qn * G;  // valid rows: columns 0..rv-1 of S^T and O^T (rv <= R)
    const int64_t tok_first = qs;
    const int pos0 = L - qn;  // position of query token 0; row n sits at pos0 + n/G
    const int kend = L;
    const int nchunks = (kend + kChunk - 1) / kChunk;
    int kbeg = 0, kstop = kend;
    if (p.split) {
        kbeg = c_grid * p.cpu * kChunk;
        kstop = min(kbeg + p.cpu * kChunk, kend);
    }
    const int t_begin = kbeg / kKeys;
    const int t_end = (kstop + kKeys - 1) / kKeys;
    const int n_it = t_end - t_begin;
    const int nck = (n_it + TPC - 1) / TPC;
    const int npages_need = (kend + 15) / 16;
    const int32_t *bt_row = p.block_tables + (int64_t)b * p.max_blocks;
    const int64_t unit_q = (int64_t)b * p.hkv + kvh;  // one query tile per request
    const int64_t rec_floats = part_record_floats(p.ws_rows, DH);
    const int64_t rec_hdr = part_header_floats(p.ws_rows);

    auto load16 = [&](int t) {
        const int pg = t * PPT + lane;
        return (lane < 16 && pg < npages_need) ? __ldg(bt_row + pg) : 0;
    };
    int ids_cur = (warp == 0) ? load16(t_begin) : 0;

    // -------------------------------------------------------------- setup --
    if (tid == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < NSK; ++s) {
            mbar_init(bar(B_KF + s), 1);
            mbar_init(bar(B_KE + s), 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(bar(B_VF + s), 1);
            mbar_init(bar(B_VE + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_SF + i), 1);
            mbar_init(bar(B_PF + i), 4);  // the four softmax warps
            mbar_init(bar(B_PV + i), 1);
            mbar_init(bar(B_CR + i), 4);  // the four softmax warps, at a chunk's end
            mbar_init(bar(B_OF + i), 4);  // the four epilogue warps have read the chunk's O^T
            mbar_init(bar(B_OD + i), 1);
        }
        mbar_init(bar(B_PROD), 1);
        mbar_init(bar(B_DONE), 1);
        mbar_init(bar(B_VZ), 1);
        sflags[0] = 0;
        sflags[3] = 0;
        sflags[4] = 0;
        sflags[5] = 0;
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
    // the last tile runs past kend: V rows of keys >= kend are zeroed after they land
    auto zero_tile = [&](int t) { return (t + 1) * kKeys > kend; };

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        bool ok = true, any_bad = false;
        int last_k_use[NSK], last_v_use[NSV];
        for (int s = 0; s < NSK; ++s) last_k_use[s] = -1;
        for (int s = 0; s < NSV; ++s) last_v_use[s] = -1;
        // Q: the box holds G heads x (NR / G) tokens per 64-column block
        const int tqd = NR / G;
        if (lane == 0)
            mbar_arrive_expect_tx(bar(B_Q), NKB * 128 * G * tqd);
        __syncwarp();
        if (lane < NKB)
            tma_load_3d(smem_addr(sQ + lane * QBLK), &p.tm_q, bar(B_Q), lane * 64, kvh * G, (int)tok_first);
        if (p.early_reads)
            griddep_wait();  // the cache write has completed and is visible
        int ids_next = 0;
        for (int it = 0; ok && it < n_it; ++it) {
            const int t = t_begin + it;
            if (it % TPL == 0) {
                if (it > 0)
                    ids_cur = ids_next;
                if (it + TPL < n_it)
                    ids_next = load16(t + TPL);
            }
            int id = __shfl_sync(0xffffffffu, ids_cur, (it % TPL) * PPT + (lane % PPT));
            const int np = min(PPT, npages_need - t * PPT);
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
                tma_load_4d(smem_addr(sK + sk * KST + kb * KBLK + pg * 2048), &p.tm_k, bar(B_KF + sk), kb * 64, kvh,
                            0, pid);
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
                tma_load_4d(smem_addr(sV + sv * KST + kb * KBLK + pg * 2048), &p.tm_v, bar(B_VF + sv), kb * 64, kvh,
                            0, pid);
            last_v_use[sv] = uv;
        }
        // zero the last tile's V rows of keys >= kend once it has landed, then
        // release the MMA issuer (stale or poisoned rows never meet P = 0)
        if (ok && n_it > 0 && zero_tile(t_end - 1)) {
            const int j = n_it - 1, sv = j % NSV, t = t_end - 1;
            const bool okz = __all_sync(0xffffffffu, wb(B_VF + sv, (j / NSV) & 1));
            if (okz) {
                const int row0 = kend - t * kKeys;
                const int nz = (kKeys - row0) * NKB * 8;
                uint8_t *vs = sV + sv * KST;
                for (int idx = lane; idx < nz; idx += 32) {
                    const int row = row0 + idx / (NKB * 8);
                    const int rem = idx % (NKB * 8);
                    *reinterpret_cast<uint4 *>(vs + (rem / 8) * KBLK + row * 128 + (rem % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(B_VZ));
            }
        }
        if (lane == 0) {
            if (any_bad) {
                record_error(p.err, kErrBadMetadata, b);
                sflags[3] = 1;
            }
            mbar_arrive(bar(B_PROD));
            if (!ok) {
                for (int s = 0; s < NSK; ++s)
                    if (last_k_use[s] >= 0)
                        wait_bar_drain(bar(B_KF + s), last_k_use[s] & 1);
                for (int s = 0; s < NSV; ++s)
                    if (last_v_use[s] >= 0)
                        wait_bar_drain(bar(B_VF + s), last_v_use[s] & 1);
                wait_bar_drain(bar(B_Q), 0);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer --
        // QK(0), QK(1), then PV(j) followed by QK(j+2): QK(j+2) overwrites the
        // S^T buffer and, through its commit, tells the softmax that PV(j) --
        // the last reader of P^T buffer j % 2 -- has completed.
        bool ok = true;
        if (lane == 0) {
            ok = wb(B_Q, 0);
            auto issue_qk = [&](int it) {
                const int sk = it % NSK;
                const uint32_t k0 = smem_addr(sK + sk * KST), q0 = smem_addr(sQ);
                tc_fence_after();
                uint64_t ad[8], bd[8];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    ad[kk] = sdesc_sw128(k0 + (kk / 4) * KBLK + (kk % 4) * 32, 16, 1024);
                    bd[kk] = sdesc_sw128(q0 + (kk / 4) * QBLK + (kk % 4) * 32, 16, 1024);
                }
                mma8_ss<1>(tmem + kSCol + (uint32_t)(it & 1) * 32, ad, bd, ID_QK, 0u);
                mma_commit(bar(B_KE + sk));
                mma_commit(bar(B_SF + (it & 1)));
            };
            auto issue_pv = [&](int j) -> bool {
                const int sv = j % NSV;
                const int t = t_begin + j;
                const bool chunk_first = (t * kKeys) % kChunk == 0;
                const int k = (t * kKeys - kbeg) / kChunk;  // chunk of this CTA
                bool okj = zero_tile(t) ? wb(B_VZ, 0) : wb(B_VF + sv, (j / NSV) & 1);
                if (okj)
                    okj = wb(B_PF + (j & 1), (j >> 1) & 1);
                if (okj && chunk_first && k >= 2)
                    okj = wb(B_OF + (k & 1), ((k >> 1) - 1) & 1);  // chunk k-2 has been read
                if (okj) {
                    tc_fence_after();
                    const uint32_t v0 = smem_addr(sV + sv * KST), p0 = smem_addr(sP + (j & 1) * PBUF);
                    uint64_t ad[8], bd[8];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        ad[kk] = sdesc_sw128(v0 + kk * 2048, KBLK, 1024);  // 16 keys per step, MN-major
                        bd[kk] = sdesc_sw128(p0 + (kk / 4) * PBLK + (kk % 4) * 32, 16, 1024);
                    }
                    mma8_ss<1>(tmem + kOCol + (uint32_t)(k & 1) * 32, ad, bd, ID_PV, chunk_first ? 0u : 1u);
                    mma_commit(bar(B_VE + sv));
                    mma_commit(bar(B_PV + (j & 1)));
                    // the chunk's last tile: its O^T is complete.  One phase per
                    // chunk of this parity, and chunk k + 2's first P.V waits for
                    // the epilogue to have read chunk k, so the epilogue's wait
                    // is never two phases behind.
                    if (j == n_it - 1 || ((t + 1) * kKeys) % kChunk == 0)
                        mma_commit(bar(B_OD + (k & 1)));
                }
                return okj;
            };
            for (int it = 0; ok && it < min(2, n_it); ++it) {
                ok = wb(B_KF + it % NSK, (it / NSK) & 1);
                if (ok)
                    issue_qk(it);
            }
            for (int j = 0; ok && j < n_it; ++j) {
                ok = issue_pv(j);
                if (ok && j + 2 < n_it) {
                    ok = wb(B_KF + (j + 2) % NSK, ((j + 2) / NSK) & 1);
                    if (ok)
                        issue_qk(j + 2);
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
        for (int it = 0; it < n_it; ++it) {
            const int t = t_begin + it;
            const int sb = it & 1;
            bool okw = !failed && wb(B_SF + sb, (it >> 1) & 1);
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
                const float tmax = __fmul_rn(fmaxf(fmaxf(s_xmax[n], s_xmax[32 + n]), fmaxf(s_xmax[64 + n], s_xmax[96 + n])),
                                             p.scale_log2);
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
                pv[n] = (n >= nlo && n < rv) ? ex2(__fmaf_rn(__uint_as_float(sr[n]), p.scale_log2, -m_run[n])) : 0.f;
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
            fence_proxy_async_smem();
            named_sync(2, 128);  // P^T and p complete; every thread has read the row maxima
            const int kc = (t * kKeys - kbeg) / kChunk;
            // O^T of this chunk must hold PV(it - 1) before it is rescaled
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
            const bool chunk_end = (it == n_it - 1) || ((t + 1) * kKeys) % kChunk == 0;
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
    } else if (warp >= 8) {
        // --------------------------------------------------- chunk epilogue --
        const int d = tid - 256;  // head-dim element = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
        float acc[R];  // in-CTA fold: the folded O^T column entries of element d
#pragma unroll
        for (int n = 0; n < R; ++n)
            acc[n] = 0.f;
        if (d < 32) {
            s_accml[2 * d] = -INFINITY;  // the folded (m, l) of row d
            s_accml[2 * d + 1] = 0.f;
        }
        named_sync(3, 128);
        for (int k = 0; k < nck; ++k) {
            const bool final_chunk = (k == nck - 1);
            bool ok = wb(B_CR + (k & 1), (k >> 1) & 1);
            if (ok)
                ok = wb(B_OD + (k & 1), (k >> 1) & 1);
            if (ok && final_chunk)
                ok = wb(B_PROD, 0);
            ok = __all_sync(0xffffffffu, ok);
            // the in-CTA fold shares the folded (m, l) through shared memory:
            // its four warps leave together (and this barrier also orders the
            // previous chunk's writes of it before this chunk's reads)
            if (!p.split) {
                if (named_sync_or(3, 128, !ok))
                    break;
            } else if (!ok) {
                break;
            }
            tc_fence_after();
            uint32_t o[R];
            tmem_ld_r<R>(tmem + lane_off + kOCol + (uint32_t)(k & 1) * 32, o);
            tmem_wait_ld();
            const float *ml = s_ml + (k & 1) * 64;  // the chunk's (m, l) per row
            const bool bad = final_chunk && sflags[3] != 0;
            const float qnan = __int_as_float(0x7FC00000);
            if (p.split) {
                // partial state of chunk c_grid*cpu + k: m, l, then the O rows
                float *part = p.ws_part + (unit_q * p.nch + (int64_t)c_grid * p.cpu + k) * rec_floats;
                if (d < rv) {
                    part[d] = bad ? 0.f : ml[2 * d];
                    part[p.ws_rows + d] = bad ? qnan : ml[2 * d + 1];
                }
#pragma unroll
                for (int n = 0; n < R; ++n)
                    if (n < rv)
                        __stcg(part + rec_hdr + (int64_t)n * DH + d, bad ? qnan : __uint_as_float(o[n]));
            } else {
                float fm_own = 0.f, fl_own = 0.f;  // row d's folded (m, l)
#pragma unroll
                for (int n = 0; n < R; ++n) {
                    if (n >= rv)
                        continue;
                    const Fold f = fold_coef(s_accml[2 * n], s_accml[2 * n + 1], ml[2 * n], ml[2 * n + 1]);
                    const float v = fold_elem(acc[n], __uint_as_float(o[n]), f);
                    if (final_chunk) {
                        const int64_t tok = tok_first + n / G;
                        const int head = kvh * G + n % G;
                        p.out[(tok * p.hq + head) * DH + d] =
                            bad ? __ushort_as_bfloat16(0x7FC0) : __float2bfloat16_rn(__fmul_rn(v, __frcp_rn(f.l)));
                        if (d == n && p.lse)
                            p.lse[tok * p.hq + head] = bad ? qnan : lse_of(f.m, f.l);
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
        }
        // Split-KV: arrive as soon as the records are written (also after a
        // failed wait, so the group's count completes)
        if (p.split)
            dec_arrive(p, unit_q, (nchunks + p.cpu - 1) / p.cpu, &sflags[2]);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // The last arrival folds, with every thread: all of this CTA's MMAs and
    // copies have completed, so the K/V stage area is free.
    if (p.split && sflags[2])
        dec_merge<R>(p, unit_q, nchunks, rv, tok_first, kvh, merge_work, kMergeWorkFloats);
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

int decode_rows(const AttnPlan &pl, int32_t max_query_len)
{
    if (pl.head_dim != 128 || pl.kt != 128 || pl.cl != 1 || pl.qtiles != 1)
        return 0;
    const long long rows = (long long)pl.group * max_query_len;
    for (int r = 4; r <= 32; r *= 2)
        if (rows <= r)
            return r;
    return 0;
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
    cfg.gridDim = dim3((unsigned)pl.grid);
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

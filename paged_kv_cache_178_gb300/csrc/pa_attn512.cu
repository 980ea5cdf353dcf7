// K2 for head dim 512: a two-CTA cluster per 128-row tile.
//
// A 128 x 512 FP32 output accumulator alone would fill a CTA's 512 TMEM
// columns, so the head dimension is split across a CTA pair ("harden compact
// peer-local KV prefill for Gemma-4", Scope: Hq=16, Hkv=2, d=512; here both
// CTAs of the pair sit on one GPU).  CTA rank c of the pair owns columns
// [256c, 256c+256) of Q, K, V and O:
//   - its Q half lives in TMEM (BF16, two per column) and is the A operand of
//     S_c = Q_c . K_c^T, the partial scores over its 256 columns;
//   - each CTA writes its partial S into the peer's shared memory (DSMEM) and
//     reads the peer's, then both form S = S_0 + S_1 (IEEE addition is
//     commutative, so both CTAs hold the same bits) and run the identical
//     softmax, so P, m and l agree bit for bit across the pair;
//   - P (BF16) goes to one shared-memory buffer in the K-major swizzled
//     layout of an MMA operand, and O_c += P . V_c (N = 256, both operands
//     from shared memory) accumulates in the CTA's own TMEM.  With P out of
//     the S buffers, Q.K^T of tile j + 2 may start as soon as S of tile j has
//     been read, two tiles ahead of P.V, so the score exchange of a tile
//     overlaps the softmax of the tile before.
// Warp roles (512 threads):
//   warp 0       K producer: one 64-column box per 16-token page, this CTA's
//                four column blocks, block ids range-checked as it goes
//   warp 2       V producer, the same for V (K never waits behind a V load)
//   warp 1       tcgen05 issuer: Q.K^T(it), then P.V(it - 2)
//   warps 4-11   softmax, two 32-column halves, one TMEM lane (row) each
//   warps 12-15  Q into TMEM, then the score sending, then the epilogue
// The fixed arithmetic follows the head-dim 128/256 kernel, with KV tiles of
// 64 keys (C1 at head dim 512) and 32-column softmax halves:
//   tile sum = (8-way interleaved sum of the half's 32 columns) for each half,
//   half0 + half1; one chunk per row (no split-KV at head dim 512).
#include <cstdio>
#include <cstring>

#include "pa_attn_common.cuh"

namespace pa {

namespace d512 {

constexpr int kKeys = 64;               // keys per KV tile
constexpr int kHalfCols = 256;          // head-dim columns per CTA of the pair
constexpr int kNKB = kHalfCols / 64;    // 64-column blocks per half
constexpr int kTileBytes = kNKB * kKeys * 128;  // one KV half tile (32 KB)
constexpr int kStagesK = 2, kStagesV = 2;
// Partial-score exchange buffer of one S buffer: [2 halves][8 blocks of 4
// columns][128 rows] of float4, so the 16-byte stores of a warp's 32 rows
// into the peer (and their loads here) cover 512 contiguous bytes
constexpr int kXBytes = 2 * 8 * kRows * 16;
constexpr int kPBytes = kRows * kKeys * 2;  // P of one tile: 128 rows x 64 keys, BF16
constexpr int kSmallBytes = 512 + 64 + 2 * 2 * kRows * 4 + kRows * 2 * 4;
constexpr uint32_t kQCol = 0;           // TMEM: Q half (128 columns of BF16 pairs)
constexpr uint32_t kSCol = 128;         // TMEM: two S buffers of 64 columns
constexpr uint32_t kOCol = 256;         // TMEM: O half (256 columns)

constexpr size_t smem_bytes()
{
    return 1024 + (size_t)kTileBytes * (kStagesK + kStagesV) + 2 * (size_t)kXBytes + kPBytes + kSmallBytes;
}

}  // namespace d512

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(512, 1) attn512_kernel(const __grid_constant__ AttnParams p)
{
    using namespace d512;
    constexpr int DH = 512;
    constexpr int NSK = kStagesK, NSV = kStagesV;
    constexpr uint32_t ID_QK = idesc_bf16_f32(kRows, kKeys, false);
    constexpr uint32_t ID_PV = idesc_bf16_f32(kRows, kHalfCols, true);
    constexpr int B_Q = 0, B_KF = 1, B_KE = B_KF + NSK, B_VF = B_KE + NSK, B_VE = B_VF + NSV;
    constexpr int B_SF = B_VE + NSV, B_PF = B_SF + 2, B_PV = B_PF + 2, B_XF = B_PV + 2, B_XE = B_XF + 2;
    constexpr int B_XS = B_XE + 2;  // the sending and softmax warps have read S of this buffer
    constexpr int B_FIN = B_XS + 2, B_PROD = B_FIN + 1, B_DONE = B_PROD + 1, NBARS = B_DONE + 1;
    static_assert(NBARS * 8 <= 512, "barrier area");
    static_assert(smem_bytes() <= kMaxSmemPerBlock, "shared-memory layout");

    // launched with programmatic stream serialization: no global read before
    // the preceding grid of the stream has completed
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sK = smem;
    uint8_t *sV = sK + NSK * kTileBytes;
    float4 *sX = reinterpret_cast<float4 *>(sV + NSV * kTileBytes);  // [2 S buffers][2 halves][8][128]
    uint8_t *sP = reinterpret_cast<uint8_t *>(sX) + 2 * kXBytes;  // P, 8-row groups of 1024 bytes, swizzled
    uint8_t *small = sP + kPBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(small);
    int *sflags = reinterpret_cast<int *>(small + 512);  // [0] abort [1] tmem [3] bad
    float *s_x = reinterpret_cast<float *>(small + 512 + 64);   // [2 exchanges][2 halves][128]
    float *s_ml = s_x + 2 * 2 * kRows;                          // [128][2]
    volatile int *abort_flag = sflags;
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    auto wb = [&](int i, uint32_t parity) { return wait_bar(bar(i), parity, abort_flag, p.err, i); };
    auto wbc = [&](int i, uint32_t parity) { return wait_bar_cluster(bar(i), parity, abort_flag, p.err, i); };
    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const uint32_t crank = cluster_ctarank();
    const uint32_t peer = crank ^ 1u;

    // ---------------------------------------------------------- work unit --
    // both CTAs of a pair take the same unit, longest work first
    const long long u = blockIdx.x >> 1;
    const long long nbh = (long long)p.num_seqs * p.hkv;
    const int qt = p.qtiles - 1 - (int)(u / nbh);
    const int kvh = (int)((u % nbh) % p.hkv);
    const int b = (int)((u % nbh) / p.hkv);
    const ReqMeta meta = read_meta(p, b);
    const int qs = meta.qs, qn = meta.qn, L = meta.L;
    const int tok0 = qt * p.tq;
    if (!meta.ok) {
        if (crank == 0) {
            if (qt == p.qtiles - 1 && tid == 0)
                record_error(p.err, kErrBadMetadata, b);
            if (meta.sane && tok0 < qn)
                write_nan_rows<DH>(p, (int64_t)qs + tok0, min(p.tq, qn - tok0), kvh);
        }
        return;
    }
    if (tok0 >= qn)
        return;
    const int ntok = min(p.tq, qn - tok0);
    const int rows_valid = ntok * p.group;
    const int64_t tok_first = (int64_t)qs + tok0;
    const int kend = L - qn + tok0 + ntok;
    const int n_it = (kend + kKeys - 1) / kKeys;
    const int npages_need = (kend + 15) / 16;
    const int32_t *bt_row = p.block_tables + (int64_t)b * p.max_blocks;
    auto load8 = [&](int t) {  // block ids of tiles t and t+1 (4 pages each)
        const int pg = t * 4 + lane;
        return (lane < 8 && pg < npages_need) ? __ldg(bt_row + pg) : 0;
    };
    int ids_cur = (warp == 0 || warp == 2) ? load8(0) : 0;

    // -------------------------------------------------------------- setup --
    if (tid == 0) {
        mbar_init(bar(B_Q), 4);
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
            mbar_init(bar(B_PF + i), 8);
            mbar_init(bar(B_PV + i), 1);
            mbar_init(bar(B_XF + i), 1);  // armed for each tile; the peer's rows land as its bytes
            mbar_init(bar(B_XE + i), 1);  // the peer's softmax threads have read what we wrote
            mbar_init(bar(B_XS + i), 12);  // the four sending warps and the eight softmax warps
        }
        mbar_init(bar(B_FIN), 8);
        mbar_init(bar(B_PROD), 1);
        mbar_init(bar(B_DONE), 1);
        // the exchange buffers' first phases (tiles 0 and 1); each later
        // phase is armed by the softmax once it has read the phase before
        for (int i = 0; i < 2 && i < n_it; ++i)
            mbar_arrive_expect_tx(bar(B_XF + i), kXBytes);
        sflags[0] = 0;
        sflags[3] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&sflags[1]), 512);
        tmem_relinquish();
    }
    if (tid == 64) {
        prefetch_tensormap(&p.tm_k);
        prefetch_tensormap(&p.tm_v);
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(sflags[1]);

    if (warp == 0 || warp == 2) {
        // ------------------------------------- producers: K (warp 0), V (warp 2) --
        // One warp per operand: a K tile is issued as soon as its stage is
        // free, not behind the V load of the tile before (which waits for the
        // P.V of two tiles back).  Both warps read the block ids; warp 0
        // reports bad ones.
        static_assert(NSK == NSV, "one stage count for both producers");
        constexpr int NS = NSK;
        const bool is_v = warp == 2;
        const int B_F = is_v ? B_VF : B_KF, B_E = is_v ? B_VE : B_KE;
        const CUtensorMap *tm = is_v ? &p.tm_v : &p.tm_k;
        uint8_t *const sbase = is_v ? sV : sK;
        bool ok = true, any_bad = false;
        int last_use[NS];
        for (int s = 0; s < NS; ++s) last_use[s] = -1;
        int ids_next = 0;
        for (int it = 0; ok && it < n_it; ++it) {
            if ((it & 1) == 0) {
                if (it > 0)
                    ids_cur = ids_next;
                if (it + 2 < n_it)
                    ids_next = load8(it + 2);
            }
            int id = __shfl_sync(0xffffffffu, ids_cur, (it & 1) * 4 + (lane & 3));
            const int np = min(4, npages_need - it * 4);
            const bool badl = lane < np && (id < 0 || (int64_t)id >= p.num_blocks);
            if (badl)
                id = 0;
            any_bad |= __any_sync(0xffffffffu, badl);
            const int my_page = lane / kNKB, my_kb = lane % kNKB;
            const int my_id = __shfl_sync(0xffffffffu, id, my_page & 3);
            const bool issue = lane < np * kNKB;
            const int col = (int)crank * kHalfCols + my_kb * 64;
            const int st = it % NS, use = it / NS;
            if (lane == 0) {
                if (use >= 1)
                    ok = wb(B_E + st, (use - 1) & 1);
                if (ok)
                    mbar_arrive_expect_tx(bar(B_F + st), np * kNKB * 2048);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            if (issue)
                tma_load_4d(smem_addr(sbase + st * kTileBytes + my_kb * 8192 + my_page * 2048), tm, bar(B_F + st),
                            col, kvh, 0, my_id);
            last_use[st] = use;
        }
        if (lane == 0) {
            if (!is_v) {
                if (any_bad) {
                    record_error(p.err, kErrBadMetadata, b);
                    sflags[3] = 1;
                }
                mbar_arrive(bar(B_PROD));
            }
            if (!ok)
                for (int s = 0; s < NS; ++s)
                    if (last_use[s] >= 0)
                        wait_bar_drain(bar(B_F + s), last_use[s] & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer --
        bool ok = true;
        if (lane == 0)
            ok = wb(B_Q, 0);  // Q half in TMEM
        ok = __shfl_sync(0xffffffffu, ok, 0);
        auto issue_pv = [&](int j) -> bool {
            const int sv = j % NSV;
            bool okj = __all_sync(0xffffffffu, wb(B_VF + sv, (j / NSV) & 1));
            if (!okj)
                return false;
            if ((j + 1) * kKeys > kend) {
                const int row0 = kend - j * kKeys;
                const int nz = (kKeys - row0) * kNKB * 8;
                uint8_t *vs = sV + sv * kTileBytes;
                for (int idx = lane; idx < nz; idx += 32) {
                    const int row = row0 + idx / (kNKB * 8);
                    const int rem = idx % (kNKB * 8);
                    *reinterpret_cast<uint4 *>(vs + (rem / 8) * 8192 + row * 128 + (rem % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) {
                okj = wb(B_PF + (j & 1), (j >> 1) & 1);
                if (okj) {
                    tc_fence_after();
                    const uint32_t pbase = smem_addr(sP);
                    const uint32_t vbase = smem_addr(sV + sv * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk) {
                        const uint64_t ad = sdesc_sw128(pbase + kk * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(vbase + kk * 2048, 8192, 1024);
                        mma_bf16_ss(tmem + kOCol, ad, bd, ID_PV, (kk > 0 || j > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(B_VE + sv));
                    mma_commit(bar(B_PV + (j & 1)));
                }
            }
            return __shfl_sync(0xffffffffu, okj, 0);
        };
        // Q.K^T(it), then P.V(it - 2): Q.K^T runs two tiles ahead
        for (int it = 0; ok && it <= n_it + 1; ++it) {
            if (it < n_it) {
                const int sk = it % NSK;
                if (lane == 0) {
                    ok = wb(B_KF + sk, (it / NSK) & 1);
                    // S buffer it & 1 was last read for tile it - 2 (sending and softmax warps)
                    if (ok && it >= 2)
                        ok = wb(B_XS + (it & 1), ((it >> 1) - 1) & 1);
                    if (ok) {
                        tc_fence_after();
                        const uint32_t kbase = smem_addr(sK + sk * kTileBytes);
#pragma unroll
                        for (int kk = 0; kk < kHalfCols / 16; ++kk) {
                            const uint64_t bd = sdesc_sw128(kbase + (kk / 4) * 8192 + (kk % 4) * 32, 16, 1024);
                            mma_bf16_ts(tmem + kSCol + (uint32_t)(it & 1) * kKeys, tmem + kQCol + kk * 8, bd, ID_QK,
                                        kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bar(B_KE + sk));
                        mma_commit(bar(B_SF + (it & 1)));
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
            if (ok && it >= 2)
                ok = issue_pv(it - 2);
        }
        if (lane == 0) {
            mma_commit(bar(B_DONE));
            wait_bar_drain(bar(B_DONE), 0);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12) {
        // --------------------------------------- softmax (2 halves, pair) --
        const int h = (warp - 4) / 4;
        const int q4 = warp % 4;
        const int r = q4 * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const bool row_valid = r < rows_valid;
        const bool warp_active = 32 * q4 < rows_valid;
        const int pos = L - qn + tok0 + r / p.group;
        float *xmax = s_x;
        float *xsum = s_x + 2 * kRows;
        float m = -INFINITY, l = 0.f;
        bool failed = false;
        for (int it = 0; it < n_it; ++it) {
            const int sb = it & 1;
            // own partial S from tensor memory (then the S buffer is released
            // for Q.K^T two tiles on), the peer's from the exchange buffer
            // (sent by the peer's sending warps as soon as its Q.K^T is done)
            bool okw = !failed && wb(B_SF + sb, (it >> 1) & 1);
            okw = __all_sync(0xffffffffu, okw);
            tc_fence_after();
            const uint32_t scol = tmem + lane_off + kSCol + sb * kKeys + 32 * h;
            uint32_t v[32];
            if (okw) {
                tmem_ld32(scol, v);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (okw && lane == 0)
                mbar_arrive(bar(B_XS + sb));
            if (okw)
                okw = wbc(B_XF + sb, (it >> 1) & 1);
            okw = __all_sync(0xffffffffu, okw);
            float s[32];
            if (okw) {
                const float4 *src = sX + ((sb * 2 + h) * 8) * kRows + r;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 x = src[i * kRows];
                    s[4 * i + 0] = __fadd_rn(__uint_as_float(v[4 * i + 0]), x.x);
                    s[4 * i + 1] = __fadd_rn(__uint_as_float(v[4 * i + 1]), x.y);
                    s[4 * i + 2] = __fadd_rn(__uint_as_float(v[4 * i + 2]), x.z);
                    s[4 * i + 3] = __fadd_rn(__uint_as_float(v[4 * i + 3]), x.w);
                }
            }
            const int nallow = row_valid ? max(0, min(32, pos - it * kKeys - 32 * h + 1)) : 0;
            float pmax = -INFINITY;
            if (okw && warp_active) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pmax = (i < nallow) ? fmaxf(pmax, s[i]) : pmax;
            }
            xmax[h * kRows + r] = pmax;
            if (named_sync_or(1, 256, !okw)) {
                failed = true;
                break;
            }
            if (tid == 128) {
                // every softmax thread has read the peer's rows (their values fed
                // the barrier above): the buffer's barrier is armed for tile
                // it + 2 (its phase of tile it is complete, so the arming falls
                // in the next phase), then the buffer is handed back to the peer
                if (it + 2 < n_it)
                    mbar_arrive_expect_tx(bar(B_XF + sb), kXBytes);
                mbar_arrive_cluster_relaxed(mapa_shared(bar(B_XE + sb), peer));
            }
            const float tmax = __fmul_rn(fmaxf(xmax[r], xmax[kRows + r]), p.scale_log2);
            float m_new = m, corr = 1.f;
            bool need = false;
            if (tmax != -INFINITY) {
                if (m == -INFINITY) {
                    m_new = tmax;
                } else if (tmax > __fadd_rn(m, kTau)) {
                    m_new = tmax;
                    corr = ex2(__fsub_rn(m, m_new));
                    need = true;
                }
            }
            float hs = 0.f;
            bool okp = true;
            if (warp_active) {
                const float negm = -m_new;
                float a[8];
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float e0 = (i < nallow) ? ex2(__fmaf_rn(s[i], p.scale_log2, negm)) : 0.f;
                    float e1 = (i + 1 < nallow) ? ex2(__fmaf_rn(s[i + 1], p.scale_log2, negm)) : 0.f;
                    if (i < 8) {
                        a[i & 7] = e0;
                        a[(i + 1) & 7] = e1;
                    } else {
                        a[i & 7] = __fadd_rn(a[i & 7], e0);
                        a[(i + 1) & 7] = __fadd_rn(a[(i + 1) & 7], e1);
                    }
                    w[i / 2] = pack_bf16x2(e0, e1);
                }
                hs = __fadd_rn(__fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3])),
                               __fadd_rn(__fadd_rn(a[4], a[5]), __fadd_rn(a[6], a[7])));
                // the one P buffer was read by P.V(it - 1)
                okp = it == 0 || __all_sync(0xffffffffu, wb(B_PV + ((it - 1) & 1), ((it - 1) >> 1) & 1));
                // P of keys [32h, 32h+32): 16-byte chunks 4h..4h+3 of row r,
                // swizzled by the row within its 8-row group
                if (okp) {
                    uint8_t *prow = sP + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4 *>(prow + (((4 * h + q) ^ (r & 7)) << 4)) =
                            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                    fence_proxy_async_smem();  // visible to the MMA's operand reads
                }
            }
            xsum[h * kRows + r] = hs;
            if (named_sync_or(1, 256, !okp)) {
                failed = true;
                break;
            }
            const float tsum = __fadd_rn(xsum[r], xsum[kRows + r]);
            // O may be rescaled: P.V(it - 1) is complete (waited above by the
            // active warps; an inactive warp never needs a rescale)
            if (__any_sync(0xffffffffu, need)) {
                tc_fence_after();
                const float f = need ? corr : 1.f;
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    uint32_t o[32];
                    const uint32_t c = tmem + lane_off + kOCol + 128 * h + g * 32;
                    tmem_ld32(c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__fmul_rn(__uint_as_float(o[i]), f));
                    tmem_st32(c, o);
                }
            }
            tmem_wait_st();
            l = need ? __fadd_rn(__fmul_rn(l, corr), tsum) : __fadd_rn(l, tsum);
            m = m_new;
            const bool last = (it == n_it - 1);
            if (last && h == 0) {
                s_ml[r * 2] = m;
                s_ml[r * 2 + 1] = l;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_PF + sb));
                if (last)
                    mbar_arrive(bar(B_FIN));
            }
        }
    } else if (warp >= 12) {
        // ------------------- Q into TMEM, the score sending, then epilogue --
        const int q4 = warp % 4;
        const int r = q4 * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const bool row_valid = r < rows_valid;
        const int G = p.group;
        const int64_t tok = tok_first + r / G;
        const int head = kvh * G + r % G;
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const __nv_bfloat16 *>(p.q) + tok * p.q_tok_stride + (int64_t)head * DH +
                (int)crank * kHalfCols);
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 x = row_valid ? __ldg(src + g * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
                    w[4 * i] = x.x;
                    w[4 * i + 1] = x.y;
                    w[4 * i + 2] = x.z;
                    w[4 * i + 3] = x.w;
                }
                tmem_st32(tmem + lane_off + kQCol + g * 32, w);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_Q));
        }
        // ------------------------------------------------ sending warps --
        // This CTA's partial scores of tile it (both 32-column halves of row
        // r) into the peer's exchange buffer with st.async, as soon as Q.K^T
        // (it) is done and the peer has read what was sent two tiles ago;
        // the bytes complete the transaction count of the peer's barrier,
        // which the peer's softmax armed when it released the buffer (the
        // setup, for tiles 0 and 1).  The softmax of a tile thus finds the
        // peer's rows waiting.
        for (int it = 0; it < n_it; ++it) {
            const int sb = it & 1;
            bool okx = wb(B_SF + sb, (it >> 1) & 1);
            if (okx && it >= 2)
                okx = wbc(B_XE + sb, ((it >> 1) - 1) & 1);
            if (!__all_sync(0xffffffffu, okx))
                break;
            tc_fence_after();
            uint32_t v0[32], v1[32];
            tmem_ld32(tmem + lane_off + kSCol + sb * kKeys, v0);
            tmem_ld32(tmem + lane_off + kSCol + sb * kKeys + 32, v1);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_XS + sb));  // Q.K^T(it + 2) may overwrite this S buffer
            const uint32_t rbar = mapa_shared(bar(B_XF + sb), peer);
            const uint32_t d0 = mapa_shared(smem_addr(sX + ((sb * 2) * 8) * kRows + r), peer);
            const uint32_t d1 = mapa_shared(smem_addr(sX + ((sb * 2 + 1) * 8) * kRows + r), peer);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                st_async_v4(d0 + i * kRows * 16, v0[4 * i], v0[4 * i + 1], v0[4 * i + 2], v0[4 * i + 3], rbar);
                st_async_v4(d1 + i * kRows * 16, v1[4 * i], v1[4 * i + 1], v1[4 * i + 2], v1[4 * i + 3], rbar);
            }
        }
        bool ok = wb(B_FIN, 0);
        if (ok)
            ok = wb(B_PV + ((n_it - 1) & 1), ((n_it - 1) >> 1) & 1);
        if (ok)
            ok = wb(B_PROD, 0);
        if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            const float mr = s_ml[r * 2], lr = s_ml[r * 2 + 1];
            const bool bad = sflags[3] != 0;
            const float inv = __frcp_rn(lr);
#pragma unroll 1
            for (int g = 0; g < kHalfCols / 32; ++g) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + kOCol + g * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    o[i] = bad ? 0x7FC00000u : __float_as_uint(__fmul_rn(__uint_as_float(o[i]), inv));
                if (row_valid)
                    store_out32(p.out + (tok * p.hq + head) * DH + (int)crank * kHalfCols + g * 32, o);
            }
            if (row_valid && crank == 0 && p.lse)
                p.lse[tok * p.hq + head] = bad ? __int_as_float(0x7FC00000) : lse_of(mr, lr);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // neither CTA leaves while the peer may still write into its shared
    // memory or arrive on its barriers
    cluster_sync_all();
}

cudaError_t init_attention512_attributes()
{
    return cudaFuncSetAttribute(attn512_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)d512::smem_bytes());
}

cudaError_t launch_attention512(const AttnArgs &a, const AttnPlan &pl, ErrState *err, cudaStream_t stream)
{
    AttnParams p;
    memset(&p, 0, sizeof(p));
    {
        const cuuint64_t dims[4] = {512, (cuuint64_t)a.num_kv_heads, 16, (cuuint64_t)a.num_blocks};
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
    p.q = a.q;
    p.q_tok_stride = a.q_tok_stride;
    p.block_tables = a.block_tables;
    p.seq_lens = a.seq_lens;
    p.qsl = a.query_start_loc;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    p.err = err;
    p.num_q_tokens = a.num_q_tokens;
    p.num_blocks = a.num_blocks;
    p.max_blocks = a.max_blocks_per_seq;
    p.num_seqs = a.num_seqs;
    p.hq = a.num_q_heads;
    p.hkv = a.num_kv_heads;
    p.group = pl.group;
    p.tq = pl.tokens_per_tile;
    p.qtiles = pl.qtiles;
    p.nch = 1;
    p.max_query_len = a.max_query_len;
    p.max_seq_len = a.max_seq_len;
    p.split = 0;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = d512::smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn512_kernel, p);
}

}  // namespace pa

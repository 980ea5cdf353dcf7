// K2: paged grouped-query attention for sm_103a (head dims 128 and 256).
//
// One CTA owns a 128-row tile of (query token, query head) rows of one
// request and one KV head: row r = t*G + hh is query token t of the tile and
// query head kvh*G + hh, so the G heads sharing a KV head share every K/V
// tile ("test(rocm): ReshapeAndCache->PagedAttention composition at real
// dims", What changed: Hq=8, Hkv=2).  Roles (512 threads):
//   warp 0       TMA producer: Q once, then per KV tile one 64-column box
//                per 16-token page for K and for V, block ids read from the
//                request's table (and range-checked) as it goes; pages past
//                the last needed key are never read ("fix(rocm): stabilize
//                direct paged CK attention for bitwise R/R", Changes: tail-page
//                padding and sanitising).
//   warp 1       tcgen05 issuer: S = Q.K^T into TMEM (two buffers), then
//                O += P.V with P read from TMEM; zeroes V rows of keys past the
//                last needed key so a zero probability never meets garbage.
//   warps 4-11   softmax, two halves: warps 4-7 own score columns 0-63, warps
//                8-11 columns 64-127, one TMEM lane (row) per thread.
//   warps 12-15  correction: chunk folds, epilogue, split partial states.
// Prefill with two or more query tiles runs on CTA pairs that share each MMA
// (cta_group::2, M = 256), so each CTA loads half of every K/V tile; the
// single-CTA form serves split-KV decode and one-tile requests.
//
// Fixed arithmetic (same page, intro and Changes: one schedule for every
// shape, no implicit FMA contraction).  Every row follows the same sequence
// of operations whatever the batch, query length, other rows or launch
// bounds, so prefill and decode agree bit for bit:
//   C1  KV tiles of 128 keys (64: second canon) from key 0; K-steps of 16 up
//       order, BF16 in, FP32 accumulate (M = 128 per CTA, or 256 over a CTA
//       pair: each output element is the same dot product either way).
//   C2  c = scale*log2 e is formed once, in fp32, on the host (scale > 0).
//       Tile max in log2 units: (max of the raw scores S over allowed keys)
//       * c, one fp32 multiply.
//   C3  lazy online softmax over a chunk's tiles: the reference max m moves
//       only when a tile max exceeds m + 8 (then l and O are scaled by
//       exp2(m_old - m_new)); p = exp2(fma(S, c, -m)) for allowed keys,
//       exactly 0 otherwise.  Tile row sum: for each half of the columns an
//       8-way interleaved sum (accumulator k sums the half's columns k, k+8,
//       .. in order, then ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7))); tile sum =
//       half0 + half1.
//   C4  P rounded to BF16 (RNE) before P.V.
//   C5  head dim 128: chunks of 256 keys aligned to key 0, each starting
//       fresh; chunk states fold left to right with one fold function
//       (in-CTA for prefill, by the last-arriving CTA for split decode).
//       Head dim 256: one chunk (no split).
//   C6  out = O * rcp_rn(l) -> BF16 RNE; lse = (m + log2 l) * ln 2.
#include <cuda_bf16.h>

#include <atomic>
#include <cstdio>
#include <cstring>

#include "pa_attn_common.cuh"
#include "pa_split.cuh"

namespace pa {

constexpr int kThreads = 512;
constexpr int kSplitCtaThreshold = 152;

template <int DH>
struct Cfg;
template <>
struct Cfg<128> {
    static constexpr int kStagesK = 3;     // K smem stages (single CTA)
    static constexpr int kStagesV = 2;     // V smem stages (single CTA)
    static constexpr int kStagesKPair = 3; // K half-tile stages (CTA pair)
    static constexpr int kStagesVPair = 3; // V half-tile stages (CTA pair)
    static constexpr int kChunk = 256;     // keys per chunk (0 = one chunk)
    static constexpr int kOCol = 256;      // TMEM column of the chunk accumulator
    static constexpr int kAccCol = 384;    // TMEM column of the folded accumulator (single CTA)
};
template <>
struct Cfg<256> {
    static constexpr int kStagesK = 1;
    static constexpr int kStagesV = 1;
    static constexpr int kStagesKPair = 2;
    static constexpr int kStagesVPair = 2;
    static constexpr int kChunk = 0;
    static constexpr int kOCol = 256;
    static constexpr int kAccCol = -1;
};

// Small shared arrays after the tiles: barriers, flags, the two per-row
// exchange buffers of the softmax halves and the chunk (m, l) hand-off.
constexpr int kSmallBytes = 512 /*barriers*/ + 64 /*flags*/ + 2 * 2 * kRows * 4 + 2 * kRows * 2 * 4;

template <int DH>
constexpr size_t tile_bytes() { return (size_t)(DH / 64) * 16384; }

// One K stage: the KT-key tile, or with a CTA pair this CTA's KT/2 keys (all
// of the head dim).  One V stage: the KT-key tile, or with a pair this CTA's
// half of the head dim (all KT keys).
template <int DH, bool PAIR, int KT>
constexpr size_t k_stage_bytes() { return (size_t)(PAIR ? KT / 2 : KT) * DH * 2; }
template <int DH, bool PAIR, int KT>
constexpr size_t v_stage_bytes() { return (size_t)KT * (PAIR ? DH / 2 : DH) * 2; }

// Stage counts are set for 128-key tiles; 64-key tiles take twice as many
// stages of half the size, so the rings hold the same bytes (the split-KV
// merge stages its operands in them).
template <int DH, bool PAIR, int KT>
constexpr int stages_k() { return (PAIR ? Cfg<DH>::kStagesKPair : Cfg<DH>::kStagesK) * (128 / KT); }
template <int DH, bool PAIR, int KT>
constexpr int stages_v() { return (PAIR ? Cfg<DH>::kStagesVPair : Cfg<DH>::kStagesV) * (128 / KT); }

// CTA pairs with chunked heads keep two chunk accumulators in TMEM (columns
// kOCol and kOCol + 128, by chunk parity) so the next chunk's P.V never waits
// for the fold of the previous one; the folded accumulator then lives in
// shared memory (fp32, 128 rows).
template <int DH, bool PAIR>
constexpr bool acc_in_smem() { return PAIR && Cfg<DH>::kChunk > 0; }
template <int DH, bool PAIR>
constexpr size_t acc_smem_bytes() { return acc_in_smem<DH, PAIR>() ? (size_t)kRows * DH * 4 : 0; }

template <int DH, bool PAIR, int KT>
constexpr size_t smem_bytes()
{
    return 1024 /*alignment slack*/ + tile_bytes<DH>() /*Q*/ + k_stage_bytes<DH, PAIR, KT>() * stages_k<DH, PAIR, KT>() +
           v_stage_bytes<DH, PAIR, KT>() * stages_v<DH, PAIR, KT>() + acc_smem_bytes<DH, PAIR>() + kSmallBytes;
}

// Row r of the shared-memory accumulator, columns 32g .. 32g+31, as 32-bit
// words: 16-byte chunk c of a row sits at chunk (c ^ (r & 7)), so the eight
// rows of a quarter warp hit eight different bank groups.
template <int DH>
__device__ __forceinline__ void acc_row_load(const float4 *acc, int r, int g, uint32_t (&v)[32])
{
    const float4 *row = acc + (size_t)r * (DH / 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 x = row[(g * 8 + i) ^ (r & 7)];
        v[4 * i] = __float_as_uint(x.x);
        v[4 * i + 1] = __float_as_uint(x.y);
        v[4 * i + 2] = __float_as_uint(x.z);
        v[4 * i + 3] = __float_as_uint(x.w);
    }
}

template <int DH>
__device__ __forceinline__ void acc_row_store(float4 *acc, int r, int g, const uint32_t (&v)[32])
{
    float4 *row = acc + (size_t)r * (DH / 4);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        row[(g * 8 + i) ^ (r & 7)] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
}

// PAIR: the CTAs of a two-CTA cluster take query tiles 2g (rank 0, the
// leader) and 2g+1 of one (request, KV head) and share every MMA
// (cta_group::2, M = 256).  Each CTA loads half of each K tile (the leader
// the first half of the keys) and half of each V tile (the lower or upper
// half of the head dim), so a CTA moves half the bytes per score it computes.
// The leader's thread issues all MMAs; tile-full barriers, P-ready and
// fold-done barriers live in the leader, stage-release and S/PV-done commits
// go to both CTAs.  Every row still sees the same operation sequence (C1-C6).
template <int DH, bool PAIR, int KT>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ AttnParams p)
{
    using C = Cfg<DH>;
    constexpr int kKeys = KT;                        // keys per KV tile (the canon's tile: C1)
    constexpr int PPT = kKeys / 16;                  // pages per KV tile
    constexpr int TPL = 16 / PPT;                    // tiles whose block ids one 16-lane read covers
    constexpr int HALF = kKeys / 2;                  // score columns per softmax half
    constexpr int NPV = kKeys / 16;                  // K-steps of one P.V (16 keys each)
    static_assert(KT == 128 || (KT == 64 && DH == 128), "KV tile");
    constexpr int NKB = DH / 64;                     // 64-column (128-byte) blocks of the head dim
    constexpr int TILE_BYTES = (int)tile_bytes<DH>();  // 128 rows x DH BF16 (the Q tile)
    constexpr int NSK = stages_k<DH, PAIR, KT>();
    constexpr int NSV = stages_v<DH, PAIR, KT>();
    constexpr int KST = (int)k_stage_bytes<DH, PAIR, KT>();
    constexpr int VST = (int)v_stage_bytes<DH, PAIR, KT>();
    constexpr int KBLK = (PAIR ? kKeys / 2 : kKeys) * 128;  // bytes of one 64-column block of a K stage
    constexpr int VBLK = kKeys * 128;                // bytes of one 64-column block of a V stage
    constexpr int VKB = PAIR ? NKB / 2 : NKB;        // 64-column blocks of a V stage
    constexpr int CL = PAIR ? 2 : 1;
    constexpr bool CHUNKED = C::kChunk > 0;
    constexpr int CHUNK_DIV = CHUNKED ? C::kChunk : 1;  // divisor used only when CHUNKED
    constexpr int TPC = CHUNKED ? C::kChunk / kKeys : 1;  // tiles per chunk
    constexpr uint32_t ACC_COL = C::kAccCol < 0 ? 0u : (uint32_t)C::kAccCol;
    constexpr bool ACC_SMEM = acc_in_smem<DH, PAIR>();  // folded accumulator in shared memory
    constexpr bool OBUF2 = ACC_SMEM;                        // two chunk accumulators (by chunk parity)
    constexpr int NSB = 2;                                  // S/P buffers in TMEM
    // TMEM column of chunk k's accumulator
    auto ocol = [](int k) { return (uint32_t)C::kOCol + (OBUF2 ? (uint32_t)(k & 1) * 128u : 0u); };
    constexpr uint32_t ID_QK = idesc_bf16_f32(CL * kRows, kKeys, false);
    constexpr uint32_t ID_PV = idesc_bf16_f32(CL * kRows, DH, true);
    // barrier slots
    constexpr int B_Q = 0, B_KF = 1, B_KE = B_KF + NSK, B_VF = B_KE + NSK, B_VE = B_VF + NSV;
    constexpr int B_SF = B_VE + NSV, B_PF = B_SF + NSB, B_PV = B_PF + NSB, B_CR = B_PV + 2;
    constexpr int B_OF = B_CR + 2, B_PROD = B_OF + (OBUF2 ? 2 : 1), B_DONE = B_PROD + 1, B_VZ = B_DONE + 1;
    constexpr int NBARS = B_VZ + 1;
    static_assert(NBARS * 8 <= 512, "barrier area");
    static_assert(smem_bytes<DH, PAIR, KT>() <= kMaxSmemPerBlock, "shared-memory layout");

    // Launched with programmatic stream serialization.  By default nothing
    // below reads global memory before the preceding grid of the stream has
    // completed.  With early_reads the preceding grid writes only the K/V
    // pool: metadata, block tables and Q are read at once and the producer
    // waits just before its first K/V copy.
    if (!p.early_reads)
        griddep_wait();
    // a grid launched after this one with programmatic serialization may be
    // scheduled now (it waits for this grid before it reads our results)
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived by indexing the shared array so the
    // compiler keeps every access in the shared state space
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem;
    uint8_t *sK = sQ + TILE_BYTES;
    uint8_t *sV = sK + NSK * KST;
    float4 *sAcc = reinterpret_cast<float4 *>(sV + NSV * VST);  // [128 rows][DH/4], 16-byte chunks XOR-swizzled
    uint8_t *small = sV + NSV * VST + acc_smem_bytes<DH, PAIR>();
    uint64_t *bars = reinterpret_cast<uint64_t *>(small);
    int *sflags = reinterpret_cast<int *>(small + 512);  // [0] abort [1] tmem [2] last [3] bad
    float *s_x = reinterpret_cast<float *>(small + 512 + 64);   // [2 exchanges][2 halves][128]
    float *s_ml = s_x + 2 * 2 * kRows;                          // [2 chunk parities][128][2]
    volatile int *abort_flag = sflags;
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    // bounded wait on barrier slot i for the given phase parity
    auto wb = [&](int i, uint32_t parity) { return wait_bar(bar(i), parity, abort_flag, p.err, i); };
    // the same for a barrier that the other CTA of a pair arrives on (acquire at
    // cluster scope)
    auto wbc = [&](int i, uint32_t parity) {
        return PAIR ? wait_bar_cluster(bar(i), parity, abort_flag, p.err, i) : wait_bar(bar(i), parity, abort_flag, p.err, i);
    };
    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    float *const merge_work = reinterpret_cast<float *>(sK);
    constexpr int kMergeWorkFloats = (NSK * KST + NSV * VST) / 4;
    // the split-KV merge's worst case (128 rows, one folder, one chunk per
    // segment): running O, two (m, l) rows, then m/l, O, coefficients and
    // mode of one chunk, with rounding slack.  Split-KV runs single CTAs.
    static_assert(PAIR || !(C::kChunk > 0) || kMergeWorkFloats >= kRows * DH + 4 * kRows + kRows * (DH + 5) + 16,
                  "split-KV merge staging does not fit the K/V stage area");

    // ---------------------------------------------------------- work unit --
    int b, kvh, qt, c_grid = 0;
    bool split_multi = false;  // the last arrivals share the fold (all units resident)
    ReqMeta meta;
    if (p.split) {
        const Unit un = split_unit(p, CHUNK_DIV, reinterpret_cast<int *>(s_x));
        if (!un.valid)
            return;
        b = un.b;
        kvh = un.kvh;
        qt = un.qt;
        c_grid = un.c;
        meta = un.meta;
        split_multi = un.total <= p.num_sms;
    } else {
        // longest work first: later query tiles see more keys.  With cl = 2
        // the CTA pair takes query tiles 2g and 2g+1 of one (request, KV head).
        const long long u = blockIdx.x / CL;
        const long long nbh = (long long)p.num_seqs * p.hkv;
        const int g = (PAIR ? p.npairs : p.qtiles) - 1 - (int)(u / nbh);
        qt = PAIR ? 2 * g + (int)cluster_ctarank() : g;
        kvh = (int)((u % nbh) % p.hkv);
        b = (int)((u % nbh) / p.hkv);
        meta = read_meta(p, b);
    }
    const int qs = meta.qs, qn = meta.qn, L = meta.L;
    const int tok0 = qt * p.tq;
    if (!meta.ok) {
        if (tid == 0 && (p.split || qt == 0))
            record_error(p.err, kErrBadMetadata, b);
        if (meta.sane && tok0 < qn)
            write_nan_rows<DH>(p, (int64_t)qs + tok0, min(p.tq, qn - tok0), kvh);
        return;  // the pair partner (same request) leaves too
    }
    // A CTA of a pair whose tile lies past the request still runs the shared
    // K/V pipeline (with no rows of its own) while its partner has work.
    const int qt_base = PAIR ? (qt & ~1) : qt;
    if (qt_base * p.tq >= qn)
        return;  // the whole pair (or the single CTA) has nothing to do
    const int ntok = max(0, min(p.tq, qn - tok0));
    const int rows_valid = ntok * p.group;
    const int64_t tok_first = (int64_t)qs + tok0;
    // keys [0, kend) are needed by some row of the pair
    const int last_tok = min(qn, (qt_base + CL) * p.tq);
    const int kend = L - qn + last_tok;
    const int nchunks = CHUNKED ? (kend + CHUNK_DIV - 1) / CHUNK_DIV : 1;
    int kbeg = 0, kstop = kend;
    if (p.split) {
        // this CTA's consecutive chunks [c_grid*cpu, c_grid*cpu + cpu)
        kbeg = c_grid * p.cpu * CHUNK_DIV;
        kstop = min(kbeg + p.cpu * CHUNK_DIV, kend);
    }
    const int t_begin = kbeg / kKeys;
    const int t_end = (kstop + kKeys - 1) / kKeys;
    const int n_it = t_end - t_begin;
    const int nck = CHUNKED ? (n_it + TPC - 1) / TPC : 1;  // chunks this CTA processes
    const int npages_need = (kend + 15) / 16;
    const int32_t *bt_row = p.block_tables + (int64_t)b * p.max_blocks;
    const int64_t unit_q = ((int64_t)b * p.hkv + kvh) * p.qtiles + qt;
    const int64_t rec_floats = part_record_floats(p.ws_rows, DH);
    const int64_t rec_hdr = part_header_floats(p.ws_rows);

    // The producer's first 16 block ids (TPL tiles) are requested before the
    // set-up barrier so the load overlaps it.
    auto load16 = [&](int t) {
        const int pg = t * PPT + lane;
        return (lane < 16 && pg < npages_need) ? __ldg(bt_row + pg) : 0;
    };
    int ids_cur = (warp == 0) ? load16(t_begin) : 0;

    // -------------------------------------------------------------- setup --
    const uint32_t crank = PAIR ? cluster_ctarank() : 0u;  // 0: the pair's leader (MMA issuer)
    const bool leader = crank == 0;
    // a barrier slot of the leader CTA as a shared::cluster address
    auto lead_bar = [&](int i) { return PAIR ? mapa_shared(bar(i), 0) : bar(i); };
    if (tid == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < NSK; ++s) {
            mbar_init(bar(B_KF + s), 1);
            mbar_init(bar(B_KE + s), 1);
        }
        for (int s = 0; s < NSV; ++s) {
            // the leader's V-full also takes the other CTA's arrival
            mbar_init(bar(B_VF + s), PAIR && leader ? 2 : 1);
            mbar_init(bar(B_VE + s), 1);
        }
        for (int i = 0; i < NSB; ++i) {
            mbar_init(bar(B_SF + i), 1);
            mbar_init(bar(B_PF + i), 8 * CL);  // softmax warps of every CTA of the pair
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_PV + i), 1);
            mbar_init(bar(B_CR + i), 8);
        }
        mbar_init(bar(B_OF), 4 * CL);
        if (OBUF2)
            mbar_init(bar(B_OF + 1), 4 * CL);
        mbar_init(bar(B_PROD), 1);
        mbar_init(bar(B_DONE), 1);
        mbar_init(bar(B_VZ), 1);
        sflags[0] = 0;
        sflags[3] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_addr(&sflags[1]), 512);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_addr(&sflags[1]), 512);
            tmem_relinquish();
        }
    }
    if (tid == 64) {
        prefetch_tensormap(&p.tm_q);
        prefetch_tensormap(&p.tm_k);
        prefetch_tensormap(&p.tm_v);
    }
    tc_fence_before();
    if (PAIR)
        cluster_sync_all();  // both CTAs' barriers and TMEM exist before either is used
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(sflags[1]);
    // The key tile is the last one and runs past kend: V rows of keys >= kend
    // are zeroed after they land (stale or poisoned data).
    auto zero_tile = [&](int t) { return (t + 1) * kKeys > kend; };

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        bool ok = true, any_bad = false;
        int last_k_use[NSK], last_v_use[NSV];
        for (int s = 0; s < NSK; ++s) last_k_use[s] = -1;
        for (int s = 0; s < NSV; ++s) last_v_use[s] = -1;
        // Q box: 64 columns x G heads x tq tokens per 64-column block; with a
        // pair both Q tiles are credited to the leader's barrier
        if (lane == 0 && leader)
            mbar_arrive_expect_tx(bar(B_Q), CL * NKB * 128 * p.group * p.tq);
        __syncwarp();
        if (lane < NKB) {
            if (PAIR)
                tma_load_3d_pair(smem_addr(sQ + lane * 16384), &p.tm_q, lead_bar(B_Q), lane * 64, kvh * p.group,
                                 (int)tok_first);
            else
                tma_load_3d(smem_addr(sQ + lane * 16384), &p.tm_q, bar(B_Q), lane * 64, kvh * p.group,
                            (int)tok_first);
        }
        if (p.early_reads)
            griddep_wait();  // the cache write has completed and is visible
        // ids of TPL consecutive tiles sit in lanes 0-15 of ids_cur; the next
        // group is requested one group ahead
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
            // K boxes: (page, 64-column block) per lane; a pair member takes the
            // pages of its half of the keys.  V boxes: all pages, its blocks.
            const int k_page = (int)crank * (PPT / CL) + lane / NKB, k_kb = lane % NKB;
            const int k_id = __shfl_sync(0xffffffffu, id, k_page % PPT);
            const bool k_issue = lane < (PPT / CL) * NKB && k_page < np;
            const int v_page = lane / VKB, v_kb = lane % VKB;
            const int v_id = __shfl_sync(0xffffffffu, id, v_page % PPT);
            const bool v_issue = lane < PPT * VKB && v_page < np;
            // K
            const int sk = it % NSK, uk = it / NSK;
            if (lane == 0) {
                if (uk >= 1)
                    ok = wb(B_KE + sk, (uk - 1) & 1);
                if (ok && leader)
                    mbar_arrive_expect_tx(bar(B_KF + sk), np * NKB * 2048);  // both halves of the tile
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            if (k_issue) {
                const uint32_t dst = smem_addr(sK + sk * KST + k_kb * KBLK + (k_page - (int)crank * (PPT / CL)) * 2048);
                if (PAIR)
                    tma_load_4d_pair(dst, &p.tm_k, lead_bar(B_KF + sk), k_kb * 64, kvh, 0, k_id);
                else
                    tma_load_4d(dst, &p.tm_k, bar(B_KF + sk), k_kb * 64, kvh, 0, k_id);
            }
            if (!PAIR || leader)
                last_k_use[sk] = uk;
            // V
            const int sv = it % NSV, uv = it / NSV;
            // with a pair, the other CTA's last, partly zeroed tile goes through
            // its own barrier first (relayed by its warp 1 after the zeroing)
            const bool v_local = PAIR && !leader && zero_tile(t);
            if (lane == 0) {
                if (uv >= 1)
                    ok = wb(B_VE + sv, (uv - 1) & 1);
                if (ok) {
                    if (!PAIR)
                        mbar_arrive_expect_tx(bar(B_VF + sv), np * NKB * 2048);
                    else if (leader)
                        mbar_arrive_expect_tx(bar(B_VF + sv), (zero_tile(t) ? 1 : 2) * np * VKB * 2048);
                    else if (v_local)
                        mbar_arrive_expect_tx(bar(B_VF + sv), np * VKB * 2048);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            if (v_issue) {
                const uint32_t dst = smem_addr(sV + sv * VST + v_kb * VBLK + v_page * 2048);
                const int col = ((int)crank * VKB + v_kb) * 64;
                if (PAIR)
                    tma_load_4d_pair(dst, &p.tm_v, v_local ? bar(B_VF + sv) : lead_bar(B_VF + sv), col, kvh, 0,
                                     v_id);
                else
                    tma_load_4d(dst, &p.tm_v, bar(B_VF + sv), col, kvh, 0, v_id);
            }
            if (PAIR && !leader && !v_local && lane == 0)
                mbar_arrive_cluster_relaxed(lead_bar(B_VF + sv));  // a count: the bytes are tracked by the copies
            if (!PAIR || leader || v_local)
                last_v_use[sv] = uv;
        }
        // The last tile's V rows of keys >= kend hold stale or poisoned data:
        // zero them once the tile has landed (the barrier is in that tile's
        // phase now: the producer starts no later phase), then release the
        // MMA issuer.  A pair's other CTA zeroes its half in its relay warp.
        if (ok && n_it > 0 && zero_tile(t_end - 1) && (!PAIR || leader)) {
            const int j = n_it - 1, sv = j % NSV, t = t_end - 1;
            const bool okz = __all_sync(0xffffffffu, wbc(B_VF + sv, (j / NSV) & 1));
            if (okz) {
                const int row0 = kend - t * kKeys;
                const int nz = (kKeys - row0) * VKB * 8;
                uint8_t *vs = sV + sv * VST;
                for (int idx = lane; idx < nz; idx += 32) {
                    const int row = row0 + idx / (VKB * 8);
                    const int rem = idx % (VKB * 8);
                    *reinterpret_cast<uint4 *>(vs + (rem / 8) * VBLK + row * 128 + (rem % 8) * 16) =
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
                // let issued copies land before the CTA's shared memory goes away
                for (int s = 0; s < NSK; ++s)
                    if (last_k_use[s] >= 0)
                        wait_bar_drain(bar(B_KF + s), last_k_use[s] & 1);
                for (int s = 0; s < NSV; ++s)
                    if (last_v_use[s] >= 0)
                        wait_bar_drain(bar(B_VF + s), PAIR && !leader ? 0 : (last_v_use[s] & 1));
                if (leader)
                    wait_bar_drain(bar(B_Q), 0);
            }
        }
        __syncwarp();
    } else if (warp == 1 && PAIR && !leader) {
        // ------------------------------------- pair member: V relay only --
        // Its last tile's V half landed on its own barrier; zero the rows of
        // keys >= kend, then hand the tile to the leader's V-full barrier.
        if (n_it > 0 && zero_tile(t_end - 1)) {
            const int j = n_it - 1, sv = j % NSV, t = t_end - 1;
            bool okz = __all_sync(0xffffffffu, wb(B_VF + sv, 0));
            if (okz) {
                const int row0 = kend - t * kKeys;
                const int nz = (kKeys - row0) * VKB * 8;
                uint8_t *vs = sV + sv * VST;
                for (int idx = lane; idx < nz; idx += 32) {
                    const int row = row0 + idx / (VKB * 8);
                    const int rem = idx % (VKB * 8);
                    *reinterpret_cast<uint4 *>(vs + (rem / 8) * VBLK + row * 128 + (rem % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster(lead_bar(B_VF + sv));
            }
        }
        // the leader's MMAs read this CTA's TMEM and shared memory until its
        // final commit
        if (lane == 0)
            wait_bar_drain(bar(B_DONE), 0);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer --
        // With two or more V stages, PV(j) and QK(j+NSB) are issued back to
        // back (PV(j) first, then the wait for K(j+NSB)), so the tensor pipe
        // goes from one group to the next and Q.K^T runs NSB tiles ahead of
        // P.V.  QK(j+NSB) overwrites the S buffer that PV(j) reads P from:
        // tcgen05 MMAs from one thread run in order.  With one V stage, K(j+2)
        // is loaded only after PV(j) has released V, so the order is QK(j+1),
        // PV(j).
        constexpr bool LOOKAHEAD = NSV >= 2;
        bool ok = true;
        if (lane == 0)
            ok = wb(B_Q, 0);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        // QK(it), K(it) already resident: Q and K advance 32 bytes per
        // 16-column step inside a 64-column block, a block after four steps
        auto issue_qk = [&](int it) {
            const int sk = it % NSK;
            const uint64_t qd0 = sdesc_sw128(smem_addr(sQ), 16, 1024);
            const uint64_t kd0 = sdesc_sw128(smem_addr(sK + sk * KST), 16, 1024);
            tc_fence_after();
#pragma unroll
            for (int g8 = 0; g8 < DH / 128; ++g8) {
                uint64_t ad[8], bd[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int kk = g8 * 8 + i;
                    ad[i] = qd0 + (uint64_t)(((kk / 4) * 16384 + (kk % 4) * 32) >> 4);
                    bd[i] = kd0 + (uint64_t)(((kk / 4) * KBLK + (kk % 4) * 32) >> 4);
                }
                mma8_ss<CL>(tmem + (uint32_t)(it % NSB) * kKeys, ad, bd, ID_QK, g8 > 0 ? 1u : 0u);
            }
            if (PAIR) {
                mma_commit_pair_mc(bar(B_KE + sk), 0x3);
                mma_commit_pair_mc(bar(B_SF + (it % NSB)), 0x3);
            } else {
                mma_commit(bar(B_KE + sk));
                mma_commit(bar(B_SF + (it % NSB)));
            }
        };
        auto wait_kf = [&](int it) { return wb(B_KF + it % NSK, (it / NSK) & 1); };
        // PV(j) and, when given (qk_next >= 0), QK(qk_next) right behind it.
        // Lane 0 alone: no warp-wide step between MMA groups.
        auto issue_pv = [&](int j, int qk_next) -> bool {
            const int sv = j % NSV;
            const int t = t_begin + j;
            // operands first: P of the first half of the keys sits in the first
            // HALF/2 columns of the S buffer, the second half from column HALF
            // (each softmax half writes its own); V: 16 keys (2 KB) per step
            const uint32_t pcol = tmem + (uint32_t)(j % NSB) * kKeys;
            const uint64_t vd0 = sdesc_sw128(smem_addr(sV + sv * VST), VBLK, 1024);
            uint32_t ad[NPV];
            uint64_t bd[NPV];
#pragma unroll
            for (int i = 0; i < NPV; ++i) {
                ad[i] = pcol + (uint32_t)((i / (NPV / 2)) * HALF + (i % (NPV / 2)) * 8);
                bd[i] = vd0 + (uint64_t)((i * 2048) >> 4);
            }
            const bool chunk_first = CHUNKED ? ((t * kKeys) % CHUNK_DIV == 0) : (j == 0);
            const int k = CHUNKED ? (t * kKeys - kbeg) / CHUNK_DIV : 0;
            // The last tile's V rows of keys >= kend are zeroed by the producer
            // first (generic writes, possibly relayed from the pair's other
            // CTA: acquire at cluster scope).  V-full (copies and a relaxed
            // count), P-ready and fold-done hand over tensor memory or TMA
            // data only: CTA-scope waits suffice.
            bool okj = zero_tile(t) ? wbc(B_VZ, 0) : wb(B_VF + sv, (j / NSV) & 1);
            if (okj)
                okj = wb(B_PF + (j % NSB), (j / NSB) & 1);
            if (OBUF2) {
                // the buffer was last read by the fold of chunk k - 2
                if (okj && chunk_first && k >= 2)
                    okj = wb(B_OF + (k & 1), ((k >> 1) - 1) & 1);
            } else if (okj && chunk_first && k > 0) {
                okj = wb(B_OF, (k - 1) & 1);
            }
            if (okj) {
                tc_fence_after();
                if constexpr (NPV == 8)
                    mma8_ts<CL>(tmem + ocol(k), ad, bd, ID_PV, chunk_first ? 0u : 1u);
                else
                    mma4_ts<CL>(tmem + ocol(k), ad, bd, ID_PV, chunk_first ? 0u : 1u);
                if (PAIR) {
                    mma_commit_pair_mc(bar(B_VE + sv), 0x3);
                    mma_commit_pair_mc(bar(B_PV + (j & 1)), 0x3);
                } else {
                    mma_commit(bar(B_VE + sv));
                    mma_commit(bar(B_PV + (j & 1)));
                }
                // K(qk_next) may still be in flight: PV(j) does not wait for it
                if (qk_next >= 0) {
                    okj = wait_kf(qk_next);
                    if (okj)
                        issue_qk(qk_next);
                }
            }
            return okj;
        };
        if (lane == 0) {
            if (LOOKAHEAD) {
                for (int it = 0; ok && it < min(NSB, n_it); ++it) {
                    ok = wait_kf(it);
                    if (ok)
                        issue_qk(it);
                }
                for (int j = 0; ok && j < n_it; ++j)
                    ok = issue_pv(j, j + NSB < n_it ? j + NSB : -1);
            } else {
                for (int it = 0; ok && it <= n_it; ++it) {
                    if (it < n_it) {
                        ok = wait_kf(it);
                        if (ok)
                            issue_qk(it);
                    }
                    if (ok && it >= 1)
                        ok = issue_pv(it - 1, -1);
                }
            }
        }
        __syncwarp();
        // all MMAs retired before TMEM is released (in both CTAs of a pair)
        if (lane == 0) {
            if (PAIR)
                mma_commit_pair_mc(bar(B_DONE), 0x3);
            else
                mma_commit(bar(B_DONE));
            wait_bar_drain(bar(B_DONE), 0);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12) {
        // --------------------------------------------- softmax (2 halves) --
        const int h = (warp - 4) / 4;       // column half
        const int q4 = warp % 4;            // TMEM lane quadrant
        const int r = q4 * 32 + lane;       // row
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const bool row_valid = r < rows_valid;
        const bool warp_active = 32 * q4 < rows_valid;
        const int pos = L - qn + tok0 + r / p.group;
        float *xmax = s_x;                  // [2][128]
        float *xsum = s_x + 2 * kRows;      // [2][128]
        float m = -INFINITY, l = 0.f;
        bool failed = false;  // a wait gave up: leave the loop together with the other half
        for (int it = 0; it < n_it; ++it) {
            const int t = t_begin + it;
            const int sb = it % NSB;
            bool okw = !failed && wb(B_SF + sb, (it / NSB) & 1);
            okw = __all_sync(0xffffffffu, okw);
            tc_fence_after();
            const int nallow = row_valid ? max(0, min(HALF, pos - t * kKeys - HALF * h + 1)) : 0;
            const uint32_t scol = tmem + lane_off + sb * kKeys + HALF * h;  // this half's S columns
            // pass 1: max of the raw scores over allowed keys of this half
            // (scale > 0, so this is the max of the scaled scores as well)
            const bool unmasked = __all_sync(0xffffffffu, nallow == HALF);
            float pmax = -INFINITY;
            uint32_t v1[32];  // columns 32-63 of the half stay in registers for pass 2
            if (warp_active && okw) {
                uint32_t v0[32];
                tmem_ld32(scol, v0);
                if (HALF == 64)
                    tmem_ld32(scol + 32, v1);
                tmem_wait_ld();
                if (unmasked) {
                    // two independent chains of three-input max (max is exact:
                    // the grouping does not change the result)
                    float pm0 = -INFINITY, pm1 = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        if (HALF == 64) {
                            pm0 = max3f(pm0, __uint_as_float(v0[i]), __uint_as_float(v1[i]));
                            pm1 = max3f(pm1, __uint_as_float(v0[i + 1]), __uint_as_float(v1[i + 1]));
                        } else {
                            pm0 = max3f(pm0, __uint_as_float(v0[i]), __uint_as_float(v0[i + 1]));
                        }
                    }
                    pmax = fmaxf(pm0, pm1);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        pmax = (i < nallow) ? fmaxf(pmax, __uint_as_float(v0[i])) : pmax;
                        if (HALF == 64)
                            pmax = (32 + i < nallow) ? fmaxf(pmax, __uint_as_float(v1[i])) : pmax;
                    }
                }
            }
            xmax[h * kRows + r] = pmax;
            if (named_sync_or(1, 256, !okw)) {
                failed = true;
                break;
            }
            // C2: the tile max in log2 units, one fp32 multiply
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
            // pass 2: p = exp2(fma(S, scale*log2e, -m)), the half's fixed-order
            // sum, P as BF16
            float hs = 0.f;
            if (warp_active) {
                // columns c and c+1 go through the paired fp32 instructions:
                // each lane is the scalar fma.rn / add.rn of the same operands
                const uint64_t c2x2 = pack_f32x2(p.scale_log2, p.scale_log2);
                const uint64_t nmx2 = pack_f32x2(-m_new, -m_new);
                uint64_t a2[4];  // accumulator k sums columns k, k+8, ..., k+HALF-8 (pairs k, k+1)
                uint32_t w[HALF / 2];
#pragma unroll
                for (int g2 = 0; g2 < HALF / 32; ++g2) {
                    uint32_t v[32];
                    if (g2 == 0) {
                        tmem_ld32(scol, v);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] = v1[i];
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const int c = g2 * 32 + i;
                        float x0, x1;
                        unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                               c2x2, nmx2),
                                     x0, x1);
                        float e0 = ex2(x0);
                        float e1 = ex2(x1);
                        if (!unmasked) {
                            e0 = (c < nallow) ? e0 : 0.f;
                            e1 = (c + 1 < nallow) ? e1 : 0.f;
                        }
                        const uint64_t e2 = pack_f32x2(e0, e1);
                        a2[(c & 7) / 2] = (c < 8) ? e2 : add_f32x2(a2[(c & 7) / 2], e2);
                        w[c / 2] = pack_bf16x2(e0, e1);
                    }
                }
                float a[8];
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2)
                    unpack_f32x2(a2[k2], a[2 * k2], a[2 * k2 + 1]);
                hs = __fadd_rn(__fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3])),
                               __fadd_rn(__fadd_rn(a[4], a[5]), __fadd_rn(a[6], a[7])));
                // P (BF16, two keys per column) overwrites this half's first
                // HALF/2 S columns, after the S loads above completed
                if constexpr (HALF == 64)
                    tmem_st32(scol, w);
                else
                    tmem_st16(scol, w);
            }
            xsum[h * kRows + r] = hs;
            named_sync(1, 256);
            const float tsum = __fadd_rn(xsum[r], xsum[kRows + r]);
            bool okr = true;
            if (__any_sync(0xffffffffu, need)) {
                // O of this chunk must hold PV(it - 1) before it is rescaled
                okr = __all_sync(0xffffffffu, wb(B_PV + ((it - 1) & 1), ((it - 1) >> 1) & 1));
                failed = !okr;
            }
            if (__any_sync(0xffffffffu, need) && okr) {
                tc_fence_after();
                const float f = need ? corr : 1.f;
#pragma unroll 1
                for (int g = 0; g < DH / 64; ++g) {
                    uint32_t v[32];
                    const uint32_t col = tmem + lane_off + ocol(CHUNKED ? it / TPC : 0) + (DH / 2) * h + g * 32;
                    tmem_ld32(col, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__fmul_rn(__uint_as_float(v[i]), f));
                    tmem_st32(col, v);
                }
            }
            tmem_wait_st();
            l = need ? __fadd_rn(__fmul_rn(l, corr), tsum) : __fadd_rn(l, tsum);
            m = m_new;
            const bool chunk_end = (it == n_it - 1) || (CHUNKED && ((t + 1) * kKeys) % CHUNK_DIV == 0);
            const int k = CHUNKED ? it / TPC : 0;
            if (chunk_end && h == 0) {
                s_ml[((k & 1) * kRows + r) * 2] = m;
                s_ml[((k & 1) * kRows + r) * 2 + 1] = l;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // P (and any O rescale) is in this CTA's tensor memory: ordered by
                // tcgen05.wait::st and the fence above, so a relaxed arrival will do
                if (PAIR)
                    mbar_arrive_cluster_relaxed(lead_bar(B_PF + sb));
                else
                    mbar_arrive(bar(B_PF + sb));
                if (chunk_end)
                    mbar_arrive(bar(B_CR + (k & 1)));
            }
            if (chunk_end) {
                m = -INFINITY;
                l = 0.f;
            }
        }
    } else if (warp >= 12) {
        // ----------------------------------------------------- correction --
        const int q4 = warp % 4;
        const int r = q4 * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const bool row_valid = r < rows_valid;
        const int G = p.group;
        const int64_t tok = tok_first + r / G;
        const int head = kvh * G + r % G;
        float m_acc = -INFINITY, l_acc = 0.f;
        int nfold = 0;  // chunks folded into the accumulator so far (CTA-uniform)
        bool ok = true;
        for (int k = 0; ok && k < nck; ++k) {
            const int it_last = CHUNKED ? min((k + 1) * TPC, n_it) - 1 : n_it - 1;
            const bool final_chunk = (k == nck - 1);
            ok = wb(B_CR + (k & 1), (k >> 1) & 1);
            if (ok)
                ok = wb(B_PV + (it_last & 1), (it_last >> 1) & 1);
            if (ok && final_chunk)
                ok = wb(B_PROD, 0);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const float m = s_ml[((k & 1) * kRows + r) * 2];
            const float l = s_ml[((k & 1) * kRows + r) * 2 + 1];
            const bool bad = final_chunk && sflags[3] != 0;
            if (p.split) {
                // partial state of chunk c_grid*cpu + k: m, l and the O row
                float *part = p.ws_part + (unit_q * p.nch + (int64_t)c_grid * p.cpu + k) * rec_floats;
                const float qnan = __int_as_float(0x7FC00000);
                if (row_valid) {
                    part[r] = bad ? 0.f : m;
                    part[p.ws_rows + r] = bad ? qnan : l;
                }
                float4 *orow = reinterpret_cast<float4 *>(part + rec_hdr + (int64_t)r * DH);
#pragma unroll 1
                for (int g = 0; g < DH / 32; ++g) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + C::kOCol + g * 32, v);
                    tmem_wait_ld();
                    if (row_valid) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            __stcg(orow + g * 8 + i,
                                   bad ? make_float4(qnan, qnan, qnan, qnan)
                                       : make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
                    }
                }
                // ordered before the arrival's release by the CTA barrier ahead of it
            } else if (final_chunk) {
                // epilogue: out = fold(acc, chunk) / l
                const Fold f = fold_coef(m_acc, l_acc, m, l);
                const float inv = __frcp_rn(f.l);
                const bool acc_live = nfold > 0;  // uniform: tcgen05.ld is warp-collective
#pragma unroll 1
                for (int g = 0; g < DH / 32; ++g) {
                    uint32_t vc[32], va[32];
                    tmem_ld32(tmem + lane_off + ocol(k) + g * 32, vc);
                    if (acc_live && !ACC_SMEM)
                        tmem_ld32(tmem + lane_off + ACC_COL + g * 32, va);
                    if (acc_live && ACC_SMEM)
                        acc_row_load<DH>(sAcc, r, g, va);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float oa = acc_live ? __uint_as_float(va[i]) : 0.f;
                        vc[i] = bad ? 0x7FC00000u
                                    : __float_as_uint(__fmul_rn(fold_elem(oa, __uint_as_float(vc[i]), f), inv));
                    }
                    if (row_valid)
                        store_out32(p.out + (tok * p.hq + head) * DH + g * 32, vc);
                }
                if (row_valid && p.lse)
                    p.lse[tok * p.hq + head] = bad ? __int_as_float(0x7FC00000) : lse_of(f.m, f.l);
            } else {
                // fold this chunk into the running accumulator (TMEM, or shared
                // memory when the chunk accumulators are double-buffered)
                const Fold f = fold_coef(m_acc, l_acc, m, l);
                const bool acc_live = nfold > 0;  // uniform: tcgen05.ld is warp-collective
#pragma unroll 1
                for (int g = 0; g < DH / 32; ++g) {
                    uint32_t vc[32], va[32];
                    tmem_ld32(tmem + lane_off + ocol(k) + g * 32, vc);
                    if (acc_live && !ACC_SMEM)
                        tmem_ld32(tmem + lane_off + ACC_COL + g * 32, va);
                    if (acc_live && ACC_SMEM)
                        acc_row_load<DH>(sAcc, r, g, va);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float oa = acc_live ? __uint_as_float(va[i]) : 0.f;
                        va[i] = __float_as_uint(fold_elem(oa, __uint_as_float(vc[i]), f));
                    }
                    if (ACC_SMEM)
                        acc_row_store<DH>(sAcc, r, g, va);
                    else
                        tmem_st32(tmem + lane_off + ACC_COL + g * 32, va);
                }
                if (!ACC_SMEM)
                    tmem_wait_st();
                m_acc = f.m;
                l_acc = f.l;
                ++nfold;
            }
            tc_fence_before();
            __syncwarp();
            if (!final_chunk && lane == 0) {
                // chunk k's accumulator may be overwritten (tensor-memory reads only)
                const int of = B_OF + (OBUF2 ? (k & 1) : 0);
                if (PAIR)
                    mbar_arrive_cluster_relaxed(lead_bar(of));
                else
                    mbar_arrive(bar(of));
            }
        }
    }

    tc_fence_before();
    if (PAIR)
        cluster_sync_all();  // both CTAs are done with TMEM, barriers and shared memory
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem, 512);
        else
            tmem_dealloc(tmem, 512);
    }  // no CTA leaves while its partner may still write into it
    if (p.split)
        split_arrive_and_merge<DH>(p, unit_q, nchunks, (nchunks + p.cpu - 1) / p.cpu, rows_valid, tok_first,
                                   kvh, merge_work, kMergeWorkFloats, &sflags[2], split_multi);
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
    pl.kt = head_dim == 512 ? 64 : 128;  // the head dim's default tile
    pl.group = G;
    pl.tokens_per_tile = kRows / G;
    pl.qtiles = max_query_len > 0 ? (max_query_len + pl.tokens_per_tile - 1) / pl.tokens_per_tile : 0;
    const int chunk = head_dim == 128 ? Cfg<128>::kChunk : 0;
    const long long full_ctas = (long long)num_seqs * num_kv_heads * pl.qtiles;
    pl.split = chunk > 0 && max_seq_len > chunk && full_ctas < kSplitCtaThreshold;
    pl.nch = pl.split ? (max_seq_len + chunk - 1) / chunk : 1;
    // Split-KV: about four waves of CTAs at most.  Larger batches give each CTA
    // several consecutive chunks (still one record per chunk, so the fold and
    // the results are the same whatever cpu is).
    pl.cpu = 1;
    if (pl.split) {
        const long long target = 4LL * kSplitCtaThreshold;
        const long long units = full_ctas * pl.nch;
        if (units > target)
            pl.cpu = (int)((units + target - 1) / target);
    }
    pl.ws_rows = G * (max_query_len < pl.tokens_per_tile ? max_query_len : pl.tokens_per_tile);
    pl.ws_counter_bytes = 0;
    pl.ws_bytes = 0;
    if (pl.split) {
        const size_t units_q = (size_t)full_ctas;
        pl.ws_counter_bytes = ((units_q * 4 + 255) / 256) * 256;
        pl.ws_bytes = pl.ws_counter_bytes + units_q * pl.nch * (size_t)part_record_floats(pl.ws_rows, head_dim) * 4;
    }
    // in-CTA schedule with several query tiles: CTA pairs share every MMA
    // (head dims 128/256)
    pl.cl = (!pl.split && head_dim != 512 && pl.qtiles >= 2) ? 2 : 1;
    const long long qgroups = pl.cl == 2 ? (pl.qtiles + 1) / 2 * 2 : pl.qtiles;
    pl.grid = (long long)num_seqs * num_kv_heads * qgroups * ((pl.nch + pl.cpu - 1) / pl.cpu) *
              (head_dim == 512 ? 2 : 1);
    *plan = pl;
    return true;
}

// Head dim 128 decode with the MMA operands swapped (pa_decode.cu).
cudaError_t init_decode_attributes();
int decode_rows(const AttnPlan &pl, int32_t max_query_len, int32_t num_seqs);
long long decode_grid(const AttnPlan &pl, int32_t num_seqs, int32_t num_kv_heads, int num_sms);
cudaError_t launch_decode(const AttnArgs &a, const AttnPlan &pl, AttnParams &p, int rows, cudaStream_t stream);

template <int DH, bool PAIR, int KT = 128>
static cudaError_t set_smem_attribute()
{
    return cudaFuncSetAttribute(attn_kernel<DH, PAIR, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<DH, PAIR, KT>());
}

cudaError_t init_attention_attributes()
{
    cudaError_t e;
    if ((e = set_smem_attribute<128, false>()) != cudaSuccess || (e = set_smem_attribute<128, true>()) != cudaSuccess ||
        (e = set_smem_attribute<128, false, 64>()) != cudaSuccess ||
        (e = set_smem_attribute<128, true, 64>()) != cudaSuccess ||
        (e = set_smem_attribute<256, false>()) != cudaSuccess || (e = set_smem_attribute<256, true>()) != cudaSuccess ||
        (e = init_decode_attributes()) != cudaSuccess)
        return e;
    return init_attention512_attributes();
}

// Limit of the split-KV fold's cross-CTA wait, read at each launch (a
// captured graph keeps the value it was captured with).
static std::atomic<uint64_t> g_fold_wait_ns{kWaitLimitNs};

uint64_t fold_wait_limit_ns() { return g_fold_wait_ns.load(std::memory_order_relaxed); }

uint64_t set_fold_wait_limit_ns(uint64_t ns) { return g_fold_wait_ns.exchange(ns, std::memory_order_relaxed); }

// SM count of the current device, looked up once per device.
static int num_sms_of_current_device()
{
    static int cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;  // 0: the fold is never shared
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cache[dev] = n;
    }
    return cache[dev];
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
    p.npairs = (pl.qtiles + 1) / 2;
    p.num_sms = num_sms_of_current_device();
    p.cpu = pl.cpu;
    p.early_reads = a.early_reads ? 1 : 0;
    p.fold_wait_ns = fold_wait_limit_ns();
    // C2: scale * log2(e) formed once, in fp32, on the host
    p.scale_log2 = a.scale * 1.4426950408889634f;
    if constexpr (DH == 128) {
        // few query rows per CTA: the decode kernel with swapped operands
        if (const int nr = decode_rows(pl, a.max_query_len, a.num_seqs))
            return launch_decode(a, pl, p, nr, stream);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(kThreads);
    const bool kt64 = DH == 128 && pl.kt == 64;
    cfg.dynamicSmemBytes = kt64 ? (pl.cl == 2 ? smem_bytes<DH, true, 64>() : smem_bytes<DH, false, 64>())
                                : (pl.cl == 2 ? smem_bytes<DH, true, 128>() : smem_bytes<DH, false, 128>());
    cfg.stream = stream;
    // the kernel may be scheduled while the preceding kernel (typically the
    // cache write) still runs; it waits for it before its first global read
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)pl.cl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pl.cl == 2 ? 2 : 1;
    if constexpr (DH == 128) {
        if (kt64)
            return pl.cl == 2 ? cudaLaunchKernelEx(&cfg, attn_kernel<DH, true, 64>, p)
                              : cudaLaunchKernelEx(&cfg, attn_kernel<DH, false, 64>, p);
    }
    if (pl.cl == 2)
        return cudaLaunchKernelEx(&cfg, attn_kernel<DH, true, 128>, p);
    return cudaLaunchKernelEx(&cfg, attn_kernel<DH, false, 128>, p);
}

cudaError_t launch_attention(const AttnArgs &a, const AttnPlan &pl, ErrState *err, cudaStream_t stream,
                             char *info, size_t info_len)
{
    const int nr = decode_rows(pl, a.max_query_len, a.num_seqs);
    // the decode kernel deals the split-KV chunks out as one wave of ranges
    const long long grid =
        nr ? decode_grid(pl, a.num_seqs, a.num_kv_heads, num_sms_of_current_device()) : pl.grid;
    if (info && info_len)
        snprintf(info, info_len,
                 "attention dh=%d schedule=%s grid=%lld qtiles=%d chunks=%d kv_tile=%d chunk=%d cpu=%d kernel=%s",
                 pl.head_dim,
                 pl.split ? "split-kv" : (pl.head_dim == 512 ? "in-cta-pair" : (pl.cl == 2 ? "in-cta-pair2sm" : "in-cta")),
                 grid, pl.qtiles, pl.nch, pl.kt, pl.head_dim == 128 ? Cfg<128>::kChunk : 0, nr ? 0 : pl.cpu,
                 nr ? "decode-swapped-r" : "rows-m128");
    if (nr && info && info_len) {
        const size_t used = strlen(info);
        snprintf(info + used, info_len - used, "%d", nr);
    }
    if (pl.grid == 0)
        return cudaSuccess;
    switch (a.head_dim) {
    case 128: return launch_dh<128>(a, pl, err, stream);
    case 256: return launch_dh<256>(a, pl, err, stream);
    case 512: return launch_attention512(a, pl, err, stream);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace pa

// Device-side pieces shared by the attention kernels (head dims 128/256 in
// pa_attn.cu, 512 in pa_attn512.cu): kernel parameters, the fixed softmax
// fold, bounded barrier waits, request metadata checks and NaN rows for
// invalid requests.
#pragma once
#include <cuda_bf16.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kRows = 128;          // M of every MMA: rows per tile
constexpr float kTau = 8.0f;        // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
// Dynamic shared memory one CTA may opt into on sm_103a (227 KB); every
// kernel's layout is checked against it at compile time.
constexpr size_t kMaxSmemPerBlock = 227 * 1024;
struct AttnParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    const void *q;              // used by the head-dim 512 kernel (loads Q itself)
    int64_t q_tok_stride;
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
    int32_t npairs;  // query-tile pairs (in-CTA schedule on CTA pairs)
    int32_t early_reads;  // only the K/V copies wait for the preceding grid
    int32_t num_sms;      // SMs of the device (split-KV: whether every unit is resident)
    int32_t cpu;          // split-KV: consecutive chunks per CTA (each still writes one record per chunk)
    uint64_t fold_wait_ns;  // limit of the split-KV fold's cross-CTA wait (0: give up at once)
    float scale_log2;
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Paired fp32 arithmetic (two lanes per instruction, each lane rounded
// exactly as the scalar .rn instruction) and three-input max: the softmax's
// instruction count, not the exp2 unit, bounds its throughput.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack_f32x2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// {a0*b0 + c0, a1*b1 + c1}, each a single-rounding fma.rn
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// {a0 + b0, a1 + b1}, each add.rn
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
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

// fold_elem with the mode picked by predicated selects (no branch): the
// same three candidate results, the same one chosen, bit for bit.
__device__ __forceinline__ float fold_elem_sel(float oa, float oc, float sa, float sc, int mode)
{
    float r;
    asm("{\n\t.reg .pred p1, p2;\n\t.reg .f32 t1, t2, t3, t4;\n\t"
        "mul.rn.f32 t1, %1, %3;\n\t"
        "mul.rn.f32 t2, %2, %4;\n\t"
        "add.rn.f32 t3, t1, t2;\n\t"
        "setp.eq.s32 p1, %5, 1;\n\t"
        "selp.f32 t4, %2, %1, p1;\n\t"
        "setp.eq.s32 p2, %5, 2;\n\t"
        "selp.f32 %0, t3, t4, p2;\n\t}"
        : "=f"(r)
        : "f"(oa), "f"(oc), "f"(sa), "f"(sc), "r"(mode));
    return r;
}

__device__ __forceinline__ float lse_of(float m, float l)
{
    return __fmul_rn(__fadd_rn(m, __log2f(l)), kLn2);
}

// Bounded mbarrier wait (inline: no call, so no register spills around it).
// Gives up when another thread of the CTA already gave up (abort flag) or
// after kWaitLimitNs, latching PA_ERR_TIMEOUT.
// The first timeout records (block index << 8) | barrier slot as its index.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         ErrState *err, int where)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            record_error(err, kErrTimeout, ((long long)blockIdx.x << 8) | where);
            return false;
        }
    }
    return true;
}

// wait_bar with acquire at cluster scope: the phase may be completed by an
// arrival from the other CTA of a cluster.
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                 ErrState *err, int where)
{
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            record_error(err, kErrTimeout, ((long long)blockIdx.x << 8) | where);
            return false;
        }
    }
    return true;
}

// Wait without the abort shortcut (drains in-flight work on exit).
__device__ __forceinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity)
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

// Named barrier that also ORs a predicate over the participating threads, so
// every participant takes the same branch afterwards.
__device__ __forceinline__ bool named_sync_or(int id, int nthreads, bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 q, %1, 0;\n\t"
                 "bar.red.or.pred p, %2, %3, q;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v), "r"(id), "r"(nthreads)
                 : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Store 32 consecutive output values (fp32 bit patterns, already
// normalised) as BF16.
__device__ __forceinline__ void store_out32(__nv_bfloat16 *dst, const uint32_t (&v)[32])
{
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float *f = reinterpret_cast<const float *>(v) + 8 * i;
        d[i] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                          pack_bf16x2(f[6], f[7]));
    }
}

template <int DH>
__device__ void write_nan_rows(const AttnParams &p, int64_t tok_first, int ntok, int kvh)
{
    const __nv_bfloat16 qnan = __ushort_as_bfloat16(0x7FC0);
    const int G = p.group;
    const int64_t total = (int64_t)ntok * G * DH;
    for (int64_t e = threadIdx.x; e < total; e += blockDim.x) {
        const int64_t row = e / DH;
        const int d = (int)(e % DH);
        const int64_t t = tok_first + row / G;
        const int h = kvh * G + (int)(row % G);
        p.out[(t * p.hq + h) * DH + d] = qnan;
        if (d == 0 && p.lse)
            p.lse[t * p.hq + h] = __int_as_float(0x7FC00000);
    }
}

// Request metadata as every CTA reads it.
struct ReqMeta {
    int qs, qn, L;
    bool sane;  // the query-token range is usable (rows can be written)
    bool ok;    // lengths are consistent with each other and with the bounds
};

__device__ __forceinline__ ReqMeta read_meta(const AttnParams &p, int b)
{
    ReqMeta m;
    const int qs = __ldg(p.qsl + b), qe = __ldg(p.qsl + b + 1), L = __ldg(p.seq_lens + b);
    m.qs = qs;
    m.qn = qe - qs;
    m.L = L;
    m.sane = qs >= 0 && m.qn >= 0 && (int64_t)qe <= p.num_q_tokens;
    m.ok = m.sane && L >= m.qn && (int64_t)L <= (int64_t)p.max_blocks * 16 && m.qn <= p.max_query_len &&
           L <= p.max_seq_len;
    return m;
}


}  // namespace pa

"""Decode with few query rows per (request, KV head): the head-dim-128 kernel
that swaps the MMA operands (keys on the tensor-memory lanes) for query
tiles of up to 32 rows, in every row-count variant (4, 8, 16, 32 rows), on
the split-KV and the single-CTA schedules.

Each case is checked against the fp64 oracle (max-abs 2e-2, lse relative
1e-3) and bit for bit against the same rows computed by a full causal
prefill of the request, which runs the 128-row kernel ("fix(rocm): stabilize
direct paged CK attention for bitwise R/R", Validation: prefill and decode
agree bitwise; Changes: one query per decode row)."""
import pytest
import torch

from paged_kv_cache_178_gb300 import pagedattn
from paged_kv_cache_178_gb300 import workloads as wl
from paged_kv_cache_178_gb300.device import DeviceWorkload
from tests.helpers import LSE_RTOL, OUT_ATOL, lse_rel_err, oracle_attention

pytestmark = pytest.mark.gpu


def _bitwise(a, b, what):
    ai = a.contiguous().view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32)
    bi = b.contiguous().view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)
    mism = int((ai != bi).sum())
    print(f"{what}: mismatch_count={mism}")
    assert mism == 0


def _suffix_batch(hq, hkv, lens, qlens, seed):
    gen = torch.Generator().manual_seed(seed)
    nb = sum(wl.pages_needed(L) for L in lens) + 16
    pages = torch.randperm(nb, generator=gen).tolist()
    rows, at = [], 0
    for L in lens:
        n = wl.pages_needed(L)
        rows.append(pages[at:at + n])
        at += n
    return wl.build(f"suffix_hq{hq}_hkv{hkv}_q{max(qlens)}", num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                    seq_lens=lens, query_lens=qlens, num_blocks=nb, block_rows=rows, layout="interleaved",
                    seed=seed)


@pytest.mark.parametrize("hq,hkv,qlens,expect_rows", [
    (8, 2, [1, 1, 1, 1], 4),          # decode, G = 4
    (8, 2, [2, 1, 2, 1], 8),          # two-token speculative steps
    (8, 2, [4, 3, 1, 2], 16),
    (8, 2, [8, 5, 1, 7], 32),
    (16, 2, [1, 2, 3, 4], 32),        # G = 8
    (2, 2, [3, 1, 4, 2], 4),          # G = 1
    (32, 2, [1, 1, 1, 1], 16),        # G = 16
])
def test_few_row_decode_matches_oracle_and_prefill(hq, hkv, qlens, expect_rows):
    lens = [4171, 513, 300, 1000]
    w = _suffix_batch(hq, hkv, lens, qlens, seed=90 + hq + sum(qlens))
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    info = pagedattn.last_launch_info()
    print(info)
    assert f"decode-swapped-r{expect_rows}" in info and "split" in info
    ref_o, ref_l = oracle_attention(w)
    err_o = float((out.float().cpu().double() - torch.from_numpy(ref_o)).abs().max())
    err_l = lse_rel_err(lse.cpu().numpy(), ref_l)
    print(f"oracle: out max_abs_diff={err_o:.3e} lse rel={err_l:.3e}")
    assert err_o <= OUT_ATOL and err_l <= LSE_RTOL
    # each request's rows against a full prefill of that request (the
    # 128-row kernel), bit for bit
    for b in range(len(lens)):
        L, qn = lens[b], qlens[b]
        kv0 = sum(lens[:b])
        q0 = int(w.query_start_loc[b])
        wp = wl.build("prefill_view", num_q_heads=hq, num_kv_heads=hkv, head_dim=128, seq_lens=[L],
                      query_lens=[L], num_blocks=w.num_blocks, block_rows=[w.block_table[b].tolist()],
                      layout=w.layout, seed=1)
        # the prefill view reads the decode workload's cache: its q rows are
        # replaced by the decode q where the decode has them
        qp = torch.zeros((L, hq, 128), dtype=torch.bfloat16)
        qp[L - qn:] = w.q[q0:q0 + qn]
        dp = DeviceWorkload(wp, fill_bits=None, with_workspace=False)
        dp.share_cache_with(dw)
        dp.q = qp.cuda()
        dp.max_query_len = L
        dp.max_seq_len = L
        op, lp = dp.attention()
        assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
        assert "decode-swapped" not in pagedattn.last_launch_info()
        _bitwise(out[q0:q0 + qn], op[L - qn:], f"request {b} (q={qn}) decode vs prefill")
        _bitwise(lse[q0:q0 + qn], lp[L - qn:], f"request {b} lse")


def test_single_cta_schedule_equals_split():
    """Enough requests that every (request, KV head) gets one CTA that folds
    its chunks itself (no split-KV records); each request alone runs the
    split schedule.  Both give the same bits."""
    lens = [1000 + 37 * i for i in range(80)]
    w = wl.decode(seq_lens=lens, num_blocks=sum(wl.pages_needed(L) for L in lens) + 8)
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    info = pagedattn.last_launch_info()
    assert "decode-swapped-r4" in info and "split" not in info, info
    dev = out.device
    for b in (0, 17, 79):
        o1, l1 = dw.attention(q=dw.q[b:b + 1], block_tables=dw.block_tables[b:b + 1].contiguous(),
                              seq_lens=dw.seq_lens[b:b + 1].contiguous(),
                              query_start_loc=torch.tensor([0, 1], dtype=torch.int32, device=dev),
                              max_seq_len=int(w.seq_lens[b]))
        assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
        assert "split" in pagedattn.last_launch_info()
        _bitwise(out[b:b + 1], o1, f"request {b}: single-CTA fold vs split-KV merge")
        _bitwise(lse[b:b + 1], l1, f"request {b} lse")
    ref_o, ref_l = oracle_attention(w, rows=[0, 17, 79])
    o = out.float().cpu().double()[[0, 17, 79]]
    assert float((o - torch.from_numpy(ref_o)).abs().max()) <= OUT_ATOL
    assert lse_rel_err(lse.cpu().numpy()[[0, 17, 79]], ref_l) <= LSE_RTOL


def _alone(dw, w, b):
    """Request b of the batch launched on its own (its q row(s), table row,
    length), sharing the batch's cache."""
    dev = dw.q.device
    q0, q1 = int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])
    o, l = dw.attention(q=dw.q[q0:q1].contiguous(), block_tables=dw.block_tables[b:b + 1].contiguous(),
                        seq_lens=dw.seq_lens[b:b + 1].contiguous(),
                        query_start_loc=torch.tensor([0, q1 - q0], dtype=torch.int32, device=dev),
                        max_seq_len=int(w.seq_lens[b]), max_query_len=max(1, q1 - q0))
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    return o, l, q0, q1


@pytest.mark.parametrize("hq,hkv,nreq,seed", [
    (8, 2, 40, 7),     # G = 4, up to 2 query tokens: 8 rows
    (8, 1, 151, 8),    # 151 groups: the largest split-KV batch, 16 rows
    (16, 4, 30, 9),    # G = 4 with four KV heads per request
])
def test_balanced_ranges_match_oracle_and_single_requests(hq, hkv, nreq, seed):
    """Split-KV deals the chunks of all (request, KV head) groups out as one
    wave of equal contiguous ranges: ranges start and end inside groups, hold
    several whole groups, and skip a request without query tokens.  Every row
    against the oracle, and chosen requests bit for bit against the same
    request launched alone (a different cut: whole groups folded in one CTA
    against records folded by the last arrival)."""
    import random
    rnd = random.Random(seed)
    lens = [rnd.choice([1, 100, 128, 129, 256, 257, 700, rnd.randint(1, 5000)]) for _ in range(nreq)]
    qlens = [min(L, rnd.choice([1, 1, 1, 2])) for L in lens]
    qlens[3] = 0
    w = _suffix_batch(hq, hkv, lens, qlens, seed=seed)
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    info = pagedattn.last_launch_info()
    print(info)
    assert "decode-swapped" in info and "split" in info
    ref_o, ref_l = oracle_attention(w)
    err_o = float((out.float().cpu().double() - torch.from_numpy(ref_o)).abs().max())
    err_l = lse_rel_err(lse.cpu().numpy(), ref_l)
    print(f"oracle: out max_abs_diff={err_o:.3e} lse rel={err_l:.3e}")
    assert err_o <= OUT_ATOL and err_l <= LSE_RTOL
    for b in sorted({0, 2, 4, nreq // 2, nreq - 1}):
        if qlens[b] == 0:
            continue
        o1, l1, q0, q1 = _alone(dw, w, b)
        _bitwise(out[q0:q1], o1, f"request {b} (L={lens[b]}) in the batch vs alone")
        _bitwise(lse[q0:q1], l1, f"request {b} lse")


def test_scaled_decode_mix_matches_single_requests():
    """The decode length mix repeated 16 times (64 requests, 2432 chunks over
    one wave of CTAs): sampled rows against the oracle, and requests of each
    length bit for bit against the same request alone."""
    lens = list(wl.DECODE_LENS) * 16
    w = wl.decode(seq_lens=lens, num_blocks=sum(wl.pages_needed(L) for L in lens) + 64)
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    info = pagedattn.last_launch_info()
    print(info)
    assert "decode-swapped-r4" in info and "split" in info
    rows = [0, 1, 2, 3, 29, 30, 41, 63]
    ref_o, ref_l = oracle_attention(w, rows=rows)
    o = out.float().cpu().double()[rows]
    assert float((o - torch.from_numpy(ref_o)).abs().max()) <= OUT_ATOL
    assert lse_rel_err(lse.cpu().numpy()[rows], ref_l) <= LSE_RTOL
    for b in (0, 1, 2, 3, 30, 63):
        o1, l1, q0, q1 = _alone(dw, w, b)
        _bitwise(out[q0:q1], o1, f"request {b} (L={lens[b]}) in the batch vs alone")
        _bitwise(lse[q0:q1], l1, f"request {b} lse")


def _deal(lens, qlens, hkv, num_sms):
    """The split-KV deal of the decode kernel, recomputed on the host: for
    each (request, KV head) group, whether one CTA's range holds all of its
    256-key chunks."""
    nch = [(L + 255) // 256 if q > 0 else 0 for L, q in zip(lens, qlens)]
    pre = [0]
    for c in nch:
        pre.append(pre[-1] + c)
    T = hkv * pre[-1]
    G = min(num_sms, T)
    cta_of = lambda x: ((x + 1) * G + T - 1) // T - 1
    whole = {}
    for b, c in enumerate(nch):
        for k in range(hkv):
            if c:
                gs = hkv * pre[b] + k * c
                whole[(b, k)] = cta_of(gs) == cta_of(gs + c - 1)
    return whole


def test_bad_block_ids_in_whole_and_cut_groups():
    """A block id out of range in a request whose groups one CTA folds alone,
    and in one whose groups are cut between CTAs: PA_ERR_BAD_METADATA, NaN
    rows for those two requests, every other row bit for bit unchanged."""
    import random
    rnd = random.Random(21)
    lens = [rnd.choice([100, 300, 700, 1500, 2500]) for _ in range(40)]
    qlens = [1] * 40
    w = _suffix_batch(8, 2, lens, qlens, seed=21)
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    assert "decode-swapped" in pagedattn.last_launch_info() and "split" in pagedattn.last_launch_info()
    whole = _deal(lens, qlens, 2, torch.cuda.get_device_properties(0).multi_processor_count)
    b_whole = next(b for b in range(40) if whole[(b, 0)] and whole[(b, 1)] and lens[b] > 16)
    b_cut = next(b for b in range(40) if not whole[(b, 0)] and not whole[(b, 1)] and b != b_whole)
    bt = dw.block_tables.clone()
    bt[b_whole, (lens[b_whole] - 1) // 16] = w.num_blocks + 3      # its last page
    bt[b_cut, 0] = -7                                                # its first page
    o2, l2 = dw.attention(block_tables=bt)
    st, idx = pagedattn.check_errors()
    assert st == pagedattn.PA_ERR_BAD_METADATA and idx in (b_whole, b_cut)
    for b in (b_whole, b_cut):
        assert torch.isnan(o2[b].float()).all() and torch.isnan(l2[b]).all(), b
    keep = [b for b in range(40) if b not in (b_whole, b_cut)]
    _bitwise(out[keep], o2[keep], f"other requests (bad ids in {b_whole} whole, {b_cut} cut)")
    _bitwise(lse[keep], l2[keep], "other requests lse")


def test_long_sequences_many_chunks_per_cta():
    """Requests up to 150,000 keys: ranges of about ten chunks per CTA, so the
    bad-id flag ring and the Q double buffer wrap, groups span several CTAs
    and short groups sit inside one range.  Every row against the oracle;
    the longest request bit for bit against the same request alone."""
    lens = [150000, 1000, 40000, 700]
    qlens = [1, 1, 1, 1]
    w = _suffix_batch(8, 2, lens, qlens, seed=33)
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    info = pagedattn.last_launch_info()
    print(info)
    assert "decode-swapped-r4" in info and "split" in info
    ref_o, ref_l = oracle_attention(w)
    err_o = float((out.float().cpu().double() - torch.from_numpy(ref_o)).abs().max())
    err_l = lse_rel_err(lse.cpu().numpy(), ref_l)
    print(f"oracle: out max_abs_diff={err_o:.3e} lse rel={err_l:.3e}")
    assert err_o <= OUT_ATOL and err_l <= LSE_RTOL
    for b in (0, 2):
        o1, l1, q0, q1 = _alone(dw, w, b)
        _bitwise(out[q0:q1], o1, f"request {b} (L={lens[b]}) in the batch vs alone")
        _bitwise(lse[q0:q1], l1, f"request {b} lse")


@pytest.mark.parametrize("nreq,hkv,qmax,split", [
    (80, 2, 8, False),   # 160 groups: one CTA per group, 32 rows
    (76, 2, 4, False),   # 152 groups: one CTA per group, 16 rows
    (30, 2, 8, True),    # 32 rows, ranges of several chunks across groups
    (50, 2, 3, True),    # 16 rows (G x 3 tokens), ranges across groups
])
def test_speculative_rows_both_schedules(nreq, hkv, qmax, split):
    """Several query tokens per request (up to 32 rows per group) on both
    schedules: every row against the oracle, and chosen requests bit for bit
    against the same request alone."""
    import random
    rnd = random.Random(nreq * 7 + qmax)
    lens = [rnd.randint(600, 3500) for _ in range(nreq)]
    qlens = [rnd.randint(1, qmax) for _ in range(nreq)]
    qlens[0] = qmax
    w = _suffix_batch(8, hkv, lens, qlens, seed=nreq + qmax)
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    info = pagedattn.last_launch_info()
    print(info)
    rows = 4 * qmax
    expect = next(r for r in (4, 8, 16, 32) if rows <= r)
    assert f"decode-swapped-r{expect}" in info and (("split" in info) == split), info
    ref_o, ref_l = oracle_attention(w)
    err_o = float((out.float().cpu().double() - torch.from_numpy(ref_o)).abs().max())
    err_l = lse_rel_err(lse.cpu().numpy(), ref_l)
    print(f"oracle: out max_abs_diff={err_o:.3e} lse rel={err_l:.3e}")
    assert err_o <= OUT_ATOL and err_l <= LSE_RTOL
    for b in (0, 1, nreq // 2, nreq - 1):
        o1, l1, q0, q1 = _alone(dw, w, b)
        _bitwise(out[q0:q1], o1, f"request {b} (L={lens[b]}, q={qlens[b]}) in the batch vs alone")
        _bitwise(lse[q0:q1], l1, f"request {b} lse")

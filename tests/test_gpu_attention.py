"""K2 (pa_paged_attention) against the fp64 oracle, and GPU-vs-GPU bitwise
properties.

Tolerances: out max-abs <= 2e-2 and lse relative <= 1e-3 against the oracle
for N(0,1) inputs; prefill vs decode and schedule changes bit-exact ("fix(rocm):
stabilize direct paged CK attention for bitwise R/R", Validation:
mismatch_count=0, max_abs_diff=0, torch.equal=true; Additional checks)."""
import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_cache_178_gb300 import pagedattn
from paged_kv_cache_178_gb300 import workloads as wl
from paged_kv_cache_178_gb300.device import DeviceWorkload
from tests.helpers import LSE_RTOL, OUT_ATOL, lse_rel_err, oracle_attention

pytestmark = pytest.mark.gpu


def _run(w, **kw):
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention(**kw)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1), pagedattn.last_launch_info()
    return dw, out, lse


def _compare(w, out, lse, rows=None, compact=False, tag=""):
    ref_o, ref_l = oracle_attention(w, rows=rows, compact=compact)
    o = out.float().cpu().numpy()
    l_ = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l_ = o[rows], l_[rows]
    assert np.isfinite(o).all() and np.isfinite(l_).all()
    err_o = float(np.max(np.abs(o - ref_o)))
    err_l = lse_rel_err(l_, ref_l)
    print(f"{w.name}{tag}: out max_abs_diff={err_o:.3e} lse rel={err_l:.3e} "
          f"[{pagedattn.last_launch_info()}]")
    assert err_o <= OUT_ATOL
    assert err_l <= LSE_RTOL


def _bitwise(a: torch.Tensor, b: torch.Tensor, what: str):
    ai = a.contiguous().view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32)
    bi = b.contiguous().view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)
    mism = int((ai != bi).sum())
    diff = float((a.float() - b.float()).abs().max()) if a.numel() else 0.0
    print(f"{what}: mismatch_count={mism} max_abs_diff={diff} torch.equal={mism == 0}")
    assert mism == 0


def _rows_sample(n, extra=(), k=96, seed=0):
    g = torch.Generator().manual_seed(seed)
    base = {0, 1, 15, 16, 17, 127, 128, 129, 255, 256, 257, 1023, 1024, n - 2, n - 1} | set(extra)
    base |= set(torch.randint(0, n, (k,), generator=g).tolist())
    return sorted(r for r in base if 0 <= r < n)


# ------------------------------------------------------------- parity ----

def test_composition_dh256():
    w = wl.composition()
    dw, out, lse = _run(w)
    _compare(w, out, lse)
    # closed form on the GPU too: row 0 sees one key, so out = v0 bit for bit
    v0 = w.value[0].cuda()
    for h in range(8):
        assert torch.equal(out[0, h], v0[h // 4])


def test_composition_anti_vacuity():
    """Swapping two in-range logical blocks after the write changes the GPU
    output (the composition review's guard).  The pool starts zeroed, as a
    freshly allocated cache would, so the swapped table reads zeros where
    nothing was written and every row stays finite; the GPU result for the
    swapped table still matches the oracle on the same zeroed pool."""
    from oracle import pa_oracle
    from tests.helpers import bits
    w = wl.composition()
    dw = DeviceWorkload(w, fill_bits=0)
    dw.write_cache()
    out, _ = dw.attention()
    bt = w.block_table.clone()
    bt[0, [0, 1]] = bt[0, [1, 0]]
    out2, lse2 = dw.attention(block_tables=bt.cuda())
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    diff = float((out2.float() - out.float()).abs().max())
    print(f"anti-vacuity: swapped in-range blocks change the output by {diff:.3f}")
    assert diff > 1e-3
    pool = pa_oracle.HostPool(w.num_blocks, 2, 256, w.layout, fill_bits=0)
    pa_oracle.reshape_and_cache(bits(w.key), bits(w.value), w.slot_mapping.numpy(), pool)
    ref_o, ref_l = pa_oracle.paged_attention(bits(w.q), pool, bt.numpy(), w.seq_lens.numpy(),
                                             w.query_start_loc.numpy(), w.scale)
    assert float(np.max(np.abs(out2.float().cpu().numpy() - ref_o))) <= OUT_ATOL
    assert lse_rel_err(lse2.cpu().numpy(), ref_l) <= LSE_RTOL


@pytest.mark.parametrize("reversed_pages", [False, True])
def test_decode(reversed_pages):
    w = wl.decode(reversed_pages=reversed_pages)
    dw, out, lse = _run(w)
    _compare(w, out, lse)


def test_decode_separate_layout():
    w = dataclasses.replace(wl.decode(), layout="separate")
    dw, out, lse = _run(w)
    _compare(w, out, lse)


def test_long_prefill_sampled():
    w = wl.long_prefill(4096)
    dw, out, lse = _run(w)
    _compare(w, out, lse, rows=_rows_sample(4096, extra=(2047, 2048, 4094)))


@pytest.mark.parametrize("qlen", [128, 17, 1])
def test_suffix_over_4gb_pool(qlen):
    w = wl.suffix(qlen)
    dw, out, lse = _run(w)
    rows = None if qlen <= 17 else _rows_sample(4 * qlen, k=64)
    _compare(w, out, lse, rows=rows, compact=True, tag=f" q={qlen}")


def test_mixed_batch_small_dims():
    """Prefill, suffix and decode requests in one call, partial pages."""
    gen = torch.Generator().manual_seed(31)
    lens = [300, 16, 700, 1, 29, 513]
    qlens = [300, 16, 9, 1, 1, 40]
    pages = torch.randperm(200, generator=gen).tolist()
    rows, at = [], 0
    for L in lens:
        n = wl.pages_needed(L)
        rows.append(pages[at:at + n])
        at += n
    w = wl.build("mixed_dh128", num_q_heads=8, num_kv_heads=2, head_dim=128, seq_lens=lens,
                 query_lens=qlens, num_blocks=200, block_rows=rows, layout="interleaved", seed=32)
    dw, out, lse = _run(w)
    _compare(w, out, lse)


@pytest.mark.parametrize("hq,hkv,dh", [(2, 2, 128), (6, 2, 128), (32, 2, 128), (128, 1, 128),
                                        (12, 4, 256)])
def test_group_sizes(hq, hkv, dh):
    """Query-head groups G = Hq/Hkv from 1 (one KV head per query head) to
    128 (one token per 128-row tile), and a G that does not divide 128 (rows
    of a tile left unused), on a batch mixing prefill, suffix and decode; the
    prefill rows of one request equal its decode view bit for bit."""
    gen = torch.Generator().manual_seed(40 + hq)
    lens = [300, 700, 1, 513, 40]
    qlens = [300, 9, 1, 1, 40]
    nb = sum(wl.pages_needed(L) for L in lens) + 8
    pages = torch.randperm(nb, generator=gen).tolist()
    rows, at = [], 0
    for L in lens:
        n = wl.pages_needed(L)
        rows.append(pages[at:at + n])
        at += n
    w = wl.build(f"groups_hq{hq}_hkv{hkv}_dh{dh}", num_q_heads=hq, num_kv_heads=hkv, head_dim=dh,
                 seq_lens=lens, query_lens=qlens, num_blocks=nb, block_rows=rows, layout="separate",
                 seed=41 + hq)
    dw, out, lse = _run(w)
    _compare(w, out, lse)
    # request 4 (a 40-token prefill) against its decode view
    q0, q1 = int(w.query_start_loc[4]), int(w.query_start_loc[5])
    kv0 = sum(lens[:4])
    wb = wl.Workload(name=w.name + "_r4", num_q_heads=hq, num_kv_heads=hkv, head_dim=dh, num_blocks=nb,
                     layout=w.layout, q=w.q[q0:q1], key=w.key[kv0:kv0 + 40], value=w.value[kv0:kv0 + 40],
                     slot_mapping=w.slot_mapping[kv0:kv0 + 40], block_table=w.block_table[4:5],
                     seq_lens=w.seq_lens[4:5], query_start_loc=torch.tensor([0, 40], dtype=torch.int32),
                     scale=w.scale)
    _prefill_vs_decode(wb, list(range(40)))


# ------------------------------------------------ prefill == decode bitwise ----

def _prefill_vs_decode(w, rows):
    dw, out, lse = _run(w)
    wd = wl.decode_batch_from_prefill(w, rows)
    dd = DeviceWorkload(wd, fill_bits=None)
    dd.share_cache_with(dw)
    out_d, lse_d = dd.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    info = pagedattn.last_launch_info()
    qoff = int(w.query_start_loc[0])
    idx = torch.tensor([qoff + r for r in rows], device=out.device)
    _bitwise(out.index_select(0, idx), out_d, f"{w.name} out prefill vs decode ({len(rows)} rows; {info})")
    _bitwise(lse.index_select(0, idx), lse_d, f"{w.name} lse prefill vs decode")
    return info


def test_long_prefill_equals_decode_all_rows():
    w = wl.long_prefill(4096)
    _prefill_vs_decode(w, list(range(4096)))


def test_long_prefill_equals_split_decode():
    """A small decode batch runs the split-KV schedule (chunk partials merged
    by the last CTA); it must still equal the prefill rows bit for bit."""
    w = wl.long_prefill(4096)
    info = _prefill_vs_decode(w, [4095, 4000, 2048, 1023, 700, 255, 16, 0])
    assert "split" in info


@pytest.mark.parametrize("qlen", [128, 17])
def test_suffix_equals_decode(qlen):
    w = wl.suffix(qlen, num_blocks=4096)
    # one request at a time: the decode view wants a single-request prefill
    for b in (0, 3):
        q0, q1 = int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])
        kv0 = sum(int(x) for x in w.seq_lens[:b])
        L = int(w.seq_lens[b])
        wb = wl.Workload(name=f"{w.name}_r{b}", num_q_heads=8, num_kv_heads=2, head_dim=128,
                         num_blocks=w.num_blocks, layout=w.layout, q=w.q[q0:q1],
                         key=w.key[kv0:kv0 + L], value=w.value[kv0:kv0 + L],
                         slot_mapping=w.slot_mapping[kv0:kv0 + L], block_table=w.block_table[b:b + 1],
                         seq_lens=w.seq_lens[b:b + 1],
                         query_start_loc=torch.tensor([0, q1 - q0], dtype=torch.int32), scale=w.scale)
        _prefill_vs_decode(wb, list(range(q1 - q0)))


# ------------------------------------------------ schedule invariance ----

def test_bounds_do_not_change_bits():
    w = wl.decode()
    dw, out, lse = _run(w)
    for mq, ms in ((1, 8192), (3, 7168), (40, 20000), (300, 7200)):
        o2, l2 = dw.attention(max_query_len=mq, max_seq_len=ms)
        assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
        _bitwise(out, o2, f"decode bounds mq={mq} ms={ms} [{pagedattn.last_launch_info()}]")
        _bitwise(lse, l2, "decode lse")


def test_batch_composition_and_order_do_not_change_bits():
    w = wl.decode()
    dw, out, lse = _run(w)
    perm = [2, 0, 3, 1]
    dev = out.device
    o2, l2 = dw.attention(q=dw.q[perm].contiguous(), block_tables=dw.block_tables[perm].contiguous(),
                          seq_lens=dw.seq_lens[perm].contiguous())
    _bitwise(out[perm], o2, "decode with requests permuted")
    _bitwise(lse[perm], l2, "lse with requests permuted")
    for b in range(4):
        o1, l1 = dw.attention(q=dw.q[b:b + 1], block_tables=dw.block_tables[b:b + 1].contiguous(),
                              seq_lens=dw.seq_lens[b:b + 1].contiguous(),
                              query_start_loc=torch.tensor([0, 1], dtype=torch.int32, device=dev),
                              max_seq_len=int(w.seq_lens[b]))
        _bitwise(out[b:b + 1], o1, f"request {b} alone")
        _bitwise(lse[b:b + 1], l1, f"request {b} alone (lse)")


@pytest.mark.parametrize("kv_tile", [0, 64])
def test_shared_fold_equals_single_fold(kv_tile):
    """Split-KV decode on a big batch (more units than SMs) and on one request
    of it alone.  In the 128-row kernel (the 64-key canon takes it) the two
    fold differently: with every unit resident the last four arrivals of a
    (request, KV head) group share the chunk fold by columns, otherwise the
    last arrival folds alone; the few-row decode kernel always folds in the
    last arrival.  A request's bits must not depend on the batch."""
    lens = [7168] + [1024] * 40
    w = wl.decode(seq_lens=lens, num_blocks=4096)
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = 2 * sum((L + 255) // 256 for L in lens)
    assert units > n_sms  # the whole batch folds with one CTA per group
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention(kv_tile=kv_tile)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    assert "split" in pagedattn.last_launch_info()
    dev = out.device
    o1, l1 = dw.attention(q=dw.q[0:1], block_tables=dw.block_tables[0:1].contiguous(),
                          seq_lens=dw.seq_lens[0:1].contiguous(),
                          query_start_loc=torch.tensor([0, 1], dtype=torch.int32, device=dev),
                          max_seq_len=7168, kv_tile=kv_tile)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    assert "split" in pagedattn.last_launch_info()
    assert 2 * 28 <= n_sms  # request 0 alone: 56 units, the fold is shared
    _bitwise(out[0:1], o1, "request 0: single-CTA fold vs shared fold")
    _bitwise(lse[0:1], l1, "request 0 lse: single-CTA fold vs shared fold")
    _compare(w, out, lse, rows=[0, 1, 17, 40], tag=" (41 requests)")


def test_prefill_bounds_and_schedule_switch():
    """The same prefill rows through in-CTA and split-KV schedules (the
    schedule follows host bounds only) stay bit-identical."""
    w = wl.long_prefill(1024, pool_factor=3)
    dw, out, lse = _run(w)
    o2, l2 = dw.attention(max_query_len=4096, max_seq_len=65536)
    _bitwise(out, o2, f"prefill larger bounds [{pagedattn.last_launch_info()}]")
    _bitwise(lse, l2, "prefill larger bounds (lse)")


# --------------------------------------------------------- edge cases ----

def test_empty_and_zero_query_requests():
    w = wl.decode(seq_lens=(513, 40, 16), num_blocks=128)
    dw, out, lse = _run(w)
    # an empty call launches nothing and succeeds
    empty = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    pagedattn.paged_attention(empty, dw.k_cache, dw.v_cache, dw.block_tables, dw.seq_lens,
                              torch.zeros(4, dtype=torch.int32, device="cuda"), w.scale, 0, 513)
    # request 1 with zero new tokens: rows of the others are unchanged
    qsl = torch.tensor([0, 1, 1, 2], dtype=torch.int32, device="cuda")
    q2 = dw.q[[0, 2]].contiguous()
    o2, l2 = dw.attention(q=q2, query_start_loc=qsl)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    _bitwise(out[[0, 2]], o2, "zero-length request in the batch")


def test_single_token_sequence():
    w = wl.decode(seq_lens=(1, 2, 17), num_blocks=64)
    dw, out, lse = _run(w)
    _compare(w, out, lse)
    v0 = w.value[0].cuda()
    for h in range(8):
        assert torch.equal(out[0, h], v0[h // 4])


# ------------------------------------------------------ invalid metadata ----

def test_bad_block_id_flags_and_nans_only_that_request():
    w = wl.decode()
    dw, out, lse = _run(w)
    bt = dw.block_tables.clone()
    bt[1, 3] = w.num_blocks + 5
    o2, l2 = dw.attention(block_tables=bt)
    st, idx = pagedattn.check_errors()
    assert st == pagedattn.PA_ERR_BAD_METADATA and idx == 1
    assert torch.isnan(o2[1].float()).all() and torch.isnan(l2[1]).all()
    keep = [0, 2, 3]
    _bitwise(out[keep], o2[keep], "other requests after a bad block id")


def test_seq_len_shorter_than_query_flags():
    w = wl.decode(seq_lens=(513, 40, 16), num_blocks=128)
    dw, out, lse = _run(w)
    sl = dw.seq_lens.clone()
    sl[2] = 0                          # one query token but no cached key
    o2, l2 = dw.attention(seq_lens=sl)
    st, idx = pagedattn.check_errors()
    assert st == pagedattn.PA_ERR_BAD_METADATA and idx == 2
    assert torch.isnan(o2[2].float()).all()
    _bitwise(out[:2], o2[:2], "other requests after seq_len < q_len")


def test_bound_violation_flags():
    w = wl.decode(seq_lens=(513, 40, 16), num_blocks=128)
    dw, out, lse = _run(w)
    o2, l2 = dw.attention(max_seq_len=100)      # request 0 has 513 keys
    st, idx = pagedattn.check_errors()
    assert st == pagedattn.PA_ERR_BAD_METADATA and idx == 0
    _bitwise(out[1:], o2[1:], "other requests after a bound violation")


# ------------------------------------------------------- head dim 512 ----

@pytest.mark.parametrize("L", list(wl.WIDE_LENS))
def test_wide_head_dh512(L):
    """Hq=16, Hkv=2, d=512 causal prefill (two-CTA pairs split the head dim)
    at every stated length ("harden compact peer-local KV prefill for
    Gemma-4", Gates: ~3k / ~11k / ~18k; Scope: 8192), on sampled rows that
    include the first and last row of a page, of a 64-key tile and of a
    1024-key span, and the last row."""
    w = wl.wide_head(L)
    dw, out, lse = _run(w)
    assert "in-cta-pair" in pagedattn.last_launch_info()
    rows = _rows_sample(L, extra=(15, 16, 63, 64, 65, 127, 128, 1023, 1024, L // 2, L - 1),
                        k=24 if L > 8192 else 48)
    _compare(w, out, lse, rows=rows)


@pytest.mark.parametrize("L,nrows", [(3072, 24), (18432, 72)])
def test_wide_head_prefill_equals_decode(L, nrows):
    """Dh=512 prefill rows equal their decode view bit for bit, up to the
    last row of the longest stated length."""
    w = wl.wide_head(L)
    fixed = {0, 15, 16, 63, 64, 127, 128, 1000, 1023, 1024, 2047, L // 2, L - 2, L - 1}
    g = torch.Generator().manual_seed(L)
    rand = set(torch.randint(0, L, (nrows,), generator=g).tolist())
    rows = sorted(fixed | rand)[:max(nrows, len(fixed))]
    rows = sorted(set(rows) | fixed)
    assert len(rows) >= min(nrows, L) and rows[-1] == L - 1
    _prefill_vs_decode(w, rows)


def test_wide_head_suffix_prefill():
    """Dh=512 suffix (chunked) prefill: two requests whose new tokens extend a
    cached context (130 new on 700, 300 new on 300, tails mid-page and
    mid-tile), against the oracle on rows of every query tile of both."""
    lens, qlens = (700, 300), (130, 300)
    g = torch.Generator().manual_seed(5121)
    pages = torch.randperm(96, generator=g).tolist()
    n0 = wl.pages_needed(lens[0])
    rows = [pages[:n0], pages[n0:n0 + wl.pages_needed(lens[1])]]
    w = wl.build("wide_suffix", num_q_heads=16, num_kv_heads=2, head_dim=512, seq_lens=list(lens),
                 query_lens=list(qlens), num_blocks=96, block_rows=rows, layout="interleaved", seed=5122)
    dw, out, lse = _run(w)
    assert "in-cta-pair" in pagedattn.last_launch_info()
    _compare(w, out, lse, rows=[0, 15, 16, 17, 63, 64, 100, 129, 130, 131, 146, 200, 300, 429])


@pytest.mark.parametrize("bad_page", ["first", "last"])
def test_wide_head_bad_block_id(bad_page):
    """Dh=512, two prefill requests: a block id past the pool in request 1
    latches the error for request 1; request 0 is bitwise unchanged.  With
    the bad id on the first page every row of request 1 reads it and is NaN;
    on the last page the rows whose keys reach it are NaN and every other row
    of request 1 is either wholly NaN or bitwise the clean result."""
    lens = (300, 200)
    g = torch.Generator().manual_seed(512)
    pages = torch.randperm(64, generator=g).tolist()
    n0 = wl.pages_needed(lens[0])
    rows = [pages[:n0], pages[n0:n0 + wl.pages_needed(lens[1])]]
    w = wl.build("wide_two_requests", num_q_heads=16, num_kv_heads=2, head_dim=512, seq_lens=list(lens),
                 query_lens=list(lens), num_blocks=64, block_rows=rows, layout="interleaved", seed=5120)
    dw, out, lse = _run(w)
    assert "in-cta-pair" in pagedattn.last_launch_info()
    _compare(w, out, lse, rows=[0, 1, 150, 299, 300, 301, 420, 499])
    bt = dw.block_tables.clone()
    col = 0 if bad_page == "first" else len(rows[1]) - 1
    bt[1, col] = w.num_blocks + 3
    o2, l2 = dw.attention(block_tables=bt)
    st, idx = pagedattn.check_errors()
    assert st == pagedattn.PA_ERR_BAD_METADATA and idx == 1
    _bitwise(out[:lens[0]], o2[:lens[0]], "request 0 beside a bad block id")
    _bitwise(lse[:lens[0]], l2[:lens[0]], "request 0 lse beside a bad block id")
    r1, l1 = o2[lens[0]:].float(), l2[lens[0]:]
    nan_rows = torch.isnan(r1).flatten(1).all(1) & torch.isnan(l1).all(1)
    reaches = torch.arange(lens[1], device=r1.device) >= 16 * col
    assert bool(nan_rows[reaches].all())
    clean = ~nan_rows
    assert not bool(torch.isnan(r1[clean]).any())
    _bitwise(out[lens[0]:][clean], o2[lens[0]:][clean], "request 1 rows clear of the bad page")
    print(f"bad {bad_page} page: {int(nan_rows.sum())} of {lens[1]} rows NaN")


def test_composition_prefill_equals_decode_all_rows():
    """The Dh=256 composition (20 tokens, table {3,1,2,0}): each of the 20
    prefill rows equals its decode view bit for bit."""
    _prefill_vs_decode(wl.composition(), list(range(20)))


# ----------------------------------------------- non-monotone query starts ----

@pytest.mark.parametrize("qsl_bad,bad_rows,bad_reqs", [
    ([0, 1, 3, 2, 4], [1, 2, 3], {1, 2, 3}),   # an inner entry decreases
    ([0, 1, 2, 4, 3], [2, 3], {2, 3}),         # the last step decreases
])
def test_non_monotone_query_start_loc(qsl_bad, bad_rows, bad_reqs):
    """A query_start_loc that decreases is invalid metadata: the request whose
    range is inverted owns no rows, the requests whose ranges now exceed the
    query bound get NaN rows, PA_ERR_BAD_METADATA names one of them, and the
    rows of the requests left intact keep every bit."""
    w = wl.decode()
    dw, out, lse = _run(w)
    qsl = torch.tensor(qsl_bad, dtype=torch.int32, device=out.device)
    o2 = torch.zeros_like(out)
    l2 = torch.zeros_like(lse)
    dw.attention(query_start_loc=qsl, out=o2, lse=l2)
    st, idx = pagedattn.check_errors()
    print(f"qsl={qsl_bad}: status={pagedattn.status_string(st)} index={idx}")
    assert st == pagedattn.PA_ERR_BAD_METADATA and idx in bad_reqs
    for r in bad_rows:
        assert torch.isnan(o2[r].float()).all() and torch.isnan(l2[r]).all()
    keep = [r for r in range(4) if r not in bad_rows]
    _bitwise(out[keep], o2[keep], f"rows {keep} beside a non-monotone query_start_loc")
    _bitwise(lse[keep], l2[keep], "their lse")

"""pa_gather_kv_head on the GPU: the compact active-block gather of one KV
head ("ROCm: harden compact peer-local KV prefill for Gemma-4", Scope and
Required hardening).

- Packed pages, compact table and offsets equal the oracle's bit for bit,
  for shuffled and reversed tables, partial tail pages, empty and one-token
  requests, head dims 128/256/512, and a pool past 2**31 elements.  Pages
  past the last packed one are untouched.
- Attention over the packed one-head pool, through the compact table, with
  the head's query group gives the same bits as attention over the full
  pool.
- A bad block id gives a NaN page and PA_ERR_BAD_METADATA; a bad length
  gives its request no pages; too small a capacity writes only the offsets
  and reports PA_ERR_WORKSPACE with the pages needed.
"""
import numpy as np
import pytest
import torch

from oracle import pa_oracle
from paged_kv_cache_178_gb300 import pagedattn
from paged_kv_cache_178_gb300 import workloads as wl
from paged_kv_cache_178_gb300.device import DeviceWorkload, bf16_fill
from tests.helpers import compact_blocks, oracle_pool

pytestmark = pytest.mark.gpu

FILL = 0x7FC3   # packed buffers start as this NaN pattern: an untouched page keeps it
TAB_FILL = 0x5A5A5A5A


def _mixed_dh256():
    """Full, partial, single-token and empty requests; Hq=8, Hkv=2, Dh=256."""
    lens = [37, 16, 50, 1, 0, 29, 300]
    gen = torch.Generator().manual_seed(91)
    n = sum(wl.pages_needed(L) for L in lens)
    pages = torch.randperm(64, generator=gen)[:n].tolist()
    rows, at = [], 0
    for L in lens:
        k = wl.pages_needed(L)
        rows.append(pages[at:at + k])
        at += k
    return wl.build("gather_mixed_dh256", num_q_heads=8, num_kv_heads=2, head_dim=256, seq_lens=lens,
                    query_lens=[min(L, 3) for L in lens], num_blocks=64, block_rows=rows,
                    layout="separate", seed=92)


CASES = {
    "decode_shuffled": lambda: wl.decode(),
    "decode_reversed": lambda: wl.decode(reversed_pages=True),
    "mixed_dh256": _mixed_dh256,
    "wide_dh512": lambda: wl.wide_head(seq_len=1000),
    "suffix_pool_past_2e31": lambda: wl.suffix(16, batch=2, seq_len=1500),
}


def _buffers(dev, cap, dh, num_seqs, max_blocks):
    pk = bf16_fill((cap, 16, 1, dh), FILL, dev)
    pv = bf16_fill((cap, 16, 1, dh), FILL, dev)
    ct = torch.full((num_seqs, max_blocks), TAB_FILL, dtype=torch.int32, device=dev)
    co = torch.full((num_seqs + 1,), TAB_FILL, dtype=torch.int32, device=dev)
    return pk, pv, ct, co


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("case", list(CASES))
def test_gather_matches_oracle(case):
    w = CASES[case]()
    dw = DeviceWorkload(w)
    dw.write_cache()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    wc, _ = compact_blocks(w) if w.num_blocks > 4096 else (w, None)
    pool = oracle_pool(wc)
    total = sum(wl.pages_needed(int(L)) for L in w.seq_lens)
    cap = total + 3
    for h in range(w.num_kv_heads):
        pk, pv, ct, co = _buffers(dw.q.device, cap, w.head_dim, w.num_seqs, w.block_table.shape[1])
        pagedattn.gather_kv_head(dw.k_cache, dw.v_cache, h, dw.block_tables, dw.seq_lens, pk, pv, ct, co)
        assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
        g = pa_oracle.gather_kv_head(pool, h, wc.block_table.numpy(), wc.seq_lens.numpy(), cap)
        assert g.bad_requests == [] and g.budget_needed is None
        mk = int((_u16(pk[:total, :, 0]) != g.packed_k).sum())
        mv = int((_u16(pv[:total, :, 0]) != g.packed_v).sum())
        print(f"{case} head {h}: {total} pages, mismatch K={mk} V={mv}")
        assert mk == 0 and mv == 0
        assert (_u16(pk[total:]) == FILL).all() and (_u16(pv[total:]) == FILL).all()
        assert np.array_equal(ct.cpu().numpy(), g.compact_tables)
        assert np.array_equal(co.cpu().numpy(), g.offsets)


@pytest.mark.parametrize("case", ["decode_shuffled", "mixed_dh256", "wide_dh512", "suffix_pool_past_2e31"])
def test_attention_on_packed_pool_equals_full_pool(case):
    w = CASES[case]()
    dw = DeviceWorkload(w)
    dw.write_cache()
    out_full, lse_full = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    G = w.num_q_heads // w.num_kv_heads
    total = sum(wl.pages_needed(int(L)) for L in w.seq_lens)
    dev = dw.q.device
    for h in range(w.num_kv_heads):
        pk, pv, ct, co = _buffers(dev, total, w.head_dim, w.num_seqs, w.block_table.shape[1])
        pagedattn.gather_kv_head(dw.k_cache, dw.v_cache, h, dw.block_tables, dw.seq_lens, pk, pv, ct, co)
        q = dw.q[:, h * G:(h + 1) * G]
        ws = pagedattn.new_workspace(w.num_seqs, G, 1, w.head_dim, w.max_query_len, w.max_seq_len, dev)
        out, lse = pagedattn.paged_attention(q, pk, pv, ct, dw.seq_lens, dw.query_start_loc, w.scale,
                                             w.max_query_len, w.max_seq_len, workspace=ws)
        assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
        mo = int((out.view(torch.int16) != out_full[:, h * G:(h + 1) * G].contiguous().view(torch.int16)).sum())
        ml = int((lse.view(torch.int32) != lse_full[:, h * G:(h + 1) * G].contiguous().view(torch.int32)).sum())
        print(f"{case} head {h}: packed-pool attention mismatch out={mo} lse={ml}")
        assert mo == 0 and ml == 0


def test_budget_exceeded_writes_offsets_only():
    w = wl.decode()
    dw = DeviceWorkload(w)
    dw.write_cache()
    total = sum(wl.pages_needed(int(L)) for L in w.seq_lens)
    pk, pv, ct, co = _buffers(dw.q.device, total - 1, 128, 4, w.block_table.shape[1])
    pagedattn.gather_kv_head(dw.k_cache, dw.v_cache, 1, dw.block_tables, dw.seq_lens, pk, pv, ct, co)
    assert pagedattn.check_errors() == (pagedattn.PA_ERR_WORKSPACE, total)
    assert (_u16(pk) == FILL).all() and (_u16(pv) == FILL).all()
    assert (ct.cpu().numpy() == TAB_FILL).all()
    g = pa_oracle.gather_kv_head(oracle_pool(w), 1, w.block_table.numpy(), w.seq_lens.numpy(), total - 1)
    assert g.budget_needed == total
    assert np.array_equal(co.cpu().numpy(), g.offsets)
    # zero capacity, no packed buffers: the offsets tell the caller the size
    co0 = torch.full((5,), TAB_FILL, dtype=torch.int32, device=dw.q.device)
    st = pagedattn.load().pa_gather_kv_head(
        pagedattn.ctypes.byref(pagedattn.cache_struct(dw.k_cache, dw.v_cache)), 0, dw.block_tables.data_ptr(),
        w.block_table.shape[1], dw.seq_lens.data_ptr(), 4, None, None, 0, ct.data_ptr(), co0.data_ptr(), None)
    assert st == pagedattn.PA_OK
    assert pagedattn.check_errors() == (pagedattn.PA_ERR_WORKSPACE, total)
    assert np.array_equal(co0.cpu().numpy(), g.offsets)


def test_bad_block_id_and_bad_length():
    w = _mixed_dh256()
    dw = DeviceWorkload(w)
    dw.write_cache()
    bt = w.block_table.clone()
    bt[2, 3] = w.num_blocks + 5       # last selected page of request 2
    lens = w.seq_lens.clone()
    dev = dw.q.device
    total = sum(wl.pages_needed(int(L)) for L in lens)
    pk, pv, ct, co = _buffers(dev, total, 256, w.num_seqs, bt.shape[1])
    pagedattn.gather_kv_head(dw.k_cache, dw.v_cache, 0, bt.to(dev), lens.to(dev), pk, pv, ct, co)
    assert pagedattn.check_errors() == (pagedattn.PA_ERR_BAD_METADATA, 2)
    g = pa_oracle.gather_kv_head(oracle_pool(w), 0, bt.numpy(), lens.numpy(), total)
    assert g.bad_requests == [2]
    assert np.array_equal(_u16(pk[:, :, 0]), g.packed_k) and np.array_equal(_u16(pv[:, :, 0]), g.packed_v)
    assert (_u16(pk[int(g.offsets[2]) + 3]) == pa_oracle.NAN_BITS).all()
    # a length past the table row: its request gets no pages
    lens[6] = 16 * bt.shape[1] + 1
    bt = w.block_table.clone()
    pk, pv, ct, co = _buffers(dev, total, 256, w.num_seqs, bt.shape[1])
    pagedattn.gather_kv_head(dw.k_cache, dw.v_cache, 1, bt.to(dev), lens.to(dev), pk, pv, ct, co)
    assert pagedattn.check_errors() == (pagedattn.PA_ERR_BAD_METADATA, 6)
    g = pa_oracle.gather_kv_head(oracle_pool(w), 1, bt.numpy(), lens.numpy(), total)
    assert g.bad_requests == [6]
    n = int(g.offsets[-1])
    assert np.array_equal(co.cpu().numpy(), g.offsets) and np.array_equal(ct.cpu().numpy(), g.compact_tables)
    assert np.array_equal(_u16(pk[:n, :, 0]), g.packed_k) and (_u16(pk[n:]) == FILL).all()


def test_prepared_gather_in_a_graph_repeats_eager():
    """The prepared call captured in a CUDA graph and replayed gives the
    eager call's bytes (metadata, packed pages), head after head."""
    w = wl.decode(reversed_pages=True)
    dw = DeviceWorkload(w)
    dw.write_cache()
    total = sum(wl.pages_needed(int(L)) for L in w.seq_lens)
    dev = dw.q.device
    ref = []
    for h in range(2):
        pk, pv, ct, co = _buffers(dev, total, 128, 4, w.block_table.shape[1])
        pagedattn.gather_kv_head(dw.k_cache, dw.v_cache, h, dw.block_tables, dw.seq_lens, pk, pv, ct, co)
        ref.append((pk, pv, ct, co))
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    s = torch.cuda.Stream()
    bufs = [_buffers(dev, total, 128, 4, w.block_table.shape[1]) for _ in range(2)]
    calls = [pagedattn.prepare_gather_kv_head(dw.k_cache, dw.v_cache, h, dw.block_tables, dw.seq_lens, *bufs[h],
                                              stream=s) for h in range(2)]
    pagedattn.init()
    with torch.cuda.stream(s):
        calls[0]()
    s.synchronize()
    for b in bufs:
        for t in b:
            t.fill_(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls[0]()
        calls[1]()
    g.replay()
    torch.cuda.synchronize()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    for h in range(2):
        for a, b, what in zip(bufs[h], ref[h], ("packed K", "packed V", "compact table", "offsets")):
            same = torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
            print(f"graph replay head {h}: {what} equal={same}")
            assert same

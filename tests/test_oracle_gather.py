"""Pins for the oracle's compact active-block gather ("ROCm: harden compact
peer-local KV prefill for Gemma-4", Scope and Required hardening): each test
checks it against something other than itself.

- The packed rows of each request, read in order, are the K/V rows that the
  generator made for that request (no pool, no table involved).
- Offsets follow the closed form sum of ceil(L / 16), spelled out by hand.
- Attention over the one-head packed pool through the compact table equals
  attention over the full pool for that head's query group.
- Table columns past a request's pages hold a poison id and are never read;
  bad ids, bad lengths and an exceeded budget are reported as stated.
"""
import numpy as np

from oracle import pa_oracle
from paged_kv_cache_178_gb300 import workloads as wl
from tests.helpers import bits, oracle_pool


def _mixed():
    """Lengths with full, partial, single-token and empty requests; shuffled
    pages in a pool with spare blocks; Hq=8, Hkv=2, Dh=32."""
    lens = [37, 16, 50, 1, 0, 29]
    rows = [[7, 2, 19], [11], [0, 13, 4, 21], [9], [], [3, 17]]
    return wl.build("gather_mixed", num_q_heads=8, num_kv_heads=2, head_dim=32, seq_lens=lens,
                    query_lens=[1 if L else 0 for L in lens], num_blocks=24, block_rows=rows,
                    layout="interleaved", seed=77)


def _request_rows(w, b):
    start = int(sum(int(x) for x in w.seq_lens[:b]))
    return start, start + int(w.seq_lens[b])


def test_offsets_closed_form():
    w = _mixed()
    g = pa_oracle.gather_kv_head(oracle_pool(w), 0, w.block_table.numpy(), w.seq_lens.numpy(), 64)
    # pages per request: 3, 1, 4, 1, 0, 2
    assert g.offsets.tolist() == [0, 3, 4, 8, 9, 9, 11]
    assert g.bad_requests == [] and g.budget_needed is None
    assert g.packed_k.shape == (11, 16, 32)
    expect = np.full((6, 4), -1)
    expect[0, :3] = [0, 1, 2]
    expect[1, :1] = [3]
    expect[2, :4] = [4, 5, 6, 7]
    expect[3, :1] = [8]
    expect[5, :2] = [9, 10]
    assert np.array_equal(g.compact_tables, expect)


def test_packed_rows_are_the_generated_tokens():
    """Request b's packed pages, flattened, start with exactly the rows the
    generator made for b (head h); the rest of its last page is the pool's
    untouched fill."""
    w = _mixed()
    pool = oracle_pool(w)
    for h in range(w.num_kv_heads):
        g = pa_oracle.gather_kv_head(pool, h, w.block_table.numpy(), w.seq_lens.numpy(), 11)
        for b in range(w.num_seqs):
            L = int(w.seq_lens[b])
            t0, t1 = _request_rows(w, b)
            o0, o1 = int(g.offsets[b]), int(g.offsets[b + 1])
            flat_k = g.packed_k[o0:o1].reshape(-1, w.head_dim)
            flat_v = g.packed_v[o0:o1].reshape(-1, w.head_dim)
            assert np.array_equal(flat_k[:L], bits(w.key[t0:t1, h]))
            assert np.array_equal(flat_v[:L], bits(w.value[t0:t1, h]))
            assert (flat_k[L:] == wl.SENTINEL_BITS).all() and (flat_v[L:] == wl.SENTINEL_BITS).all()


def test_attention_on_packed_pool_equals_full_pool():
    w = _mixed()
    pool = oracle_pool(w)
    G = w.num_q_heads // w.num_kv_heads
    full_o, full_l = pa_oracle.paged_attention(bits(w.q), pool, w.block_table.numpy(), w.seq_lens.numpy(),
                                               w.query_start_loc.numpy(), w.scale)
    for h in range(w.num_kv_heads):
        g = pa_oracle.gather_kv_head(pool, h, w.block_table.numpy(), w.seq_lens.numpy(), 16)
        packed = pa_oracle.pool_from_packed(g.packed_k, g.packed_v, 16)
        o, l = pa_oracle.paged_attention(bits(w.q[:, h * G:(h + 1) * G]), packed, g.compact_tables,
                                         w.seq_lens.numpy(), w.query_start_loc.numpy(), w.scale)
        assert np.array_equal(o, full_o[:, h * G:(h + 1) * G])
        assert np.array_equal(l, full_l[:, h * G:(h + 1) * G])


def test_wrong_head_or_page_order_is_caught():
    """The invariants above are sharp: swapping two pages of a request, or
    taking the other head, moves the packed rows off the generated tokens."""
    w = _mixed()
    pool = oracle_pool(w)
    bt = w.block_table.numpy().copy()
    bt[2, [0, 1]] = bt[2, [1, 0]]
    g = pa_oracle.gather_kv_head(pool, 0, bt, w.seq_lens.numpy(), 11)
    t0, t1 = _request_rows(w, 2)
    flat = g.packed_k[4:8].reshape(-1, w.head_dim)[:50]
    assert not np.array_equal(flat, bits(w.key[t0:t1, 0]))
    g1 = pa_oracle.gather_kv_head(pool, 1, w.block_table.numpy(), w.seq_lens.numpy(), 11)
    assert not np.array_equal(g1.packed_k[4:8].reshape(-1, w.head_dim)[:50], bits(w.key[t0:t1, 0]))


def test_bad_metadata_and_budget():
    w = _mixed()
    pool = oracle_pool(w)
    bt = w.block_table.numpy().copy()
    bt[2, 3] = w.num_blocks  # the last selected page of request 2: out of the pool
    lens = w.seq_lens.numpy().copy()
    lens[5] = 16 * bt.shape[1] + 1  # longer than its table row
    g = pa_oracle.gather_kv_head(pool, 1, bt, lens, 64)
    assert g.bad_requests == [2, 5]
    assert g.offsets.tolist() == [0, 3, 4, 8, 9, 9, 9]
    assert (g.packed_k[7] == pa_oracle.NAN_BITS).all() and (g.packed_v[7] == pa_oracle.NAN_BITS).all()
    assert (g.compact_tables[5] == -1).all()
    # budget: 11 pages needed, 10 available -> offsets only
    g = pa_oracle.gather_kv_head(pool, 0, w.block_table.numpy(), w.seq_lens.numpy(), 10)
    assert g.budget_needed == 11 and g.packed_k is None and g.compact_tables is None
    assert g.offsets.tolist() == [0, 3, 4, 8, 9, 9, 11]

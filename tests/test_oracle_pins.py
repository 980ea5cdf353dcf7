"""Pins for the CPU oracle: each test checks it against something other than
itself -- a value the pages print, a library routine on an equivalent dense
problem, closed forms, brute force on tiny inputs, or an invariant -- so that
a dropped term, a wrong index or sign, or a transposed operand fails here.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, logsumexp

from oracle import pa_oracle
from paged_kv_cache_178_gb300 import workloads as wl
from tests.helpers import bits, bits_to_f64, oracle_attention, oracle_pool

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out


# ---------------------------------------------------------------- slots ----

def test_composition_slots_match_page():
    """The review of the composition PR prints the physical slots that
    logical positions 0..19 map to through table {3,1,2,0}."""
    g = _golden("composition_slots.txt")
    w = wl.composition()
    assert [int(x) for x in g["table"].split()] == w.block_table[0, :4].tolist()
    assert w.slot_mapping.tolist() == [int(x) for x in g["read_slots"].split()]


def test_vacuous_write_mapping_is_detected():
    """Writing with the rejected (i*7+3)%64 rule leaves most read positions
    unwritten; the oracle reads only table slots, so the sentinel shows up as
    NaN instead of a silent match."""
    w = wl.composition()
    vac = np.array([(i * 7 + 3) % 64 for i in range(20)], dtype=np.int64)
    read = set(w.slot_mapping.tolist())
    assert len(read & set(vac.tolist())) < 20
    pool = pa_oracle.HostPool(4, 2, 256, "separate")
    assert pa_oracle.reshape_and_cache(bits(w.key), bits(w.value), vac, pool) == 0
    out, lse = oracle_attention(w, pool=pool)
    assert np.isnan(out).any()
    out2, lse2 = oracle_attention(w)
    assert np.isfinite(out2).all() and np.isfinite(lse2).all()


# -------------------------------------------------------------- scatter ----

@pytest.mark.parametrize("layout", ["separate", "interleaved"])
def test_scatter_matches_numpy_assignment(layout):
    gen = torch.Generator().manual_seed(5)
    nb, hkv, dh, n = 6, 2, 8, 40
    key = wl.bf16_randn((n, hkv, dh), gen)
    val = wl.bf16_randn((n, hkv, dh), gen)
    slots = torch.randperm(nb * 16, generator=gen)[:n].to(torch.int64)
    slots[3] = -1
    slots[17] = -5
    pool = pa_oracle.HostPool(nb, hkv, dh, layout)
    assert pa_oracle.reshape_and_cache(bits(key), bits(val), slots.numpy(), pool) == 0
    ref_k = np.full((nb, 16, hkv, dh), wl.SENTINEL_BITS, dtype=np.uint16)
    ref_v = ref_k.copy()
    s = slots.numpy()
    keep = s >= 0
    ref_k[s[keep] // 16, s[keep] % 16] = bits(key)[keep]
    ref_v[s[keep] // 16, s[keep] % 16] = bits(val)[keep]
    assert np.array_equal(pool.view("k"), ref_k)
    assert np.array_equal(pool.view("v"), ref_v)


def test_scatter_reports_out_of_range_slot():
    gen = torch.Generator().manual_seed(6)
    key = wl.bf16_randn((4, 1, 8), gen)
    pool = pa_oracle.HostPool(2, 1, 8, "separate")
    slots = np.array([0, 31, 32, 5], dtype=np.int64)
    assert pa_oracle.reshape_and_cache(bits(key), bits(key), slots, pool) == 3
    assert np.array_equal(pool.view("k")[1, 15, 0], bits(key)[1, 0])


# ------------------------------------------------- dense library special case ----

def _dense_reference(w):
    """torch SDPA in fp64 on each request's contiguous K/V, taken straight from
    the generator's per-token rows (no pool, no table), with K/V heads
    repeated per query group; LSE from scipy's logsumexp of q.k*scale."""
    outs, lses = [], []
    G = w.num_q_heads // w.num_kv_heads
    kv_at = 0
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        q0, q1 = int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])
        qn = q1 - q0
        q = torch.from_numpy(bits_to_f64(bits(w.q[q0:q1]))).permute(1, 0, 2)   # [Hq, qn, Dh]
        k = torch.from_numpy(bits_to_f64(bits(w.key[kv_at:kv_at + L]))).permute(1, 0, 2)
        v = torch.from_numpy(bits_to_f64(bits(w.value[kv_at:kv_at + L]))).permute(1, 0, 2)
        kv_at += L
        k = k.repeat_interleave(G, dim=0)
        v = v.repeat_interleave(G, dim=0)
        mask = torch.arange(L)[None, :] <= (L - qn + torch.arange(qn))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None], k[None], v[None], attn_mask=mask, scale=float(w.scale))[0]
        scores = np.einsum("hqd,hkd->hqk", q.numpy(), k.numpy()) * float(w.scale)
        scores = np.where(mask.numpy()[None], scores, -np.inf)
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(logsumexp(scores, axis=-1).T)
    return np.concatenate(outs), np.concatenate(lses)


def _mixed_workload():
    """Two prefills, a suffix and two decodes at small sizes, Hq=8/Hkv=2."""
    gen = torch.Generator().manual_seed(11)
    lens = [37, 16, 50, 1, 29]
    qlens = [37, 16, 9, 1, 1]
    pages = torch.randperm(40, generator=gen).tolist()
    rows, at = [], 0
    for L in lens:
        n = wl.pages_needed(L)
        rows.append(pages[at:at + n])
        at += n
    return wl.build("mixed", num_q_heads=8, num_kv_heads=2, head_dim=32, seq_lens=lens,
                    query_lens=qlens, num_blocks=40, block_rows=rows, layout="interleaved",
                    seed=12)


def _wide_small():
    """Hq=16, Hkv=2 (G=8), Dh=512: the wide-head geometry at a small length."""
    return wl.build("wide_small", num_q_heads=16, num_kv_heads=2, head_dim=512, seq_lens=[40, 17],
                    query_lens=[40, 5], num_blocks=8, block_rows=[[5, 2, 7], [0, 3]],
                    layout="interleaved", seed=41)


@pytest.mark.parametrize("make", [wl.composition, _mixed_workload, _wide_small])
def test_matches_dense_sdpa(make):
    w = make()
    out, lse = oracle_attention(w)
    ref_o, ref_l = _dense_reference(w)
    assert np.max(np.abs(out - ref_o)) < 1e-12
    assert np.max(np.abs(lse - ref_l)) < 1e-12


def test_decode_lengths_match_dense_sdpa():
    """Decode over partial tail pages (4171 = 260*16 + 11, 513 = 32*16 + 1),
    Dh=128, unwritten tail slots hold the NaN sentinel."""
    w = wl.decode(seq_lens=(4171, 513, 40), num_blocks=512)
    out, lse = oracle_attention(w)
    ref_o, ref_l = _dense_reference(w)
    assert np.isfinite(out).all()
    assert np.max(np.abs(out - ref_o)) < 1e-12
    assert np.max(np.abs(lse - ref_l)) < 1e-12


# ------------------------------------------------------------ brute force ----

def test_brute_force_tiny():
    """n <= 8 keys, Dh = 4, every softmax term written out with Python floats."""
    gen = torch.Generator().manual_seed(13)
    lens, qlens = [7, 3, 8], [7, 2, 1]
    w = wl.build("tiny", num_q_heads=4, num_kv_heads=2, head_dim=4, seq_lens=lens,
                 query_lens=qlens, num_blocks=5, block_rows=[[4], [0], [2]],
                 layout="separate", seed=14, scale=0.7)
    out, lse = oracle_attention(w)
    qf = bits_to_f64(bits(w.q))
    kf = bits_to_f64(bits(w.key))
    vf = bits_to_f64(bits(w.value))
    kv_at, row = 0, 0
    for b, (L, qn) in enumerate(zip(lens, qlens)):
        for i in range(qn):
            pos = L - qn + i
            for h in range(4):
                g = h // 2
                terms = []
                for j in range(pos + 1):
                    s = 0.0
                    for d in range(4):
                        s += float(qf[row, h, d]) * float(kf[kv_at + j, g, d])
                    terms.append(float(np.float32(0.7)) * s)
                m = max(terms)
                e = [math.exp(t - m) for t in terms]
                z = math.fsum(e)
                for d in range(4):
                    want = math.fsum(e[j] / z * float(vf[kv_at + j, g, d]) for j in range(pos + 1))
                    assert abs(out[row, h, d] - want) < 1e-13
                assert abs(lse[row, h] - (m + math.log(z))) < 1e-13
            row += 1
        kv_at += L


# ----------------------------------------------------------- closed forms ----

def test_first_row_is_first_value():
    """Causal row 0 sees one key: out = v0 exactly, lse = s0."""
    w = wl.composition()
    out, lse = oracle_attention(w, rows=[0])
    v0 = bits_to_f64(bits(w.value[0]))            # [Hkv, Dh]
    k0 = bits_to_f64(bits(w.key[0]))
    q0 = bits_to_f64(bits(w.q[0]))
    for h in range(8):
        assert np.array_equal(out[0, h], v0[h // 4])
        assert abs(lse[0, h] - float(w.scale) * float(np.dot(q0[h], k0[h // 4]))) < 1e-12


def test_two_keys_sigmoid():
    """Row 1 sees two keys: weights are logistic functions of s0 - s1."""
    w = wl.composition()
    out, lse = oracle_attention(w, rows=[1])
    q = bits_to_f64(bits(w.q[1]))
    k = bits_to_f64(bits(w.key[:2]))
    v = bits_to_f64(bits(w.value[:2]))
    for h in range(8):
        g = h // 4
        s0 = float(w.scale) * np.dot(q[h], k[0, g])
        s1 = float(w.scale) * np.dot(q[h], k[1, g])
        want = expit(s0 - s1) * v[0, g] + expit(s1 - s0) * v[1, g]
        assert np.max(np.abs(out[0, h] - want)) < 1e-12
        assert abs(lse[0, h] - np.logaddexp(s0, s1)) < 1e-12


def test_identical_keys_and_zero_query_give_mean():
    """All keys equal (or q = 0): uniform weights, out = mean(V),
    lse = s + ln(n)."""
    w = wl.composition()
    key = w.key.clone()
    key[:] = key[5]
    w2 = wl.Workload(**{**w.__dict__, "key": key})
    out, lse = oracle_attention(w2)
    q = bits_to_f64(bits(w.q))
    k5 = bits_to_f64(bits(w.key[5]))
    vf = bits_to_f64(bits(w.value))
    for t in range(20):
        for h in range(8):
            g = h // 4
            assert np.max(np.abs(out[t, h] - vf[: t + 1, g].mean(axis=0))) < 1e-12
            s = float(w.scale) * float(np.dot(q[t, h], k5[g]))
            assert abs(lse[t, h] - (s + math.log(t + 1))) < 1e-12
    qz = torch.zeros_like(w.q)
    w3 = wl.Workload(**{**w.__dict__, "q": qz})
    out3, lse3 = oracle_attention(w3)
    assert np.max(np.abs(lse3[:, 0] - np.log(np.arange(1, 21)))) < 1e-12
    assert np.max(np.abs(out3[7, 3] - vf[:8, 0].mean(axis=0))) < 1e-12


# ------------------------------------------------------------- invariants ----

def test_block_permutation_invariance():
    """Relabelling physical blocks, with table and slots remapped the same
    way, leaves every output bit unchanged."""
    w = _mixed_workload()
    out, lse = oracle_attention(w)
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(99))
    bt = w.block_table.clone()
    for r in range(bt.shape[0]):
        for c in range(wl.pages_needed(int(w.seq_lens[r]))):
            bt[r, c] = int(perm[int(bt[r, c])])
    sm = torch.tensor([int(perm[s // 16]) * 16 + s % 16 for s in w.slot_mapping.tolist()])
    w2 = wl.Workload(**{**w.__dict__, "block_table": bt, "slot_mapping": sm})
    out2, lse2 = oracle_attention(w2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_batch_composition_invariance():
    """A request's rows do not depend on the other requests in the batch."""
    w = _mixed_workload()
    out, lse = oracle_attention(w)
    pool = oracle_pool(w)
    for b in range(w.num_seqs):
        q0, q1 = int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])
        o1, l1 = pa_oracle.paged_attention(
            bits(w.q[q0:q1]), pool, w.block_table[b:b + 1].numpy(), w.seq_lens[b:b + 1].numpy(),
            np.array([0, q1 - q0], dtype=np.int32), w.scale)
        assert np.array_equal(o1, out[q0:q1]) and np.array_equal(l1, lse[q0:q1])


def test_row_sampling_matches_full():
    w = _mixed_workload()
    out, lse = oracle_attention(w)
    rows = [0, 5, 36, 40, 61, 62]
    o2, l2 = oracle_attention(w, rows=rows)
    assert np.array_equal(o2, out[rows]) and np.array_equal(l2, lse[rows])


# ---------------------------------------------------------- anti-vacuity ----

def test_in_range_block_swap_changes_output():
    """Swapping logical blocks 0 and 1 (both hold real tokens) after the write
    must change the result; swapping two columns past the last page must not
    (such a guard would be vacuous, as the composition review found)."""
    w = wl.composition()
    pool = oracle_pool(w)
    out, _ = oracle_attention(w, pool=pool)
    swapped = w.block_table.clone()
    swapped[0, [0, 1]] = swapped[0, [1, 0]]
    w_in = wl.Workload(**{**w.__dict__, "block_table": swapped})
    out_in, _ = oracle_attention(w_in, pool=pool)
    # rows 0..3 now read tokens 16..19 (finite, different); later rows also
    # reach unwritten slots of the partial block and turn NaN.
    assert np.isfinite(out_in[:4]).all()
    assert np.max(np.abs(out_in[:4] - out[:4])) > 1e-3
    assert np.isnan(out_in[4:]).all()
    beyond = w.block_table.clone()
    beyond[0, [2, 3]] = beyond[0, [3, 2]]
    w_out = wl.Workload(**{**w.__dict__, "block_table": beyond})
    out_out, _ = oracle_attention(w_out, pool=pool)
    assert np.array_equal(out_out, out)


def test_one_written_value_moves_output():
    w = wl.composition()
    pool = oracle_pool(w)
    out, _ = oracle_attention(w, pool=pool)
    pool.view("v")[1, 2, 0, :] = bits(torch.full((256,), 3.0, dtype=torch.bfloat16))
    out2, _ = oracle_attention(w, pool=pool)
    # logical position 18 lives in block 1 (table column 1), offset 2
    assert np.max(np.abs(out2[18:, :4] - out[18:, :4])) > 1e-3
    assert np.array_equal(out2[:18], out[:18])


def test_bad_block_id_reports_and_nans():
    w = wl.composition()
    pool = oracle_pool(w)
    bt = w.block_table.clone()
    bt[0, 1] = 7
    o, l = pa_oracle.paged_attention(bits(w.q), pool, bt.numpy(), w.seq_lens.numpy(),
                                     w.query_start_loc.numpy(), w.scale)
    assert np.isnan(o[16:]).all() and np.isfinite(o[:16]).all()

"""pa_reshape_and_paged_attention: ReshapeAndCache followed by PagedAttention
in one library call ("test(rocm): ReshapeAndCache->PagedAttention composition
at real dims", What changed).  Its attention grid reads metadata, tables and
q while the cache write still runs; only its K/V copies wait for the write.

Checked here: the pool it leaves and its out / lse are bit-identical to the
two separate calls; the decode pattern, where the attention must see the
token written in the same call, matches the oracle; a graph replay of the
prepared call repeats the eager bits."""
import numpy as np
import pytest
import torch

from paged_kv_cache_178_gb300 import pagedattn
from paged_kv_cache_178_gb300 import workloads as wl
from paged_kv_cache_178_gb300.device import DeviceWorkload
from tests.helpers import LSE_RTOL, OUT_ATOL, lse_rel_err, oracle_attention

pytestmark = pytest.mark.gpu


def _bits_equal(a: torch.Tensor, b: torch.Tensor, what: str):
    ai = a.contiguous().view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32)
    bi = b.contiguous().view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)
    mism = int((ai != bi).sum())
    print(f"{what}: mismatch_count={mism}")
    assert mism == 0


def _two_calls(w):
    dw = DeviceWorkload(w)
    dw.write_cache()
    out, lse = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    return dw, out, lse


CASES = {
    "composition_dh256": lambda: wl.composition(),
    "decode": lambda: wl.decode(),
    "decode_reversed": lambda: wl.decode(reversed_pages=True),
    "prefill_1024": lambda: wl.long_prefill(1024),
    "prefill_4096_pair": lambda: wl.long_prefill(4096),
    "suffix_q17": lambda: wl.suffix(17, num_blocks=4096),
    "wide_dh512_3072": lambda: wl.wide_head(3072),
}


@pytest.mark.parametrize("name", list(CASES))
def test_one_call_equals_two_calls(name):
    w = CASES[name]()
    ref, out_r, lse_r = _two_calls(w)
    dw = DeviceWorkload(w)
    out, lse = dw.write_and_attend()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    info = pagedattn.last_launch_info()
    print(info)
    assert info.startswith("reshape_and_cache")
    assert ("early_reads" in info) == (w.head_dim != 512)
    _bits_equal(dw.pool, ref.pool, f"{name}: pool")
    _bits_equal(out, out_r, f"{name}: out")
    _bits_equal(lse, lse_r, f"{name}: lse")


def test_decode_step_sees_the_token_it_writes():
    """The decode pattern: the pool holds every token but each request's last
    one (its slot keeps the sentinel fill); one call writes the new token and
    attends over it.  A read of K/V before the write completed would see the
    sentinel (a NaN) or stale bits."""
    w = wl.decode()
    lens = [int(x) for x in w.seq_lens]
    last = np.cumsum(lens) - 1
    keep = np.setdiff1d(np.arange(sum(lens)), last)
    dw = DeviceWorkload(w)
    idx_keep = torch.as_tensor(keep, device="cuda")
    idx_new = torch.as_tensor(last, device="cuda")
    pagedattn.reshape_and_cache(dw.key[idx_keep], dw.value[idx_keep], dw.k_cache, dw.v_cache,
                                dw.slot_mapping[idx_keep].contiguous())
    out, lse = dw.write_and_attend(key=dw.key[idx_new].contiguous(), value=dw.value[idx_new].contiguous(),
                                   slot_mapping=dw.slot_mapping[idx_new].contiguous())
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    ref_o, ref_l = oracle_attention(w)
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    err_o = float(np.max(np.abs(o - ref_o)))
    err_l = lse_rel_err(lse.cpu().numpy().astype(np.float64), ref_l)
    print(f"decode step in one call: out max_abs_diff={err_o:.3e} lse rel={err_l:.3e}")
    assert err_o <= OUT_ATOL and err_l <= LSE_RTOL
    _, out_r, lse_r = _two_calls(w)
    _bits_equal(out, out_r, "decode step: out vs two calls")
    _bits_equal(lse, lse_r, "decode step: lse vs two calls")


def test_prepared_call_in_a_graph_repeats_the_bits():
    w = wl.decode()
    dw = DeviceWorkload(w)
    out = torch.empty((w.q.shape[0], 8, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.q.shape[0], 8), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    call = pagedattn.prepare_reshape_and_paged_attention(
        dw.key, dw.value, dw.slot_mapping, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.seq_lens,
        dw.query_start_loc, w.scale, dw.max_query_len, dw.max_seq_len, out, lse, dw.workspace, stream=s)
    pagedattn.init()
    with torch.cuda.stream(s):
        call()
    s.synchronize()
    out0, lse0 = out.clone(), lse.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    _bits_equal(out, out0, "graph replay: out")
    _bits_equal(lse, lse0, "graph replay: lse")


def test_overlapping_output_is_rejected_before_launch():
    w = wl.decode(seq_lens=(40, 17), num_blocks=16)
    dw = DeviceWorkload(w)
    tq = w.q.shape[0]
    # out placed inside the pool: the attention would write it while the
    # cache write may still run
    out_in_pool = dw.pool.view(-1)[:tq * 8 * 128].view(tq, 8, 128)
    with pytest.raises(pagedattn.PagedAttnError) as e:
        dw.write_and_attend(out=out_in_pool)
    assert e.value.status == pagedattn.PA_ERR_INVALID_ARG
    # q inside the pool: read before the cache write is complete
    q_in_pool = dw.pool.view(-1)[:tq * 8 * 128].view(tq, 8, 128)
    with pytest.raises(pagedattn.PagedAttnError) as e:
        pagedattn.reshape_and_paged_attention(dw.key, dw.value, dw.slot_mapping, q_in_pool, dw.k_cache,
                                              dw.v_cache, dw.block_tables, dw.seq_lens, dw.query_start_loc,
                                              w.scale, dw.max_query_len, dw.max_seq_len,
                                              workspace=dw.workspace)
    assert e.value.status == pagedattn.PA_ERR_INVALID_ARG


def _rewrite_case(seed=5):
    """Decode workload with the whole cache written; new K/V for a mix of
    positions: a first page, a middle page (key 1300: the first tile of the
    sixth 256-key chunk), a last page, a block no table row holds, and a
    padding slot (-1)."""
    w = wl.decode()
    dw = DeviceWorkload(w)
    dw.write_cache()
    torch.cuda.synchronize()
    table = w.block_table
    used = {int(x) for b, L in enumerate(w.seq_lens.tolist()) for x in table[b, :wl.pages_needed(L)].tolist()}
    free = next(x for x in range(w.num_blocks) if x not in used)
    slots = [int(table[1, 0]) * 16 + 0, int(table[0, 1300 // 16]) * 16 + 1300 % 16,
             int(table[2, (4171 - 1) // 16]) * 16 + (4171 - 1) % 16, int(table[3, 0]) * 16 + 5,
             free * 16 + 3, -1]
    gen = torch.Generator().manual_seed(seed)
    key = wl.bf16_randn((len(slots), 2, 128), gen).cuda()
    value = wl.bf16_randn((len(slots), 2, 128), gen).cuda()
    return w, dw, key, value, torch.tensor(slots, dtype=torch.int64, device="cuda")


def test_rewrites_anywhere_in_the_tables_are_seen():
    """With few new tokens the attention copies the pages they do not touch
    before the write completes and waits only at the first tile holding one
    of them.  New values in first, middle and last pages must all be seen:
    the result equals the write followed by a separate attention call, and
    differs from the attention over the old cache."""
    w, dw, key, value, slots = _rewrite_case()
    out_old, lse_old = dw.attention()
    out, lse = dw.write_and_attend(key=key, value=value, slot_mapping=slots)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    w2, ref, key2, value2, slots2 = _rewrite_case()
    pagedattn.reshape_and_cache(key2, value2, ref.k_cache, ref.v_cache, slots2)
    out_r, lse_r = ref.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    _bits_equal(dw.pool, ref.pool, "rewrites: pool")
    _bits_equal(out, out_r, "rewrites: out vs two calls")
    _bits_equal(lse, lse_r, "rewrites: lse vs two calls")
    changed = (lse.view(torch.int32) != lse_old.view(torch.int32)).any(dim=1).cpu().tolist()
    print(f"requests whose lse moved: {changed}")
    assert changed == [True, True, True, True]


def test_write_outside_the_batch_leaves_attention_unchanged():
    """New tokens only in a block no table row holds (and padding): no tile
    of the attention waits for the write, the attention equals the one over
    the old cache, and the write still lands."""
    w, dw, key, value, slots = _rewrite_case()
    out_old, lse_old = dw.attention()
    sl = slots.clone()
    sl[:4] = -1
    out, lse = dw.write_and_attend(key=key, value=value, slot_mapping=sl)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    _bits_equal(out, out_old, "write outside the batch: out")
    _bits_equal(lse, lse_old, "write outside the batch: lse")
    free_slot = int(sl[4])
    got = dw.k_cache[free_slot // 16, free_slot % 16]
    _bits_equal(got, key[4], "write outside the batch: the written K row")

"""K1 (pa_reshape_and_cache) against the oracle's scatter: bit-exact pools.

Written slots must hold the input bits; every other slot must keep the NaN
sentinel ("ReshapeAndCache->PagedAttention composition at real dims", review
rework: slots derived from the table).  The >4 GB pool exercises 64-bit
offsets ("stabilize direct paged CK attention for bitwise R/R", Changes:
64-bit global addressing)."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import pa_oracle
from paged_kv_cache_178_gb300 import pagedattn
from paged_kv_cache_178_gb300 import workloads as wl
from paged_kv_cache_178_gb300.device import DeviceWorkload
from tests.helpers import bits, compact_blocks, oracle_pool

pytestmark = pytest.mark.gpu


def _pool_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).ravel()


@pytest.mark.parametrize("make", [wl.composition, wl.decode, lambda: wl.decode(reversed_pages=True),
                                  lambda: wl.long_prefill(4096)])
def test_scatter_bit_exact(make):
    w = make()
    dw = DeviceWorkload(w, with_workspace=False)
    dw.write_cache()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    ref = oracle_pool(w)
    got = _pool_bits(dw.pool)
    assert got.size == ref.storage.size
    mism = int(np.count_nonzero(got != ref.storage))
    print(f"{w.name}: mismatch_count={mism} of {got.size}")
    assert mism == 0


def test_scatter_over_4gb_pool():
    w = wl.suffix(128)
    dw = DeviceWorkload(w, with_workspace=False)
    assert dw.pool.numel() * 2 > 4 * 2**30
    dw.write_cache()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    wc, remap = compact_blocks(w)
    ref = oracle_pool(wc)
    used = torch.tensor(sorted(remap), dtype=torch.int64, device=dw.pool.device)
    assert int(used[-1]) == w.num_blocks - 1
    got = _pool_bits(dw.pool.index_select(0, used))
    assert np.array_equal(got, ref.storage)
    untouched = sorted(set(range(0, w.num_blocks, 997)) - set(remap))[:50]
    blk = _pool_bits(dw.pool[torch.tensor(untouched, device=dw.pool.device)])
    assert np.all(blk == wl.SENTINEL_BITS)


def test_negative_slots_skipped_and_strided_inputs():
    """Padding tokens (slot < 0) are not written; key/value may be views of a
    fused QKV buffer whose padding is poisoned and must never be copied."""
    gen = torch.Generator().manual_seed(21)
    n, hq, hkv, dh, nb = 45, 8, 2, 128, 8
    qkv = wl.bf16_randn((n, (hq + 2 * hkv) * dh + 64), gen)
    qkv[:, -64:] = float("nan")
    key = qkv[:, hq * dh:(hq + hkv) * dh].view(n, hkv, dh)
    value = qkv[:, (hq + hkv) * dh:(hq + 2 * hkv) * dh].view(n, hkv, dh)
    slots = torch.randperm(nb * 16, generator=gen)[:n].to(torch.int64)
    slots[[0, 7, 44]] = -1
    w = wl.Workload(name="strided", num_q_heads=hq, num_kv_heads=hkv, head_dim=dh, num_blocks=nb,
                    layout="interleaved", q=qkv[:1, :hq * dh].view(1, hq, dh), key=key, value=value,
                    slot_mapping=slots, block_table=torch.zeros((1, 1), dtype=torch.int32),
                    seq_lens=torch.ones(1, dtype=torch.int32),
                    query_start_loc=torch.tensor([0, 1], dtype=torch.int32), scale=0.1)
    dw = DeviceWorkload(w, with_workspace=False)
    big = qkv.cuda()
    k_view = big[:, hq * dh:(hq + hkv) * dh].view(n, hkv, dh)
    v_view = big[:, (hq + hkv) * dh:(hq + 2 * hkv) * dh].view(n, hkv, dh)
    assert k_view.stride(0) == (hq + 2 * hkv) * dh + 64
    pagedattn.reshape_and_cache(k_view, v_view, dw.k_cache, dw.v_cache, dw.slot_mapping)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    ref = pa_oracle.HostPool(nb, hkv, dh, "interleaved")
    assert pa_oracle.reshape_and_cache(bits(key), bits(value), slots.numpy(), ref) == 0
    assert np.array_equal(_pool_bits(dw.pool), ref.storage)


def test_out_of_range_slot_reported_not_written():
    w = wl.composition()
    sm = w.slot_mapping.clone()
    sm[5] = w.num_blocks * 16          # one past the pool
    w2 = dataclasses.replace(w, slot_mapping=sm)
    dw = DeviceWorkload(w2, with_workspace=False)
    dw.write_cache()
    st, idx = pagedattn.check_errors()
    assert st == pagedattn.PA_ERR_BAD_METADATA and idx == 5
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)   # latch cleared
    sm_ok = sm.clone()
    sm_ok[5] = -1
    ref = pa_oracle.HostPool(w.num_blocks, 2, 256, "separate")
    pa_oracle.reshape_and_cache(bits(w.key), bits(w.value), sm_ok.numpy(), ref)
    assert np.array_equal(_pool_bits(dw.pool), ref.storage)

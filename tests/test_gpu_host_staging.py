"""Step inputs in pinned host memory: the library's staging kernel
(pa_copy_to_device) copies them to the device, and the attention kernels
write out and lse straight into pinned host memory.  The results are the
device-resident call's, bit for bit."""
import pytest
import torch

from paged_kv_cache_178_gb300 import pagedattn
from paged_kv_cache_178_gb300 import workloads as wl
from paged_kv_cache_178_gb300.device import DeviceWorkload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("src_ready", [False, True])
@pytest.mark.parametrize("nbytes", [16, 1000, 19524, 1 << 20, (1 << 20) + 7])
def test_copy_to_device_exact_bytes(nbytes, src_ready):
    gen = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=gen).pin_memory()
    dst = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
    pagedattn.copy_to_device(dst, src, src_ready=src_ready)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)
    # device to device as well
    dst2 = torch.zeros_like(dst)
    pagedattn.copy_to_device(dst2, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst2, dst)


def _bitwise(a, b, what):
    ai = a.contiguous().view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32)
    bi = b.contiguous().view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)
    mism = int((ai.cpu() != bi.cpu()).sum())
    print(f"{what}: mismatch_count={mism}")
    assert mism == 0


def test_host_staged_composed_call_equals_device_call():
    w = wl.decode()
    last = [int(x) - 1 for x in torch.cumsum(w.seq_lens, 0)]
    a = DeviceWorkload(w)   # both pools start from the same fill pattern
    b = DeviceWorkload(w)
    a.write_cache()
    b.write_cache()
    idx = torch.tensor(last)
    host = [w.key[idx].contiguous(), w.value[idx].contiguous(), w.slot_mapping[idx].contiguous(), w.q,
            w.block_table.contiguous(), w.seq_lens, w.query_start_loc]
    h = [t.pin_memory() for t in host]
    d = [torch.empty_like(t, device="cuda") for t in host]
    for dt, ht in zip(d, h):
        pagedattn.copy_to_device(dt, ht, src_ready=True)   # only the host writes h
    k, v, s, q, bt, sl, qsl = d
    h_out = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    h_lse = torch.full(w.q.shape[:2], float("nan"), dtype=torch.float32).pin_memory()
    pagedattn.reshape_and_paged_attention(k, v, s, q, a.k_cache, a.v_cache, bt, sl, qsl, w.scale, w.max_query_len,
                                          w.max_seq_len, out=h_out, lse=h_lse, workspace=a.workspace)
    torch.cuda.synchronize()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    dk, dv, ds = (t.cuda() for t in host[:3])
    o2, l2 = b.write_and_attend(key=dk, value=dv, slot_mapping=ds)
    torch.cuda.synchronize()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    _bitwise(h_out, o2, "out written to pinned host memory vs device")
    _bitwise(h_lse, l2, "lse written to pinned host memory vs device")
    # bit patterns: the fill of unwritten slots is a NaN pattern
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))

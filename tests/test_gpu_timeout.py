"""The timeout path of the one cross-CTA wait in split-KV attention, made to
run out on purpose on a small decode, with nothing in flight while it waits.
The wait belongs to the 128-row kernel's shared fold (the few-row decode
kernel never waits for another CTA: its last arrival folds alone), so the
decode runs in the 64-key canon, which takes the 128-row kernel.

"ROCm: harden compact peer-local KV prefill for Gemma-4", Required hardening:
waits are bounded and a failure after submit is reported, never retried.
With the limit at 0 the CTAs that would wait for the rest of their
(request, KV head) group give up at once: the call latches PA_ERR_TIMEOUT,
their share of the output columns stays unwritten, the kernel ends normally,
and after the workspace is zero-filled again the next call is bitwise the
reference."""
import pytest
import torch

from paged_kv_cache_178_gb300 import pagedattn
from paged_kv_cache_178_gb300 import workloads as wl
from paged_kv_cache_178_gb300.device import DeviceWorkload

pytestmark = pytest.mark.gpu


def test_fold_wait_timeout_is_reported_and_the_workspace_recovers():
    # 8 and 4 chunks of 256 keys per (request, KV head): 24 CTAs, every one
    # resident at once, so the last four arrivals of each group share the fold
    w = wl.decode(seq_lens=(2048, 1024), num_blocks=256)
    dw = DeviceWorkload(w)
    dw.write_cache()
    ref_out, ref_lse = dw.attention(kv_tile=64)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    info = pagedattn.last_launch_info()
    assert "split" in info and "rows-m128" in info, info
    o2 = torch.zeros_like(ref_out)
    l2 = torch.zeros_like(ref_lse)
    prev = pagedattn.set_fold_wait_limit_ns(0)
    try:
        dw.attention(out=o2, lse=l2, kv_tile=64)
        st, idx = pagedattn.check_errors()
    finally:
        assert pagedattn.set_fold_wait_limit_ns(prev) == 0
    print(f"limit 0: status={pagedattn.status_string(st)} index={idx:#x}")
    assert st == pagedattn.PA_ERR_TIMEOUT
    assert idx & 0xFF == 0xFF             # the fold's wait, not a barrier slot
    # the last arrival of each group does not wait: its quarter of the
    # columns is written, and bit for bit the reference
    q = w.head_dim // 4
    assert torch.equal(o2[:, :, 3 * q:].view(torch.int16), ref_out[:, :, 3 * q:].view(torch.int16))
    # the CTAs that gave up wrote nothing
    assert int(o2[:, :, :3 * q].view(torch.int16).abs().sum()) == 0
    # zero-fill the workspace again, as the header asks after a timeout
    dw.workspace.zero_()
    o3, l3 = dw.attention(kv_tile=64)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    assert torch.equal(o3.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(l3.view(torch.int32), ref_lse.view(torch.int32))

"""The allocation-free attention entry point against the regular one.

pa_paged_attention_noalloc exists for callers that cannot call cudaMalloc
(for instance code running while a CUDA graph is captured, or an engine whose
device memory belongs entirely to its own pool allocator): it takes no
workspace and uses a scratch array built into the library instead.  This
file is named to run last so that, if it fails, a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

from paged_kv_cache_178_gb300 import pagedattn
from paged_kv_cache_178_gb300 import workloads as wl
from paged_kv_cache_178_gb300.device import DeviceWorkload
from tests.helpers import LSE_RTOL, OUT_ATOL, lse_rel_err

pytestmark = pytest.mark.gpu


def test_noalloc_matches_regular_entry_point_twice():
    w = wl.decode()                    # split-KV decode: the path that needs scratch
    dw = DeviceWorkload(w)
    dw.write_cache()
    ref_out, ref_lse = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    assert pagedattn.workspace_size(w.num_seqs, 8, 2, 128, w.max_query_len, w.max_seq_len) > 0
    for call in range(2):              # the scratch keeps the previous call's contents
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = pagedattn.paged_attention_noalloc(dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                               dw.seq_lens, dw.query_start_loc, w.scale,
                                               w.max_query_len, w.max_seq_len, out, lse)
        assert st == pagedattn.PA_OK, pagedattn.status_string(st)
        assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
        err_o = float((out.float() - ref_out.float()).abs().max())
        err_l = lse_rel_err(lse.cpu().numpy(), ref_lse.cpu().numpy())
        mism = int((out.view(torch.int16) != ref_out.view(torch.int16)).sum()) + \
            int((lse.view(torch.int32) != ref_lse.view(torch.int32)).sum())
        print(f"no-alloc call {call}: out max_abs_diff={err_o} lse rel={err_l} mismatch_count={mism}")
        assert err_o <= OUT_ATOL and err_l <= LSE_RTOL
        # the same kernel on the same inputs: the same bits
        assert mism == 0


def test_noalloc_rejects_bounds_beyond_its_scratch():
    w = wl.decode(seq_lens=(513, 40, 16), num_blocks=128)
    dw = DeviceWorkload(w)
    dw.write_cache()
    big = 1 << 20                      # a bound whose scratch exceeds the built-in array
    assert pagedattn.workspace_size(w.num_seqs, 8, 2, 128, 1, big) > pagedattn.NOALLOC_SCRATCH_BYTES
    out = torch.zeros_like(dw.q)
    st = pagedattn.paged_attention_noalloc(dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.seq_lens,
                                           dw.query_start_loc, w.scale, 1, big, out)
    assert st == pagedattn.PA_ERR_WORKSPACE
    assert int(out.abs().sum()) == 0   # nothing was launched


def test_noalloc_in_the_64_key_canon_equals_regular():
    """The tile rides in the pool descriptor, so the allocation-free entry
    point runs the same canon: bit for bit the regular call's results."""
    w = wl.decode()
    dw = DeviceWorkload(w)
    dw.write_cache()
    ref_out, ref_lse = dw.attention(kv_tile=64)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    st = pagedattn.paged_attention_noalloc(dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.seq_lens,
                                           dw.query_start_loc, w.scale, w.max_query_len, w.max_seq_len, out, lse,
                                           kv_tile=64)
    assert st == pagedattn.PA_OK, pagedattn.status_string(st)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    assert "kv_tile=64" in pagedattn.last_launch_info()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))

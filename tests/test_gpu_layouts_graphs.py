"""Graph capture with a shrinking batch, an HND page layout and a fused-QKV
q stride.

- A decode step recorded once in a CUDA graph for a bound of four requests
  is replayed with 4, 3, 2 and 1 active requests. Inactive rows get
  seq_len 0, an empty query range and slot -1. Each replay's rows equal, bit
  for bit, an eager call on the compact batch ("fix(rocm): stabilize direct
  paged CK attention for bitwise R/R", Changes: graph identity; one query
  per row of metadata).
- A pool laid out head-major inside each page ([block][head][token][d]) is
  described by strides alone. It gives the same bits as the token-major
  pool.
- q taken from a fused QKV buffer (token stride 2.5x the q row, K and V
  columns poisoned with NaN) gives the same bits as a contiguous q.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_178_gb300 import pagedattn
from paged_kv_cache_178_gb300 import workloads as wl
from paged_kv_cache_178_gb300.device import DeviceWorkload, bf16_fill
from tests.helpers import LSE_RTOL, OUT_ATOL, lse_rel_err, oracle_attention

pytestmark = pytest.mark.gpu


def _same_bits(a: torch.Tensor, b: torch.Tensor, what: str):
    ai = a.contiguous().view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32)
    bi = b.contiguous().view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)
    mism = int((ai != bi).sum())
    print(f"{what}: mismatch_count={mism}")
    assert mism == 0


def test_graph_replay_with_shrinking_batch():
    w = wl.decode()
    lens = [int(x) for x in w.seq_lens]
    last = np.cumsum(lens) - 1
    keep = np.setdiff1d(np.arange(sum(lens)), last)
    dw = DeviceWorkload(w)
    dev = dw.q.device
    ik = torch.as_tensor(keep, device=dev)
    pagedattn.reshape_and_cache(dw.key[ik], dw.value[ik], dw.k_cache, dw.v_cache,
                                dw.slot_mapping[ik].contiguous())
    il = torch.as_tensor(last, device=dev)
    new_k, new_v = dw.key[il].contiguous(), dw.value[il].contiguous()
    all_slots = dw.slot_mapping[il].contiguous()
    # step buffers sized for the bound of four requests; the graph records
    # their addresses, the contents change between replays
    slots = all_slots.clone()
    seq_lens = dw.seq_lens.clone()
    qsl = dw.query_start_loc.clone()
    tables = dw.block_tables.clone()
    out = torch.zeros((4, 8, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((4, 8), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    call = pagedattn.prepare_reshape_and_paged_attention(
        new_k, new_v, slots, dw.q, dw.k_cache, dw.v_cache, tables, seq_lens, qsl, w.scale, 1, 7168, out, lse,
        dw.workspace, stream=s)
    pagedattn.init()
    with torch.cuda.stream(s):
        call()  # warm: attributes and tensor maps
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for n in (4, 3, 2, 1):
        with torch.no_grad():
            slots.copy_(torch.where(torch.arange(4, device=dev) < n, all_slots, torch.full_like(all_slots, -1)))
            seq_lens.copy_(torch.where(torch.arange(4, device=dev) < n, dw.seq_lens,
                                       torch.zeros_like(dw.seq_lens)))
            qsl.copy_(torch.tensor([min(b, n) for b in range(5)], dtype=torch.int32, device=dev))
            out.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
        o_ref, l_ref = pagedattn.paged_attention(
            dw.q[:n].contiguous(), dw.k_cache, dw.v_cache, dw.block_tables[:n].contiguous(),
            dw.seq_lens[:n].contiguous(), torch.arange(n + 1, dtype=torch.int32, device=dev), w.scale, 1, 7168,
            workspace=pagedattn.new_workspace(n, 8, 2, 128, 1, 7168, dev))
        assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
        _same_bits(out[:n], o_ref, f"graph replay with {n} active requests: out")
        _same_bits(lse[:n], l_ref, f"graph replay with {n} active requests: lse")
        if n < 4:
            assert int(out[n:].view(torch.int16).abs().sum()) == 0  # rows of no request: untouched
    ref_o, ref_l = oracle_attention(w)
    o = out[:1].float().cpu().numpy()
    assert float(np.max(np.abs(o - ref_o[:1]))) <= OUT_ATOL
    assert lse_rel_err(lse[:1].cpu().numpy(), ref_l[:1]) <= LSE_RTOL


def test_head_major_page_layout():
    """[block][head][token][d] inside each page: the same logical cache, other
    strides; attention bits equal the token-major pool's."""
    w = wl.decode(seq_lens=(7168, 513, 40), num_blocks=1024)
    ref = DeviceWorkload(w)
    ref.write_cache()
    out_r, lse_r = ref.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    dev = ref.q.device
    hnd = bf16_fill((w.num_blocks, 2, 2, 16, 128), wl.SENTINEL_BITS, dev)  # [block][K/V][head][token][d]
    k_cache = hnd[:, 0].permute(0, 2, 1, 3)  # [block][token][head][d] view
    v_cache = hnd[:, 1].permute(0, 2, 1, 3)
    assert k_cache.stride() == (2 * 2 * 16 * 128, 128, 16 * 128, 1)
    pagedattn.reshape_and_cache(ref.key, ref.value, k_cache, v_cache, ref.slot_mapping)
    out, lse = pagedattn.paged_attention(ref.q, k_cache, v_cache, ref.block_tables, ref.seq_lens,
                                         ref.query_start_loc, w.scale, w.max_query_len, w.max_seq_len,
                                         workspace=pagedattn.new_workspace(3, 8, 2, 128, 1, 7168, dev))
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    _same_bits(out, out_r, "head-major pool vs token-major pool: out")
    _same_bits(lse, lse_r, "head-major pool vs token-major pool: lse")


@pytest.mark.parametrize("qlen", [1, 64])
def test_fused_qkv_q_stride_with_poison(qlen):
    """q as the first Hq*Dh columns of a fused [T, (Hq + 2 Hkv) * Dh] buffer
    whose K and V columns hold NaN: nothing outside q's rows is read."""
    w = wl.suffix(qlen, num_blocks=2048, batch=2, seq_len=1500)
    dw = DeviceWorkload(w)
    dw.write_cache()
    out_r, lse_r = dw.attention()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    T = dw.q.shape[0]
    fused = bf16_fill((T, (8 + 2 * 2) * 128), 0x7FC0, dw.q.device)
    fused[:, : 8 * 128] = dw.q.reshape(T, 8 * 128)
    q = fused[:, : 8 * 128].view(T, 8, 128)
    assert q.stride(0) == 12 * 128
    out, lse = dw.attention(q=q)
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    _same_bits(out, out_r, f"fused-QKV q (q={qlen}): out")
    _same_bits(lse, lse_r, f"fused-QKV q (q={qlen}): lse")


def test_metadata_shared_across_layers_in_one_graph():
    """Two layers (two pools, two query sets) read one set of step metadata
    -- block tables, lengths, query starts -- with no copy per layer
    ("stabilize direct paged CK attention for bitwise R/R", Changes: share
    prepared attention metadata across layers without dense KV
    materialization).  Both prepared calls captured in one graph give each
    layer's eager bits."""
    w0 = wl.decode(seed=1790)
    rows = [w0.block_table[b, :wl.pages_needed(L)].tolist() for b, L in enumerate(w0.seq_lens.tolist())]
    w1 = wl.build("decode_second_layer", num_q_heads=8, num_kv_heads=2, head_dim=128,
                  seq_lens=w0.seq_lens.tolist(), query_lens=[1] * 4, num_blocks=w0.num_blocks, block_rows=rows,
                  layout=w0.layout, seed=1791)  # same lengths and tables, other K/V and q
    assert torch.equal(w0.block_table, w1.block_table) and not torch.equal(w0.q, w1.q)
    layers = [DeviceWorkload(w) for w in (w0, w1)]
    for dw in layers:
        dw.write_cache()
    meta = layers[0]
    dev = meta.q.device
    eager = [dw.attention(block_tables=meta.block_tables, seq_lens=meta.seq_lens,
                          query_start_loc=meta.query_start_loc) for dw in layers]
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    s = torch.cuda.Stream()
    outs = [torch.empty_like(o) for o, _ in eager]
    lses = [torch.empty_like(l_) for _, l_ in eager]
    ws = [pagedattn.new_workspace(4, 8, 2, 128, 1, 7168, dev) for _ in layers]
    calls = [pagedattn.prepare_paged_attention(dw.q, dw.k_cache, dw.v_cache, meta.block_tables, meta.seq_lens,
                                               meta.query_start_loc, dw.w.scale, 1, 7168, outs[i], lses[i], ws[i],
                                               stream=s)
             for i, dw in enumerate(layers)]
    pagedattn.init()
    with torch.cuda.stream(s):
        for c in calls:
            c()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in calls:
            c()
    for o in outs:
        o.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert pagedattn.check_errors() == (pagedattn.PA_OK, -1)
    for i in range(2):
        _same_bits(outs[i], eager[i][0], f"layer {i} in the shared-metadata graph: out")
        _same_bits(lses[i], eager[i][1], f"layer {i} in the shared-metadata graph: lse")

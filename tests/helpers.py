"""Shared test utilities: BF16 bit conversions and running the oracle on a
workload.  Nothing here calls the CUDA library."""
from __future__ import annotations

from typing import Dict, Optional, Sequence, Tuple

import numpy as np
import torch

from oracle import pa_oracle
from paged_kv_cache_178_gb300 import workloads as wl


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> numpy uint16 bit patterns (same shape)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def compact_blocks(w: wl.Workload) -> Tuple[wl.Workload, Dict[int, int]]:
    """Relabel the physical blocks a workload touches to 0..n-1 (table and
    slots remapped consistently).  Output is invariant under such a relabel
    (pinned in the oracle tests), so a >4 GB pool can be checked with a
    small host pool."""
    used = sorted({int(s) // wl.BLOCK_SIZE for s in w.slot_mapping.tolist() if s >= 0} |
                  {int(b) for row, L in zip(w.block_table.tolist(), w.seq_lens.tolist())
                   for b in row[: wl.pages_needed(L)]})
    remap = {b: i for i, b in enumerate(used)}
    bt = w.block_table.clone()
    for r in range(bt.shape[0]):
        for c in range(wl.pages_needed(int(w.seq_lens[r]))):
            bt[r, c] = remap[int(bt[r, c])]
    sm = w.slot_mapping.clone()
    for i, s in enumerate(sm.tolist()):
        if s >= 0:
            sm[i] = remap[s // wl.BLOCK_SIZE] * wl.BLOCK_SIZE + s % wl.BLOCK_SIZE
    import dataclasses
    return dataclasses.replace(w, block_table=bt, slot_mapping=sm, num_blocks=len(used)), remap


def oracle_pool(w: wl.Workload, fill_bits: int = wl.SENTINEL_BITS) -> pa_oracle.HostPool:
    pool = pa_oracle.HostPool(w.num_blocks, w.num_kv_heads, w.head_dim, w.layout, fill_bits)
    bad = pa_oracle.reshape_and_cache(bits(w.key), bits(w.value), w.slot_mapping.numpy(), pool)
    assert bad == 0
    return pool


def oracle_attention(w: wl.Workload, rows: Optional[Sequence[int]] = None,
                     pool: Optional[pa_oracle.HostPool] = None, num_threads: int = 0,
                     compact: bool = False):
    """Oracle out [R, Hq, Dh] / lse [R, Hq] (float64) for a workload whose
    cache is written from its own key/value/slot_mapping."""
    if compact:
        w, _ = compact_blocks(w)
    if pool is None:
        pool = oracle_pool(w)
    return pa_oracle.paged_attention(bits(w.q), pool, w.block_table.numpy(), w.seq_lens.numpy(),
                                     w.query_start_loc.numpy(), w.scale, rows=rows,
                                     num_threads=num_threads)


def lse_rel_err(a: np.ndarray, b: np.ndarray) -> float:
    """|a-b| / max(|b|, 1): a causal row 0 has lse = s0, which may be near 0."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b) / np.maximum(np.abs(b), 1.0)))


OUT_ATOL = 2e-2      # attention output, max-abs vs the fp64 oracle (N(0,1) inputs)
LSE_RTOL = 1e-3      # LSE relative error vs the fp64 oracle

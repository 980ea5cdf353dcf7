"""Device-resident copy of a workload: the BF16 pool (K and V views), the
query, the new K/V tokens and the metadata, plus thin calls into the library.
Used by the tests, the smoke check and the benchmark."""
from __future__ import annotations

from typing import Optional

import torch

from . import pagedattn
from .workloads import BLOCK_SIZE, SENTINEL_BITS, Workload


def bf16_fill(shape, bits: int, device) -> torch.Tensor:
    v = bits - (1 << 16) if bits >= (1 << 15) else bits
    return torch.full(shape, v, dtype=torch.int16, device=device).view(torch.bfloat16)


class DeviceWorkload:
    def __init__(self, w: Workload, device: str = "cuda", fill_bits: Optional[int] = SENTINEL_BITS,
                 with_workspace: bool = True):
        self.w = w
        self.device = torch.device(device)
        nb, hkv, dh = w.num_blocks, w.num_kv_heads, w.head_dim
        if w.layout == "interleaved":
            shape = (nb, 2, BLOCK_SIZE, hkv, dh)
        else:
            shape = (2, nb, BLOCK_SIZE, hkv, dh)
        if fill_bits is None:
            self.pool = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
        else:
            self.pool = bf16_fill(shape, fill_bits, self.device)
        if w.layout == "interleaved":
            self.k_cache, self.v_cache = self.pool[:, 0], self.pool[:, 1]
        else:
            self.k_cache, self.v_cache = self.pool[0], self.pool[1]
        to = dict(device=self.device)
        self.q = w.q.to(**to)
        self.key = w.key.to(**to)
        self.value = w.value.to(**to)
        self.slot_mapping = w.slot_mapping.to(**to)
        self.block_tables = w.block_table.to(**to)
        self.seq_lens = w.seq_lens.to(**to)
        self.query_start_loc = w.query_start_loc.to(**to)
        self.max_query_len = w.max_query_len
        self.max_seq_len = w.max_seq_len
        self.workspace = None
        if with_workspace:
            self.workspace = pagedattn.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads, dh,
                                                     self.max_query_len, self.max_seq_len, self.device)

    def write_cache(self, stream=None) -> None:
        pagedattn.reshape_and_cache(self.key, self.value, self.k_cache, self.v_cache,
                                    self.slot_mapping, stream=stream)

    def attention(self, out=None, lse=None, want_lse=True, max_query_len=None, max_seq_len=None,
                  block_tables=None, q=None, seq_lens=None, query_start_loc=None, workspace=None,
                  stream=None, kv_tile=0):
        mq = self.max_query_len if max_query_len is None else max_query_len
        ms = self.max_seq_len if max_seq_len is None else max_seq_len
        if workspace is not None:
            ws = workspace
        elif max_query_len is None and max_seq_len is None:
            ws = self.workspace
        else:
            ws = None  # the binding allocates a zeroed workspace for other bounds
        return pagedattn.paged_attention(
            self.q if q is None else q, self.k_cache, self.v_cache,
            self.block_tables if block_tables is None else block_tables,
            self.seq_lens if seq_lens is None else seq_lens,
            self.query_start_loc if query_start_loc is None else query_start_loc,
            self.w.scale, mq, ms, out=out, lse=lse, want_lse=want_lse, workspace=ws, stream=stream,
            kv_tile=kv_tile)

    def write_and_attend(self, key=None, value=None, slot_mapping=None, out=None, lse=None, want_lse=True,
                         stream=None, kv_tile=0):
        """The cache write of (key, value, slot_mapping) -- by default every
        token of the workload -- and the attention, in one library call."""
        return pagedattn.reshape_and_paged_attention(
            self.key if key is None else key, self.value if value is None else value,
            self.slot_mapping if slot_mapping is None else slot_mapping, self.q, self.k_cache, self.v_cache,
            self.block_tables, self.seq_lens, self.query_start_loc, self.w.scale, self.max_query_len,
            self.max_seq_len, out=out, lse=lse, want_lse=want_lse, workspace=self.workspace, stream=stream,
            kv_tile=kv_tile)

    def share_cache_with(self, other: "DeviceWorkload") -> None:
        """Point this workload at another's pool (same geometry)."""
        self.pool, self.k_cache, self.v_cache = other.pool, other.k_cache, other.v_cache

"""Seeded synthetic inputs for the paged KV-cache composition.

This module only *builds inputs*: random BF16 tensors, shuffled block tables,
sequence lengths and the slot mapping a model layer would hand to
ReshapeAndCache.  It holds none of the arithmetic under test (no scatter, no
gather, no attention), so both the CUDA path and the CPU oracle can draw their
inputs from it without sharing any computation.

Workload shapes follow the pages:
  * composition case: Dh=256, Hq=8, Hkv=2, page 16, table {3,1,2,0}, 20 tokens,
    slots derived from the table ("ReshapeAndCache->PagedAttention composition
    at real dims", What changed and the review rework);
  * decode / suffix / long-prefill shapes and the separate, interleaved and
    >2 GB pool layouts with reversed physical pages ("stabilize direct paged CK
    attention for bitwise R/R", Operator benchmarks and Additional checks);
  * the Hq=16, Hkv=2, d=512 wide-head prefill at ~3k/~8k/~11k/~18k tokens
    ("harden compact peer-local KV prefill for Gemma-4", Scope and Gates).
No public dataset is involved: values are N(0,1) rounded to BF16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

BLOCK_SIZE = 16
# Table columns past a request's last page are never read; they hold this
# value so that a read of one would be out of range and detectable.
TABLE_POISON = 2**31 - 1
# Quiet-NaN BF16 bit pattern used to pre-fill pools: any read of a slot that
# nothing wrote turns the result into NaN.
SENTINEL_BITS = 0x7FC1


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    layout: str                    # "interleaved" or "separate"
    q: torch.Tensor                # [Tq, Hq, Dh] bf16 (CPU)
    key: torch.Tensor              # [N, Hkv, Dh] bf16: tokens to write
    value: torch.Tensor            # [N, Hkv, Dh] bf16
    slot_mapping: torch.Tensor     # [N] int64
    block_table: torch.Tensor      # [B, max_blocks] int32
    seq_lens: torch.Tensor         # [B] int32 (includes the new tokens)
    query_start_loc: torch.Tensor  # [B+1] int32
    scale: float
    block_size: int = BLOCK_SIZE

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def max_query_len(self) -> int:
        ql = self.query_start_loc[1:] - self.query_start_loc[:-1]
        return int(ql.max().item()) if ql.numel() else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0

    @property
    def num_q_tokens(self) -> int:
        return int(self.q.shape[0])


def bf16_randn(shape: Sequence[int], gen: torch.Generator) -> torch.Tensor:
    """N(0,1) drawn in fp32 from a seeded CPU generator, rounded to BF16."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def softmax_scale(head_dim: int) -> float:
    """1/sqrt(Dh) rounded to fp32 (the value both sides receive)."""
    return float(torch.tensor(1.0 / math.sqrt(head_dim), dtype=torch.float32).item())


def pages_needed(seq_len: int) -> int:
    return (seq_len + BLOCK_SIZE - 1) // BLOCK_SIZE


def table_slots(table_row: Sequence[int], positions: Sequence[int]) -> List[int]:
    """Slot handed to the cache write for logical positions, derived from the
    request's own block table (the mapping the composition review asks for)."""
    return [int(table_row[p // BLOCK_SIZE]) * BLOCK_SIZE + p % BLOCK_SIZE for p in positions]


def _table_tensor(rows: List[List[int]], max_blocks: int) -> torch.Tensor:
    t = torch.full((len(rows), max_blocks), TABLE_POISON, dtype=torch.int32)
    for b, r in enumerate(rows):
        if r:
            t[b, : len(r)] = torch.tensor(r, dtype=torch.int32)
    return t


def build(name: str, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
          seq_lens: Sequence[int], query_lens: Sequence[int], num_blocks: int,
          block_rows: List[List[int]], layout: str, seed: int,
          write_all_tokens: bool = True, max_blocks: Optional[int] = None,
          scale: Optional[float] = None) -> Workload:
    """Assemble a workload.  Request b owns physical pages block_rows[b] (its
    table row, in logical order).  K/V for every cached token of each request
    is drawn and handed to the cache write with table-derived slots; q holds
    the last query_lens[b] positions of each request."""
    gen = torch.Generator().manual_seed(seed)
    B = len(seq_lens)
    assert len(query_lens) == B and len(block_rows) == B
    for L, qn, row in zip(seq_lens, query_lens, block_rows):
        assert 0 <= qn <= L and len(row) >= pages_needed(L)
    if max_blocks is None:
        max_blocks = max([len(r) for r in block_rows] + [1])
    tq = int(sum(query_lens))
    q = bf16_randn((tq, num_q_heads, head_dim), gen)
    n_kv = int(sum(seq_lens)) if write_all_tokens else tq
    key = bf16_randn((n_kv, num_kv_heads, head_dim), gen)
    value = bf16_randn((n_kv, num_kv_heads, head_dim), gen)
    slots: List[int] = []
    for L, qn, row in zip(seq_lens, query_lens, block_rows):
        first = 0 if write_all_tokens else L - qn
        slots += table_slots(row, range(first, L))
    qsl = [0]
    for qn in query_lens:
        qsl.append(qsl[-1] + int(qn))
    return Workload(
        name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, num_blocks=num_blocks, layout=layout, q=q, key=key,
        value=value, slot_mapping=torch.tensor(slots, dtype=torch.int64),
        block_table=_table_tensor(block_rows, max_blocks),
        seq_lens=torch.tensor(list(seq_lens), dtype=torch.int32),
        query_start_loc=torch.tensor(qsl, dtype=torch.int32),
        scale=softmax_scale(head_dim) if scale is None else scale)


def _split_pages(pages: List[int], seq_lens: Sequence[int]) -> List[List[int]]:
    rows, at = [], 0
    for L in seq_lens:
        n = pages_needed(L)
        rows.append(pages[at: at + n])
        at += n
    return rows


# --------------------------------------------------------------------------
# The five workloads.
# --------------------------------------------------------------------------

def composition(table=(3, 1, 2, 0), seed: int = 1781) -> Workload:
    """One request, 20 tokens of causal prefill, Dh=256, Hq=8, Hkv=2, page 16,
    a pool of 4 physical blocks and the shuffled table {3,1,2,0}."""
    return build("composition_dh256_t20", num_q_heads=8, num_kv_heads=2, head_dim=256,
                 seq_lens=[20], query_lens=[20], num_blocks=4,
                 block_rows=[list(table)], layout="separate", seed=seed)


DECODE_LENS = (7168, 7168, 4171, 513)


def decode(reversed_pages: bool = False, seed: int = 1782, num_blocks: int = 2048,
           seq_lens: Sequence[int] = DECODE_LENS) -> Workload:
    """B=4 single-query decode over KV lengths {7168,7168,4171,513} (partial
    tail pages), Hq=8, Hkv=2, Dh=128, interleaved pool of 2048 blocks.  Pages
    come from a seeded permutation, or run backwards from the last block."""
    gen = torch.Generator().manual_seed(seed + 7)
    total = sum(pages_needed(L) for L in seq_lens)
    if reversed_pages:
        pages = list(range(num_blocks - 1, num_blocks - 1 - total, -1))
    else:
        pages = torch.randperm(num_blocks, generator=gen)[:total].tolist()
    tag = "reversed" if reversed_pages else "shuffled"
    return build(f"decode_b{len(seq_lens)}_dh128_{tag}", num_q_heads=8, num_kv_heads=2,
                 head_dim=128, seq_lens=list(seq_lens), query_lens=[1] * len(seq_lens),
                 num_blocks=num_blocks, block_rows=_split_pages(pages, seq_lens),
                 layout="interleaved", seed=seed)


def suffix(query_len: int = 128, seed: int = 1783, num_blocks: int = 300_000,
           batch: int = 4, seq_len: int = 7168) -> Workload:
    """B=4 suffix/chunked prefill: query_len new tokens at the end of a
    7168-token sequence, Dh=128, interleaved pool of 300k blocks (>4 GB);
    request 0's last page sits in the pool's last block so element offsets
    pass 2**31."""
    gen = torch.Generator().manual_seed(seed + 7)
    lens = [seq_len] * batch
    total = sum(pages_needed(L) for L in lens)
    pages = torch.randperm(num_blocks - 1, generator=gen)[:total].tolist()
    rows = _split_pages(pages, lens)
    rows[0][-1] = num_blocks - 1
    return build(f"suffix_b{batch}_q{query_len}_kv{seq_len}_dh128", num_q_heads=8,
                 num_kv_heads=2, head_dim=128, seq_lens=lens, query_lens=[query_len] * batch,
                 num_blocks=num_blocks, block_rows=rows, layout="interleaved", seed=seed)


def long_prefill(seq_len: int = 4096, seed: int = 1784, pool_factor: int = 2) -> Workload:
    """B=1 causal prefill, Q=KV=4096, Dh=128, shuffled table in a pool twice
    the needed size."""
    gen = torch.Generator().manual_seed(seed + 7)
    n = pages_needed(seq_len)
    nb = pool_factor * n
    pages = torch.randperm(nb, generator=gen)[:n].tolist()
    return build(f"prefill_b1_q{seq_len}_dh128", num_q_heads=8, num_kv_heads=2, head_dim=128,
                 seq_lens=[seq_len], query_lens=[seq_len], num_blocks=nb, block_rows=[pages],
                 layout="interleaved", seed=seed)


WIDE_LENS = (3072, 8192, 11264, 18432)


def wide_head(seq_len: int = 3072, seed: int = 1785) -> Workload:
    """B=1 causal prefill, Hq=16, Hkv=2, Dh=512, shuffled table in a pool of
    2*ceil(L/16) blocks."""
    gen = torch.Generator().manual_seed(seed + 7)
    n = pages_needed(seq_len)
    nb = 2 * n
    pages = torch.randperm(nb, generator=gen)[:n].tolist()
    return build(f"wide_b1_q{seq_len}_dh512", num_q_heads=16, num_kv_heads=2, head_dim=512,
                 seq_lens=[seq_len], query_lens=[seq_len], num_blocks=nb, block_rows=[pages],
                 layout="interleaved", seed=seed + seq_len)


def decode_batch_from_prefill(w: Workload, rows: Optional[Sequence[int]] = None) -> Workload:
    """The decode view of a single-request prefill: one request per prefill
    row p, seq_len p+1, the same table and q = row p.  Nothing is written:
    the cache already holds the prefill's K/V."""
    assert w.num_seqs == 1
    L = int(w.seq_lens[0])
    qoff = int(w.query_start_loc[0])
    qn = int(w.query_start_loc[1]) - qoff
    rows = list(range(qn)) if rows is None else list(rows)
    pos = [L - qn + r for r in rows]
    q = w.q[[qoff + r for r in rows]].clone()
    B = len(rows)
    return Workload(
        name=w.name + "_as_decode", num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, num_blocks=w.num_blocks, layout=w.layout, q=q,
        key=w.key[:0], value=w.value[:0], slot_mapping=w.slot_mapping[:0],
        block_table=w.block_table[0:1].expand(B, -1).contiguous(),
        seq_lens=torch.tensor([p + 1 for p in pos], dtype=torch.int32),
        query_start_loc=torch.arange(B + 1, dtype=torch.int32), scale=w.scale)


def pool_shape(w: Workload):
    if w.layout == "interleaved":
        return (w.num_blocks, 2, BLOCK_SIZE, w.num_kv_heads, w.head_dim)
    return (w.num_blocks, BLOCK_SIZE, w.num_kv_heads, w.head_dim)

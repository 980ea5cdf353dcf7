"""Python face of the CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
module.  It wraps the plain fp64 C oracle (pa_oracle.c, built with gcc) and
works on numpy arrays of BF16 *bit patterns* (uint16), so nothing here
depends on the CUDA library or on torch's BF16 arithmetic.

  reshape_and_cache  -- slot-mapped bit copy into a host pool
                        ("ReshapeAndCache->PagedAttention composition at real
                        dims", What changed and review rework)
  paged_attention    -- fp64 GQA causal softmax attention through the block
                        table ("stabilize direct paged CK attention for bitwise
                        R/R", Additional checks: full/suffix execution,
                        causal/LSE vs decode)
  gather_kv_head     -- the block-table-selected pages of one KV head packed
                        in request order, with compact table and offsets
                        ("ROCm: harden compact peer-local KV prefill for
                        Gemma-4", Scope and Required hardening)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpaoracle.so")
_lock = threading.Lock()
_lib = None

BLOCK_SIZE = 16


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (fp64, OpenMP, no fast-math, no FMA
    contraction).  Returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared",
               "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            lib.pao_reshape_and_cache.restype = i64
            lib.pao_reshape_and_cache.argtypes = [p, i64, p, i64, i64, i32, i32, p, p, i64, i64,
                                                  i64, i64, p]
            lib.pao_paged_attention.restype = i64
            lib.pao_paged_attention.argtypes = [p, i64, i32, p, p, i64, i64, i64, i64, i32, i32,
                                                p, i32, p, p, i32, ctypes.c_float, p, i64, p, p,
                                                i32]
            lib.pao_max_threads.restype = i32
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().pao_max_threads())


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class HostPool:
    """A K view and a V view over host uint16 storage with one shared set of
    element strides (block, token-in-block, head); Dh is contiguous.
    'interleaved' stores [NB, 2, 16, Hkv, Dh] (K at [:,0], V at [:,1]);
    'separate' stores two [NB, 16, Hkv, Dh] arrays."""

    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int, layout: str,
                 fill_bits: int = 0x7FC1):
        self.num_blocks, self.num_kv_heads, self.head_dim, self.layout = (
            num_blocks, num_kv_heads, head_dim, layout)
        per_block = BLOCK_SIZE * num_kv_heads * head_dim
        if layout == "interleaved":
            self.storage = np.full(num_blocks * 2 * per_block, fill_bits, dtype=np.uint16)
            self.k_offset, self.v_offset = 0, per_block
            self.block_stride = 2 * per_block
        elif layout == "separate":
            self.storage = np.full(num_blocks * 2 * per_block, fill_bits, dtype=np.uint16)
            self.k_offset, self.v_offset = 0, num_blocks * per_block
            self.block_stride = per_block
        else:
            raise ValueError(layout)
        self.token_stride = num_kv_heads * head_dim
        self.head_stride = head_dim

    def k_ptr(self) -> int:
        return _ptr(self.storage) + 2 * self.k_offset

    def v_ptr(self) -> int:
        return _ptr(self.storage) + 2 * self.v_offset

    def view(self, which: str) -> np.ndarray:
        """[NB, 16, Hkv, Dh] numpy view of the K or V cache."""
        off = self.k_offset if which == "k" else self.v_offset
        s = self.storage.itemsize
        return np.lib.stride_tricks.as_strided(
            self.storage[off:], shape=(self.num_blocks, BLOCK_SIZE, self.num_kv_heads,
                                       self.head_dim),
            strides=(self.block_stride * s, self.token_stride * s, self.head_stride * s, s),
            writeable=True)


def reshape_and_cache(key_bits: np.ndarray, value_bits: np.ndarray, slots: np.ndarray,
                      pool: HostPool) -> int:
    """Scatter [N, Hkv, Dh] K/V bit patterns into the pool at slots[i].
    Returns 0, or 1 + the first token whose slot is past the pool."""
    key_bits = np.ascontiguousarray(key_bits, dtype=np.uint16)
    value_bits = np.ascontiguousarray(value_bits, dtype=np.uint16)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    n, hkv, dh = key_bits.shape
    assert hkv == pool.num_kv_heads and dh == pool.head_dim
    return int(_load().pao_reshape_and_cache(
        _ptr(key_bits), hkv * dh, _ptr(value_bits), hkv * dh, n, hkv, dh, pool.k_ptr(),
        pool.v_ptr(), pool.num_blocks, pool.block_stride, pool.token_stride, pool.head_stride,
        _ptr(slots)))


def paged_attention(q_bits: np.ndarray, pool: HostPool, block_tables: np.ndarray,
                    seq_lens: np.ndarray, query_start_loc: np.ndarray, scale: float,
                    rows: Optional[Sequence[int]] = None, num_threads: int = 0
                    ) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 attention for query tokens `rows` (default: all).  q_bits is
    [Tq, Hq, Dh] uint16.  Returns out [R, Hq, Dh] and lse [R, Hq] (float64)."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    tq, hq, dh = q_bits.shape
    assert dh == pool.head_dim and hq % pool.num_kv_heads == 0
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    if rows is None:
        rows_arr = None
        nrows = tq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    out = np.empty((nrows, hq, dh), dtype=np.float64)
    lse = np.empty((nrows, hq), dtype=np.float64)
    _load().pao_paged_attention(
        _ptr(q_bits), hq * dh, hq, pool.k_ptr(), pool.v_ptr(), pool.num_blocks,
        pool.block_stride, pool.token_stride, pool.head_stride, pool.num_kv_heads, dh,
        _ptr(bt), bt.shape[1], _ptr(sl), _ptr(qsl), sl.size, float(scale),
        0 if rows_arr is None else _ptr(rows_arr), nrows, _ptr(out), _ptr(lse),
        int(num_threads))
    return out, lse


NAN_BITS = 0x7FC0  # BF16 quiet NaN written for a page whose block id is bad


class Gathered:
    """Result of gather_kv_head: packed K/V [total, 16, Dh] bit patterns (None
    when over budget), compact table [B, max_blocks] (None when over budget),
    offsets [B + 1], the requests with bad metadata (ascending) and, when
    over budget, the pages needed (else None)."""

    def __init__(self, packed_k, packed_v, compact_tables, offsets, bad_requests, budget_needed):
        self.packed_k, self.packed_v = packed_k, packed_v
        self.compact_tables, self.offsets = compact_tables, offsets
        self.bad_requests, self.budget_needed = bad_requests, budget_needed


def gather_kv_head(pool: HostPool, kv_head: int, block_tables: np.ndarray, seq_lens: np.ndarray,
                   capacity_pages: int) -> Gathered:
    """Pack the pages that request b selects -- block_tables[b][p] for
    p < ceil(L_b / 16) -- of head kv_head, request after request, page after
    page ("ROCm: harden compact peer-local KV prefill for Gemma-4", Scope:
    compact active block-table-selected K/V head).  Hardening, same source:
    a length outside [0, 16 * max_blocks] selects no page and marks its
    request bad; a block id outside the pool gives a NaN page and marks its
    request bad; more pages than capacity_pages writes the offsets only and
    reports the pages needed."""
    bt = np.asarray(block_tables, dtype=np.int64)
    lens = [int(x) for x in np.asarray(seq_lens).reshape(-1)]
    num_seqs, max_blocks = bt.shape
    bad = set()
    pages = []
    for b, L in enumerate(lens):
        if L < 0 or L > BLOCK_SIZE * max_blocks:
            bad.add(b)
            pages.append(0)
        else:
            pages.append(-(-L // BLOCK_SIZE))
    offsets = np.zeros(num_seqs + 1, dtype=np.int64)
    for b in range(num_seqs):
        offsets[b + 1] = offsets[b] + pages[b]
    total = int(offsets[num_seqs])
    if total > capacity_pages:
        return Gathered(None, None, None, offsets, sorted(bad), total)
    compact = np.full((num_seqs, max_blocks), -1, dtype=np.int64)
    dh = pool.head_dim
    packed_k = np.zeros((total, BLOCK_SIZE, dh), dtype=np.uint16)
    packed_v = np.zeros((total, BLOCK_SIZE, dh), dtype=np.uint16)
    kview, vview = pool.view("k"), pool.view("v")
    for b in range(num_seqs):
        for p in range(pages[b]):
            c = int(offsets[b]) + p
            compact[b, p] = c
            blk = int(bt[b, p])
            if 0 <= blk < pool.num_blocks:
                packed_k[c] = kview[blk, :, kv_head, :]
                packed_v[c] = vview[blk, :, kv_head, :]
            else:
                bad.add(b)
                packed_k[c] = NAN_BITS
                packed_v[c] = NAN_BITS
    return Gathered(packed_k, packed_v, compact, offsets, sorted(bad), None)


def pool_from_packed(packed_k: np.ndarray, packed_v: np.ndarray, capacity_pages: int) -> HostPool:
    """A one-head HostPool ('separate' layout) whose first pages hold the
    packed K/V bit patterns; pages past them keep the pool's NaN fill."""
    total, bs, dh = packed_k.shape
    pool = HostPool(max(capacity_pages, 1), 1, dh, "separate")
    pool.view("k")[:total, :, 0, :] = packed_k
    pool.view("v")[:total, :, 0, :] = packed_v
    return pool

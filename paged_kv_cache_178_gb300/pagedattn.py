"""Python binding of libpagedattn.so (ctypes).

Argument marshalling only: torch tensors supply device pointers, strides and
the current CUDA stream; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the library is missing or a call
fails, an exception is raised.

    reshape_and_cache(key, value, k_cache, v_cache, slot_mapping)
    paged_attention(q, k_cache, v_cache, block_tables, seq_lens,
                    query_start_loc, scale, max_query_len, max_seq_len)
    prepare_reshape_and_cache(...) / prepare_paged_attention(...)
        the same calls validated once, re-issued by calling the result

k_cache / v_cache are [num_blocks, 16, Hkv, Dh] BF16 views (they may be
slices of one interleaved [num_blocks, 2, 16, Hkv, Dh] pool) with identical
strides and a contiguous head dimension.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedattn.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_BAD_METADATA = 4
PA_ERR_TIMEOUT = 5
PA_ERR_CUDA = 6

EXPORTED = ("pa_init", "pa_reshape_and_cache", "pa_paged_attention_workspace_size",
            "pa_paged_attention", "pa_paged_attention_noalloc", "pa_reshape_and_paged_attention",
            "pa_gather_kv_head", "pa_check_errors", "pa_set_fold_wait_limit_ns",
            "pa_copy_to_device", "pa_status_string", "pa_last_launch_info")
NOALLOC_SCRATCH_BYTES = 8 << 20


class PaKvCache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_blocks", ctypes.c_int64),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("kv_tile", ctypes.c_int32),
                ("block_stride", ctypes.c_int64), ("token_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64)]


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m paged_kv_cache_178_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        lib.pa_init.restype = i32
        lib.pa_init.argtypes = []
        lib.pa_reshape_and_cache.restype = i32
        lib.pa_reshape_and_cache.argtypes = [vp, i64, vp, i64, i64, ctypes.POINTER(PaKvCache), vp, vp]
        lib.pa_paged_attention_workspace_size.restype = sz
        lib.pa_paged_attention_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.pa_paged_attention.restype = i32
        lib.pa_paged_attention.argtypes = [vp, i64, i64, i32, ctypes.POINTER(PaKvCache), vp, i32, vp,
                                           vp, i32, i32, i32, ctypes.c_float, vp, vp, vp, sz, vp]
        lib.pa_paged_attention_noalloc.restype = i32
        lib.pa_paged_attention_noalloc.argtypes = [vp, i64, i64, i32, ctypes.POINTER(PaKvCache), vp, i32,
                                                   vp, vp, i32, i32, i32, ctypes.c_float, vp, vp, vp]
        lib.pa_reshape_and_paged_attention.restype = i32
        lib.pa_reshape_and_paged_attention.argtypes = [
            vp, i64, vp, i64, i64, vp, vp, i64, i64, i32, ctypes.POINTER(PaKvCache), vp, i32, vp, vp, i32,
            i32, i32, ctypes.c_float, vp, vp, vp, sz, vp]
        lib.pa_gather_kv_head.restype = i32
        lib.pa_gather_kv_head.argtypes = [ctypes.POINTER(PaKvCache), i32, vp, i32, vp, i32, vp, vp, i64, vp,
                                          vp, vp]
        lib.pa_check_errors.restype = i32
        lib.pa_check_errors.argtypes = [vp, ctypes.POINTER(i64)]
        lib.pa_set_fold_wait_limit_ns.restype = ctypes.c_uint64
        lib.pa_set_fold_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.pa_copy_to_device.restype = i32
        lib.pa_copy_to_device.argtypes = [vp, vp, sz, i32, vp]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_status_string.argtypes = [i32]
        lib.pa_last_launch_info.restype = None
        lib.pa_last_launch_info.argtypes = [ctypes.c_char_p, sz]
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != PA_OK:
        raise PagedAttnError(status, what)


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def init() -> None:
    _check(load().pa_init(), "pa_init")


def set_fold_wait_limit_ns(limit_ns: int) -> int:
    """Time limit of the split-KV fold's cross-CTA wait (default 2 s); returns
    the previous limit.  0 makes the waiting CTAs give up at once (a test of
    the timeout path)."""
    return int(load().pa_set_fold_wait_limit_ns(int(limit_ns)))


def last_launch_info() -> str:
    buf = ctypes.create_string_buffer(256)
    load().pa_last_launch_info(buf, 256)
    return buf.value.decode()


def cache_struct(k_cache: torch.Tensor, v_cache: torch.Tensor, kv_tile: int = 0) -> PaKvCache:
    """Describe a [num_blocks, 16, Hkv, Dh] K/V pair for the C ABI.  kv_tile:
    the attention's KV tile (0: the head dim's default; 64 or 128 at Dh=128)."""
    for t in (k_cache, v_cache):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4:
            raise ValueError("caches must be 4-D BF16 CUDA tensors [num_blocks, 16, Hkv, Dh]")
        if t.stride(3) != 1:
            raise ValueError("the head dimension of the caches must be contiguous")
    if k_cache.shape != v_cache.shape or k_cache.stride() != v_cache.stride():
        raise ValueError("K and V caches must have the same shape and strides")
    nb, bs, hkv, dh = k_cache.shape
    return PaKvCache(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, hkv, dh, int(kv_tile), k_cache.stride(0),
                     k_cache.stride(1), k_cache.stride(2))


def _validate_write(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor) -> int:
    """Checks the cache-write inputs; returns the token count."""
    for t in (key, value):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 3 or t.stride(2) != 1 \
                or t.stride(1) != t.shape[2]:
            raise ValueError("key/value must be [N, Hkv, Dh] BF16 CUDA tensors with contiguous heads")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 CUDA tensor")
    n = key.shape[0]
    if value.shape[0] != n or slot_mapping.numel() != n:
        raise ValueError("key, value and slot_mapping disagree on the token count")
    return n


def _validate_attention(q: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                        query_start_loc: torch.Tensor) -> Tuple[int, int, int, int]:
    """Checks the attention inputs; returns (Tq, Hq, Dh, num_seqs)."""
    if q.dtype != torch.bfloat16 or not q.is_cuda or q.dim() != 3 or q.stride(2) != 1 \
            or q.stride(1) != q.shape[2]:
        raise ValueError("q must be a [Tq, Hq, Dh] BF16 CUDA tensor with contiguous heads")
    tq, hq, dh = q.shape
    for name, t in (("block_tables", block_tables), ("seq_lens", seq_lens),
                    ("query_start_loc", query_start_loc)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    num_seqs = seq_lens.numel()
    if query_start_loc.numel() != num_seqs + 1 or block_tables.dim() != 2 \
            or block_tables.shape[0] != num_seqs:
        raise ValueError("metadata shapes disagree")
    return tq, hq, dh, num_seqs


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                      stream: Optional[torch.cuda.Stream] = None) -> None:
    """Write key/value [N, Hkv, Dh] into the caches at slot_mapping [N] (int64);
    negative slots are skipped."""
    c = cache_struct(k_cache, v_cache)
    n = _validate_write(key, value, slot_mapping)
    _check(load().pa_reshape_and_cache(key.data_ptr(), key.stride(0), value.data_ptr(), value.stride(0),
                                       n, ctypes.byref(c), slot_mapping.data_ptr(),
                                       _stream_handle(stream)), "pa_reshape_and_cache")


def workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   max_query_len: int, max_seq_len: int) -> int:
    return int(load().pa_paged_attention_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                        max_query_len, max_seq_len))


def new_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                  max_query_len: int, max_seq_len: int, device=None) -> torch.Tensor:
    """Zero-filled scratch for pa_paged_attention (reusable across calls)."""
    n = workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_query_len, max_seq_len)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def paged_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    block_tables: torch.Tensor, seq_lens: torch.Tensor,
                    query_start_loc: torch.Tensor, scale: float, max_query_len: int,
                    max_seq_len: int, out: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, want_lse: bool = True,
                    workspace: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None, kv_tile: int = 0
                    ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Causal GQA attention of q [Tq, Hq, Dh] over the paged caches.
    Returns (out [Tq, Hq, Dh] BF16, lse [Tq, Hq] fp32 or None).  kv_tile
    selects the fixed arithmetic's KV tile (see cache_struct)."""
    c = cache_struct(k_cache, v_cache, kv_tile)
    tq, hq, dh, num_seqs = _validate_attention(q, block_tables, seq_lens, query_start_loc)
    if out is None:
        out = torch.empty((tq, hq, dh), dtype=torch.bfloat16, device=q.device)
    elif out.shape != (tq, hq, dh) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [Tq, Hq, Dh] BF16 tensor")
    if lse is None and want_lse:
        lse = torch.empty((tq, hq), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (tq, hq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous [Tq, Hq] fp32 tensor")
    _check_result_tensor("out", out)
    if lse is not None:
        _check_result_tensor("lse", lse)
    need = workspace_size(num_seqs, hq, c.num_kv_heads, dh, max_query_len, max_seq_len)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pa_paged_attention(
        q.data_ptr(), tq, q.stride(0), hq, ctypes.byref(c), block_tables.data_ptr(),
        block_tables.shape[1], seq_lens.data_ptr(), query_start_loc.data_ptr(), num_seqs,
        int(max_query_len), int(max_seq_len), float(scale), out.data_ptr(),
        lse.data_ptr() if lse is not None else 0, ws_ptr, ws_len, _stream_handle(stream)),
        "pa_paged_attention")
    return out, lse


def paged_attention_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor,
                            query_start_loc: torch.Tensor, scale: float, max_query_len: int,
                            max_seq_len: int, out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None, kv_tile: int = 0) -> int:
    """paged_attention for callers that cannot allocate: no workspace and no
    output allocation here (out, and lse if wanted, are passed in); the
    library's built-in scratch array is used instead.  Returns the status
    code (PA_ERR_WORKSPACE when the bounds need more than
    NOALLOC_SCRATCH_BYTES) rather than raising."""
    c = cache_struct(k_cache, v_cache, kv_tile)
    tq, hq, dh = q.shape
    return int(load().pa_paged_attention_noalloc(
        q.data_ptr(), tq, q.stride(0), hq, ctypes.byref(c), block_tables.data_ptr(),
        block_tables.shape[1], seq_lens.data_ptr(), query_start_loc.data_ptr(), seq_lens.numel(),
        int(max_query_len), int(max_seq_len), float(scale), out.data_ptr(),
        lse.data_ptr() if lse is not None else 0, _stream_handle(stream)))


class PreparedCall:
    """A library call validated and marshalled once.  Calling it re-issues the
    same C-ABI call with the same pointers: the tensors' contents may change
    between calls, their storage must stay alive and in place (the object
    keeps references to them)."""

    def __init__(self, fn, args, what: str, keep):
        self._fn, self._args, self._what, self._keep = fn, args, what, keep

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != PA_OK:
            raise PagedAttnError(st, self._what)


def _check_result_tensor(name: str, t: torch.Tensor) -> None:
    """out / lse: device memory, or page-locked host memory the kernels write
    directly (mapped into the device's address space)."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")


def prepare_copy_to_device(dst: torch.Tensor, src: torch.Tensor,
                           stream: Optional[torch.cuda.Stream] = None, src_ready: bool = False) -> PreparedCall:
    """pa_copy_to_device of all of src's bytes into dst (a CUDA tensor of the
    same byte size; src a pinned host tensor or a CUDA tensor), validated now
    and issued by each call of the result.  src_ready: no kernel in flight
    writes src (e.g. host memory the host fills), so it is read at once."""
    nbytes = src.numel() * src.element_size()
    if not dst.is_cuda or not dst.is_contiguous() or not src.is_contiguous() \
            or dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst must be a contiguous CUDA tensor of src's byte size")
    if not (src.is_cuda or src.is_pinned()):
        raise ValueError("src must be a pinned host tensor or a CUDA tensor")
    lib = load()
    return PreparedCall(lib.pa_copy_to_device,
                        (dst.data_ptr(), src.data_ptr(), nbytes, 1 if src_ready else 0, _stream_handle(stream)),
                        "pa_copy_to_device", (dst, src))


def copy_to_device(dst: torch.Tensor, src: torch.Tensor, stream: Optional[torch.cuda.Stream] = None,
                   src_ready: bool = False) -> None:
    """Copy src (pinned host or CUDA) into the CUDA tensor dst with the
    library's staging kernel."""
    prepare_copy_to_device(dst, src, stream, src_ready)()


def prepare_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                              v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                              stream: Optional[torch.cuda.Stream] = None) -> PreparedCall:
    """reshape_and_cache, validated now and issued by each call of the result."""
    c = cache_struct(k_cache, v_cache)
    n = _validate_write(key, value, slot_mapping)
    lib = load()
    args = (key.data_ptr(), key.stride(0), value.data_ptr(), value.stride(0), n, ctypes.byref(c),
            slot_mapping.data_ptr(), _stream_handle(stream))
    return PreparedCall(lib.pa_reshape_and_cache, args, "pa_reshape_and_cache",
                        (key, value, k_cache, v_cache, slot_mapping, c))


def prepare_paged_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor,
                            query_start_loc: torch.Tensor, scale: float, max_query_len: int,
                            max_seq_len: int, out: torch.Tensor, lse: Optional[torch.Tensor],
                            workspace: Optional[torch.Tensor],
                            stream: Optional[torch.cuda.Stream] = None, kv_tile: int = 0) -> PreparedCall:
    """paged_attention into given out / lse / workspace, validated now and
    issued by each call of the result."""
    c = cache_struct(k_cache, v_cache, kv_tile)
    tq, hq, dh, num_seqs = _validate_attention(q, block_tables, seq_lens, query_start_loc)
    if out.shape != (tq, hq, dh) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [Tq, Hq, Dh] BF16 tensor")
    if lse is not None and (lse.shape != (tq, hq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous [Tq, Hq] fp32 tensor")
    _check_result_tensor("out", out)
    if lse is not None:
        _check_result_tensor("lse", lse)
    need = workspace_size(num_seqs, hq, c.num_kv_heads, dh, max_query_len, max_seq_len)
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if ws_len < need:
        raise ValueError(f"workspace needs {need} bytes")
    lib = load()
    args = (q.data_ptr(), tq, q.stride(0), hq, ctypes.byref(c), block_tables.data_ptr(),
            block_tables.shape[1], seq_lens.data_ptr(), query_start_loc.data_ptr(), num_seqs,
            int(max_query_len), int(max_seq_len), ctypes.c_float(float(scale)), out.data_ptr(),
            lse.data_ptr() if lse is not None else 0, workspace.data_ptr() if workspace is not None else 0,
            ws_len, _stream_handle(stream))
    return PreparedCall(lib.pa_paged_attention, args, "pa_paged_attention",
                        (q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, out, lse, workspace, c))


def _composition_args(key, value, slot_mapping, q, k_cache, v_cache, block_tables, seq_lens,
                      query_start_loc, scale, max_query_len, max_seq_len, out, lse, workspace, stream, kv_tile):
    c = cache_struct(k_cache, v_cache, kv_tile)
    n = _validate_write(key, value, slot_mapping)
    tq, hq, dh, num_seqs = _validate_attention(q, block_tables, seq_lens, query_start_loc)
    if out.shape != (tq, hq, dh) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [Tq, Hq, Dh] BF16 tensor")
    if lse is not None and (lse.shape != (tq, hq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous [Tq, Hq] fp32 tensor")
    _check_result_tensor("out", out)
    if lse is not None:
        _check_result_tensor("lse", lse)
    need = workspace_size(num_seqs, hq, c.num_kv_heads, dh, max_query_len, max_seq_len)
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if ws_len < need:
        raise ValueError(f"workspace needs {need} bytes")
    args = (key.data_ptr(), key.stride(0), value.data_ptr(), value.stride(0), n, slot_mapping.data_ptr(),
            q.data_ptr(), tq, q.stride(0), hq, ctypes.byref(c), block_tables.data_ptr(),
            block_tables.shape[1], seq_lens.data_ptr(), query_start_loc.data_ptr(), num_seqs,
            int(max_query_len), int(max_seq_len), ctypes.c_float(float(scale)), out.data_ptr(),
            lse.data_ptr() if lse is not None else 0, workspace.data_ptr() if workspace is not None else 0,
            ws_len, _stream_handle(stream))
    keep = (key, value, slot_mapping, q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, out, lse,
            workspace, c)
    return args, keep


def reshape_and_paged_attention(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
                                q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                query_start_loc: torch.Tensor, scale: float, max_query_len: int,
                                max_seq_len: int, out: Optional[torch.Tensor] = None,
                                lse: Optional[torch.Tensor] = None, want_lse: bool = True,
                                workspace: Optional[torch.Tensor] = None,
                                stream: Optional[torch.cuda.Stream] = None, kv_tile: int = 0
                                ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """reshape_and_cache of key/value at slot_mapping, then paged_attention of q
    over the updated caches, in one library call whose attention grid starts
    its set-up while the cache write runs.  Returns (out, lse or None)."""
    tq, hq, dh = q.shape
    if out is None:
        out = torch.empty((tq, hq, dh), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((tq, hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = workspace_size(seq_lens.numel(), hq, k_cache.shape[2], dh, max_query_len, max_seq_len)
        if need > 0:
            workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    args, _keep = _composition_args(key, value, slot_mapping, q, k_cache, v_cache, block_tables, seq_lens,
                                    query_start_loc, scale, max_query_len, max_seq_len, out, lse, workspace,
                                    stream, kv_tile)
    _check(load().pa_reshape_and_paged_attention(*args), "pa_reshape_and_paged_attention")
    return out, lse


def prepare_reshape_and_paged_attention(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
                                        q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                        block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                        query_start_loc: torch.Tensor, scale: float, max_query_len: int,
                                        max_seq_len: int, out: torch.Tensor, lse: Optional[torch.Tensor],
                                        workspace: Optional[torch.Tensor],
                                        stream: Optional[torch.cuda.Stream] = None,
                                        kv_tile: int = 0) -> PreparedCall:
    """reshape_and_paged_attention into given out / lse / workspace, validated
    now and issued by each call of the result."""
    args, keep = _composition_args(key, value, slot_mapping, q, k_cache, v_cache, block_tables, seq_lens,
                                   query_start_loc, scale, max_query_len, max_seq_len, out, lse, workspace,
                                   stream, kv_tile)
    return PreparedCall(load().pa_reshape_and_paged_attention, args, "pa_reshape_and_paged_attention", keep)


def _validate_gather(k_cache: torch.Tensor, kv_head: int, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                     packed_k: torch.Tensor, packed_v: torch.Tensor, compact_tables: torch.Tensor,
                     compact_offsets: torch.Tensor) -> int:
    """Checks the gather inputs; returns the packed capacity in pages."""
    num_seqs = seq_lens.numel()
    for name, t in (("block_tables", block_tables), ("seq_lens", seq_lens), ("compact_tables", compact_tables),
                    ("compact_offsets", compact_offsets)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    if block_tables.dim() != 2 or block_tables.shape[0] != num_seqs or compact_tables.shape != block_tables.shape \
            or compact_offsets.numel() != num_seqs + 1:
        raise ValueError("metadata shapes disagree")
    dh = k_cache.shape[3]
    for t in (packed_k, packed_v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4 \
                or tuple(t.shape[1:]) != (16, 1, dh):
            raise ValueError("packed buffers must be contiguous BF16 CUDA tensors [capacity_pages, 16, 1, Dh]")
    if packed_k.shape != packed_v.shape:
        raise ValueError("packed K and V must have the same capacity")
    if not 0 <= kv_head < k_cache.shape[2]:
        raise ValueError("kv_head out of range")
    return packed_k.shape[0]


def gather_kv_head(k_cache: torch.Tensor, v_cache: torch.Tensor, kv_head: int, block_tables: torch.Tensor,
                   seq_lens: torch.Tensor, packed_k: torch.Tensor, packed_v: torch.Tensor,
                   compact_tables: torch.Tensor, compact_offsets: torch.Tensor,
                   stream: Optional[torch.cuda.Stream] = None) -> None:
    """Pack the pages that block_tables/seq_lens select for one KV head into
    packed_k/packed_v [capacity_pages, 16, 1, Dh] (a one-head pool of their
    own), writing the compact table [B, max_blocks] and page offsets [B + 1]."""
    c = cache_struct(k_cache, v_cache)
    cap = _validate_gather(k_cache, kv_head, block_tables, seq_lens, packed_k, packed_v, compact_tables,
                           compact_offsets)
    _check(load().pa_gather_kv_head(ctypes.byref(c), kv_head, block_tables.data_ptr(), block_tables.shape[1],
                                    seq_lens.data_ptr(), seq_lens.numel(), packed_k.data_ptr(),
                                    packed_v.data_ptr(), cap, compact_tables.data_ptr(),
                                    compact_offsets.data_ptr(), _stream_handle(stream)), "pa_gather_kv_head")


def prepare_gather_kv_head(k_cache: torch.Tensor, v_cache: torch.Tensor, kv_head: int, block_tables: torch.Tensor,
                           seq_lens: torch.Tensor, packed_k: torch.Tensor, packed_v: torch.Tensor,
                           compact_tables: torch.Tensor, compact_offsets: torch.Tensor,
                           stream: Optional[torch.cuda.Stream] = None) -> "PreparedCall":
    """gather_kv_head validated and marshalled once; calling the result
    re-issues the same C-ABI call (tensor contents may change, not storage)."""
    c = cache_struct(k_cache, v_cache)
    cap = _validate_gather(k_cache, kv_head, block_tables, seq_lens, packed_k, packed_v, compact_tables,
                           compact_offsets)
    keep = (c, k_cache, v_cache, block_tables, seq_lens, packed_k, packed_v, compact_tables, compact_offsets)
    args = (ctypes.byref(c), kv_head, block_tables.data_ptr(), block_tables.shape[1], seq_lens.data_ptr(),
            seq_lens.numel(), packed_k.data_ptr(), packed_v.data_ptr(), cap, compact_tables.data_ptr(),
            compact_offsets.data_ptr(), _stream_handle(stream))
    return PreparedCall(load().pa_gather_kv_head, args, "pa_gather_kv_head", keep)


def check_errors(stream: Optional[torch.cuda.Stream] = None) -> Tuple[int, int]:
    """Synchronise the stream, read and clear the device error latch.
    Returns (status, first_bad_index)."""
    idx = ctypes.c_int64(-1)
    st = load().pa_check_errors(_stream_handle(stream), ctypes.byref(idx))
    return int(st), int(idx.value)

"""The C-ABI boundary without a GPU: the library builds and loads, exports
every entry point the header declares, and rejects bad arguments on the
host before touching CUDA."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_178_gb300 import build as pa_build
from paged_kv_cache_178_gb300 import pagedattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return pagedattn.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = _declared()
    assert set(pagedattn.EXPORTED) <= set(names)
    assert "pa_reshape_and_cache" in names and "pa_paged_attention" in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(["PA_OK", "PA_ERR_INVALID_ARG", "PA_ERR_UNSUPPORTED",
                                 "PA_ERR_WORKSPACE", "PA_ERR_BAD_METADATA", "PA_ERR_TIMEOUT",
                                 "PA_ERR_CUDA"]):
        assert pagedattn.status_string(code) == name


FAKE = 0x10000000  # aligned, never dereferenced: validation fails before any CUDA call


def _cache(**kw):
    c = dict(k=FAKE, v=FAKE + 0x1000, num_blocks=2048, block_size=16, num_kv_heads=2, head_dim=128,
             kv_tile=0, block_stride=2 * 16 * 2 * 128, token_stride=2 * 128, head_stride=128)
    c.update(kw)
    return pagedattn.PaKvCache(**c)


def _rc(lib, cache, key=FAKE, value=FAKE, kstride=256, vstride=256, n=4, slots=FAKE):
    return lib.pa_reshape_and_cache(key, kstride, value, vstride, n, ctypes.byref(cache), slots, None)


def test_cache_write_validation(lib):
    assert _rc(lib, _cache(block_size=8)) == pagedattn.PA_ERR_UNSUPPORTED
    assert _rc(lib, _cache(head_dim=64)) == pagedattn.PA_ERR_UNSUPPORTED
    assert _rc(lib, _cache(k=FAKE + 2)) == pagedattn.PA_ERR_INVALID_ARG
    assert _rc(lib, _cache(token_stride=250)) == pagedattn.PA_ERR_INVALID_ARG
    assert _rc(lib, _cache(num_blocks=0)) == pagedattn.PA_ERR_INVALID_ARG
    assert _rc(lib, _cache(), key=FAKE + 8) == pagedattn.PA_ERR_INVALID_ARG
    assert _rc(lib, _cache(), kstride=128) == pagedattn.PA_ERR_INVALID_ARG
    assert _rc(lib, _cache(), slots=FAKE + 4) == pagedattn.PA_ERR_INVALID_ARG
    assert _rc(lib, _cache(), n=-1) == pagedattn.PA_ERR_INVALID_ARG
    assert _rc(lib, _cache(), n=0) == pagedattn.PA_OK          # nothing to launch
    assert lib.pa_reshape_and_cache(FAKE, 256, FAKE, 256, 4, None, FAKE, None) == \
        pagedattn.PA_ERR_INVALID_ARG


def _attn(lib, cache, q=FAKE, ntok=4, qstride=1024, hq=8, bt=FAKE, maxblk=448, sl=FAKE, qsl=FAKE,
          nseq=4, mq=1, ms=7168, scale=0.088, out=FAKE, lse=0, ws=0, ws_len=0):
    return lib.pa_paged_attention(q, ntok, qstride, hq, ctypes.byref(cache), bt, maxblk, sl, qsl, nseq,
                                  mq, ms, ctypes.c_float(scale), out, lse, ws, ws_len, None)


def test_attention_validation(lib):
    c = _cache()
    ws = pagedattn.workspace_size(4, 8, 2, 128, 1, 7168)
    assert _attn(lib, c, hq=7) == pagedattn.PA_ERR_UNSUPPORTED           # Hq % Hkv
    assert _attn(lib, c, hq=2 * 129) == pagedattn.PA_ERR_UNSUPPORTED     # group > 128
    assert _attn(lib, c, q=FAKE + 2) == pagedattn.PA_ERR_INVALID_ARG
    assert _attn(lib, c, qstride=1000) == pagedattn.PA_ERR_INVALID_ARG
    assert _attn(lib, c, out=0) == pagedattn.PA_ERR_INVALID_ARG
    assert _attn(lib, c, lse=FAKE + 2) == pagedattn.PA_ERR_INVALID_ARG
    assert _attn(lib, c, scale=float("nan")) == pagedattn.PA_ERR_INVALID_ARG
    assert _attn(lib, c, scale=-0.1) == pagedattn.PA_ERR_INVALID_ARG
    assert _attn(lib, c, scale=0.0) == pagedattn.PA_ERR_INVALID_ARG
    assert _attn(lib, c, ws=0, ws_len=0) == pagedattn.PA_ERR_WORKSPACE
    assert _attn(lib, c, ws=FAKE, ws_len=ws - 1) == pagedattn.PA_ERR_WORKSPACE
    assert _attn(lib, c, ws=FAKE + 16, ws_len=ws) == pagedattn.PA_ERR_INVALID_ARG
    assert _attn(lib, c, nseq=0) == pagedattn.PA_OK                        # empty batch
    assert _attn(lib, c, mq=-1) == pagedattn.PA_ERR_INVALID_ARG
    # the attention's KV tile: 0 or a tile the head dim has
    assert _attn(lib, _cache(kv_tile=32)) == pagedattn.PA_ERR_INVALID_ARG
    assert _attn(lib, _cache(kv_tile=64), nseq=0) == pagedattn.PA_OK
    assert _attn(lib, _cache(kv_tile=128), nseq=0) == pagedattn.PA_OK
    dh256 = dict(head_dim=256, head_stride=256, token_stride=512, block_stride=2 * 16 * 512)
    assert _attn(lib, _cache(kv_tile=64, **dh256)) == pagedattn.PA_ERR_UNSUPPORTED
    dh512 = dict(head_dim=512, head_stride=512, token_stride=1024, block_stride=2 * 16 * 1024)
    assert _attn(lib, _cache(kv_tile=128, **dh512)) == pagedattn.PA_ERR_UNSUPPORTED
    assert _rc(lib, _cache(kv_tile=32), n=0) == pagedattn.PA_OK           # the cache write ignores it


# Buffers for the one-call composition, 16 MB apart and clear of the fake
# pool (2048 blocks x 8192 elements x 2 bytes from FAKE).
_BUF = {name: 0x20000000 + i * 0x1000000
        for i, name in enumerate(("key", "value", "slots", "q", "bt", "sl", "qsl", "out", "lse", "ws"))}


def _rpa(lib, cache, **kw):
    a = dict(_BUF)
    a.update(kw)
    ws_len = pagedattn.workspace_size(4, 8, 2, 128, 1, 7168)
    return lib.pa_reshape_and_paged_attention(
        a["key"], 256, a["value"], 256, a.get("n", 4), a["slots"], a["q"], 4, 1024, a.get("hq", 8),
        ctypes.byref(cache), a["bt"], 448, a["sl"], a["qsl"], 4, 1, 7168, ctypes.c_float(0.088), a["out"],
        a["lse"], a["ws"], ws_len, None)


def test_composition_validation_and_overlap(lib):
    import torch
    c = _cache()
    # either half's checks apply before anything is launched
    assert _rpa(lib, c, key=_BUF["key"] + 8) == pagedattn.PA_ERR_INVALID_ARG
    assert _rpa(lib, c, hq=7) == pagedattn.PA_ERR_UNSUPPORTED
    assert _rpa(lib, _cache(block_size=8)) == pagedattn.PA_ERR_UNSUPPORTED
    # the attention writes out / lse / workspace while the cache write may run
    assert _rpa(lib, c, out=FAKE + 4096) == pagedattn.PA_ERR_INVALID_ARG      # inside the pool
    assert _rpa(lib, c, out=_BUF["key"]) == pagedattn.PA_ERR_INVALID_ARG      # over key
    assert _rpa(lib, c, lse=_BUF["slots"] + 16) == pagedattn.PA_ERR_INVALID_ARG
    assert _rpa(lib, c, ws=_BUF["value"]) == pagedattn.PA_ERR_INVALID_ARG
    # q and the metadata are read early: none may lie in the pool
    assert _rpa(lib, c, q=FAKE + (1 << 20)) == pagedattn.PA_ERR_INVALID_ARG
    assert _rpa(lib, c, bt=FAKE + 256) == pagedattn.PA_ERR_INVALID_ARG
    assert _rpa(lib, c, qsl=FAKE + 2047 * 8192 * 2) == pagedattn.PA_ERR_INVALID_ARG  # last block
    # just past the V view's last byte is fine; sharing bytes among the
    # read-only inputs (q over key) is fine too
    end = FAKE + 0x1000 + (2047 * 8192 + 15 * 256 + 128 + 128) * 2
    assert _rpa(lib, c, sl=end - 4) == pagedattn.PA_ERR_INVALID_ARG
    ok = pagedattn.PA_OK if torch.cuda.is_available() else pagedattn.PA_ERR_CUDA
    if not torch.cuda.is_available():
        assert _rpa(lib, c, sl=end) == ok
        assert _rpa(lib, c, q=_BUF["key"]) == ok


def test_workspace_size_is_host_arithmetic(lib):
    # decode: 4 requests x 2 KV heads, one 4-row query tile each, 28 chunks
    # of 256 keys, records of (m, l, O[128]) per row + 256 B of counters
    assert pagedattn.workspace_size(4, 8, 2, 128, 1, 7168) == 256 + 8 * 28 * 4 * 130 * 4
    # a long prefill runs in-CTA: no scratch at all
    assert pagedattn.workspace_size(1, 8, 2, 128, 4096, 4096) == 0
    # short sequences fit one chunk: no scratch
    assert pagedattn.workspace_size(4, 8, 2, 128, 1, 256) == 0
    # invalid geometry
    assert pagedattn.workspace_size(4, 8, 3, 128, 1, 7168) == 0


def test_no_gpu_calls_report_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    idx = ctypes.c_int64(7)
    assert lib.pa_check_errors(None, ctypes.byref(idx)) == pagedattn.PA_ERR_CUDA
    assert lib.pa_init() == pagedattn.PA_ERR_CUDA
    assert _rc(lib, _cache()) == pagedattn.PA_ERR_CUDA


def test_launch_info_is_a_string(lib):
    s = pagedattn.last_launch_info()
    assert isinstance(s, str) and len(s) > 0


def _gkv(lib, cache, head=0, bt=_BUF["bt"], maxblk=448, sl=_BUF["sl"], nseq=4, pk=_BUF["out"],
         pv=_BUF["lse"], cap=1800, ct=_BUF["ws"], co=_BUF["qsl"]):
    return lib.pa_gather_kv_head(ctypes.byref(cache), head, bt, maxblk, sl, nseq, pk, pv, cap, ct, co, None)


def test_gather_validation_and_overlap(lib):
    import torch
    c = _cache()
    assert _gkv(lib, c, head=2) == pagedattn.PA_ERR_INVALID_ARG
    assert _gkv(lib, c, head=-1) == pagedattn.PA_ERR_INVALID_ARG
    assert _gkv(lib, c, maxblk=0) == pagedattn.PA_ERR_INVALID_ARG
    assert _gkv(lib, c, cap=-1) == pagedattn.PA_ERR_INVALID_ARG
    assert _gkv(lib, c, nseq=513) == pagedattn.PA_ERR_UNSUPPORTED
    assert _gkv(lib, c, nseq=512, maxblk=1 << 23) == pagedattn.PA_ERR_UNSUPPORTED  # table indices past int32
    assert _gkv(lib, c, pk=_BUF["out"] + 8) == pagedattn.PA_ERR_INVALID_ARG
    assert _gkv(lib, c, co=_BUF["qsl"] + 2) == pagedattn.PA_ERR_INVALID_ARG
    assert _gkv(lib, c, ct=0) == pagedattn.PA_ERR_INVALID_ARG
    assert _gkv(lib, _cache(head_dim=64)) == pagedattn.PA_ERR_UNSUPPORTED
    assert _gkv(lib, c, nseq=0) == pagedattn.PA_OK                        # nothing to launch
    # outputs may not overlap the pool, the metadata or each other
    assert _gkv(lib, c, pk=FAKE + 4096) == pagedattn.PA_ERR_INVALID_ARG
    assert _gkv(lib, c, ct=_BUF["bt"] + 64) == pagedattn.PA_ERR_INVALID_ARG
    assert _gkv(lib, c, pv=_BUF["out"] + 1799 * 4096) == pagedattn.PA_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert _gkv(lib, c) == pagedattn.PA_ERR_CUDA
        assert _gkv(lib, c, pv=_BUF["out"] + 1800 * 4096) == pagedattn.PA_ERR_CUDA  # adjacent: fine
        assert _gkv(lib, c, cap=0, pk=0, pv=0) == pagedattn.PA_ERR_CUDA  # offsets only


def _noalloc(lib, cache, q=FAKE, ntok=4, qstride=1024, hq=8, bt=FAKE, maxblk=448, sl=FAKE, qsl=FAKE,
             nseq=4, mq=1, ms=7168, scale=0.088, out=FAKE, lse=0):
    return lib.pa_paged_attention_noalloc(q, ntok, qstride, hq, ctypes.byref(cache), bt, maxblk, sl, qsl,
                                          nseq, mq, ms, ctypes.c_float(scale), out, lse, None)


def test_noalloc_validates_before_any_cuda_call(lib):
    """The allocation-free entry point runs every host check of the regular
    one, against its built-in scratch size, before it touches CUDA: on a
    machine without a GPU a bad call returns its own status, and only a
    valid call reaches the CUDA runtime (PA_ERR_CUDA here)."""
    import torch
    c = _cache()
    assert _noalloc(lib, c, hq=7) == pagedattn.PA_ERR_UNSUPPORTED               # Hq % Hkv
    assert _noalloc(lib, _cache(head_dim=64)) == pagedattn.PA_ERR_UNSUPPORTED    # head dim
    assert _noalloc(lib, _cache(num_kv_heads=0)) == pagedattn.PA_ERR_INVALID_ARG
    assert _noalloc(lib, c, mq=-1) == pagedattn.PA_ERR_INVALID_ARG
    assert _noalloc(lib, c, q=0) == pagedattn.PA_ERR_INVALID_ARG
    assert _noalloc(lib, c, out=FAKE + 8) == pagedattn.PA_ERR_INVALID_ARG
    assert _noalloc(lib, c, scale=0.0) == pagedattn.PA_ERR_INVALID_ARG
    assert lib.pa_paged_attention_noalloc(FAKE, 4, 1024, 8, None, FAKE, 448, FAKE, FAKE, 4, 1, 7168,
                                          ctypes.c_float(0.088), FAKE, 0, None) == pagedattn.PA_ERR_INVALID_ARG
    big = 1 << 20                      # bounds whose scratch exceeds the built-in array
    assert pagedattn.workspace_size(4, 8, 2, 128, 1, big) > pagedattn.NOALLOC_SCRATCH_BYTES
    assert _noalloc(lib, c, ms=big) == pagedattn.PA_ERR_WORKSPACE
    assert _noalloc(lib, c, nseq=0) == pagedattn.PA_OK                          # empty batch
    if not torch.cuda.is_available():
        assert _noalloc(lib, c) == pagedattn.PA_ERR_CUDA                        # valid: reaches CUDA


def test_copy_to_device_validates_before_any_cuda_call(lib):
    ok, bad = pagedattn.PA_OK, pagedattn.PA_ERR_INVALID_ARG
    assert lib.pa_copy_to_device(FAKE, FAKE + 4096, 0, 0, None) == ok          # nothing to copy
    assert lib.pa_copy_to_device(None, FAKE, 64, 0, None) == bad
    assert lib.pa_copy_to_device(FAKE, None, 64, 0, None) == bad
    assert lib.pa_copy_to_device(FAKE, FAKE + 32, 64, 0, None) == bad          # overlapping ranges
    assert lib.pa_copy_to_device(FAKE + 32, FAKE, 64, 0, None) == bad
    assert lib.pa_copy_to_device(FAKE + 8, FAKE + 4096, 64, 0, None) == bad    # dst not 16-byte aligned
    assert lib.pa_copy_to_device(FAKE, FAKE + 4100, 64, 0, None) == bad        # src not 16-byte aligned

"""Python binding of libpkv: paged decode attention (fp16 / INT8 KV) for GB300.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of ``libpkv.so`` behind the C ABI declared in ``include/pkv.h``;
PyTorch supplies device memory and streams.  There is no fallback: if the
library has not been built (``paged_kv_cache_234_gb300.build.build()``), every
call raises.

The functions carry the C names and take torch tensors:

* ``pkv_quantize_blocks``     fp16 K/V tiles -> INT8 codes + fp32 scales
* ``pkv_paged_decode_fp16``   decode-step attention over fp16 K/V pools
* ``pkv_paged_decode_int8``   decode-step attention over INT8 K/V pools
* ``pkv_quantize_blocks_fp8`` fp16 K/V tiles -> FP8 (E4M3) codes + fp32 scales
* ``pkv_paged_decode_fp8``    decode-step attention over FP8 K/V pools
* ``pkv_append_fp16``         write one new token per sequence into fp16 pools
* ``pkv_append_int8``         the same, re-quantizing every tile it writes
* ``pkv_evict_select``        eviction scores of every block + the k to evict
* ``BlockManager``            host block manager (``pkv_bm_*``: free list,
                              reference counts, prefix sharing, copy-on-write)
* ``pkv_copy_blocks``         the batched block copies copy-on-write asks for
* ``pkv_decode_workspace_size``, ``pkv_set_decode_workers``,
  ``pkv_status_string``

``prepare_paged_decode_fp16`` / ``_int8`` / ``_fp8`` and
``prepare_quantize_blocks`` / ``_fp8`` take the same arguments as the calls
above and return a ``PreparedCall``: the arguments checked and marshalled
once, each call of the object issuing the same C call again (for serving
loops that update the same buffers in place every step).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "_build", "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_UNSUPPORTED = 2
PKV_ERR_MISALIGNED = 3
PKV_ERR_WORKSPACE = 4
PKV_ERR_CUDA = 5
PKV_ERR_EXHAUSTED = 6

PKV_DEV_BAD_BLOCK = 1
PKV_DEV_BAD_CTX = 2
PKV_DEV_TIMEOUT = 4

EXPORTED = ("pkv_quantize_blocks", "pkv_paged_decode_fp16", "pkv_paged_decode_int8",
            "pkv_quantize_blocks_fp8", "pkv_paged_decode_fp8",
            "pkv_paged_decode_int8_static_workspace", "pkv_append_fp16", "pkv_append_int8",
            "pkv_append_fp8",
            "pkv_evict_select", "pkv_bm_create", "pkv_bm_destroy", "pkv_bm_allocate",
            "pkv_bm_free", "pkv_bm_fork", "pkv_bm_cow", "pkv_bm_set_fill", "pkv_bm_stats",
            "pkv_bm_refcounts", "pkv_copy_blocks", "pkv_decode_workspace_size",
            "pkv_set_decode_workers", "pkv_status_string")

# weights of the least-reference-count + age eviction score
EVICT_ALPHA = 0.7
EVICT_BETA = 0.3

# size of the scratch array behind pkv_paged_decode_int8_static_workspace
PKV_STATIC_WORKSPACE_BYTES = 32 << 20

_lock = threading.Lock()
_lib = None
_debug_lib = None


class BmStats(ctypes.Structure):
    _fields_ = [("free_blocks", ctypes.c_int64), ("used_blocks", ctypes.c_int64),
                ("shared_blocks", ctypes.c_int64), ("logical_blocks", ctypes.c_int64),
                ("tokens", ctypes.c_int64), ("internal_fragmentation", ctypes.c_double),
                ("sharing_saving", ctypes.c_double)]


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {pkv_status_string(status)} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded C library with argument types set (raises if not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libpkv is not built ({LIB_PATH} missing); run "
                "paged_kv_cache_234_gb300.build.build() first -- there is no fallback")
        _lib = _declare(ctypes.CDLL(LIB_PATH))
        return _lib


def debug_lib() -> ctypes.CDLL:
    """The library built with the decode kernel's debug checks
    (``build.build_debug()``), argument types set, plus ``pkv_debug_flags``.
    Test support only: the calls of this module always use ``lib()``."""
    global _debug_lib
    with _lock:
        if _debug_lib is None:
            from . import build as _build
            L = _declare(ctypes.CDLL(_build.build_debug()))
            for name in ("pkv_debug_flags", "pkv_debug_evict_flags"):
                getattr(L, name).restype = ctypes.c_uint
                getattr(L, name).argtypes = [ctypes.c_int]
            L.pkv_debug_set_stage_wait_ns.restype = ctypes.c_int
            L.pkv_debug_set_stage_wait_ns.argtypes = [ctypes.c_longlong]
            _debug_lib = L
        return _debug_lib


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    """Argument and result types of every C ABI entry point on ``L``."""
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.pkv_quantize_blocks.restype = I
    L.pkv_quantize_blocks.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, P]
    dec = [P, P, P, P, I, P, I, P, I, I, I, I, I, I, F, P, Z, P, P]
    L.pkv_paged_decode_fp16.restype = I
    L.pkv_paged_decode_fp16.argtypes = dec
    L.pkv_paged_decode_int8.restype = I
    L.pkv_paged_decode_int8.argtypes = dec[:4] + [P, P] + dec[4:]
    L.pkv_paged_decode_fp8.restype = I
    L.pkv_paged_decode_fp8.argtypes = dec[:4] + [P, P] + dec[4:]
    L.pkv_quantize_blocks_fp8.restype = I
    L.pkv_quantize_blocks_fp8.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, P]
    L.pkv_paged_decode_int8_static_workspace.restype = I
    L.pkv_paged_decode_int8_static_workspace.argtypes = dec[:4] + [P, P] + dec[4:15] + dec[17:]
    app = [P, P, I, P, P, P, I, P, I, I, I, I, P, P]
    L.pkv_append_fp16.restype = I
    L.pkv_append_fp16.argtypes = app
    L.pkv_append_int8.restype = I
    L.pkv_append_int8.argtypes = app[:2] + [P, P, P, P] + app[2:]
    L.pkv_append_fp8.restype = I
    L.pkv_append_fp8.argtypes = app[:2] + [P, P, P, P] + app[2:]
    L.pkv_evict_select.restype = I
    L.pkv_evict_select.argtypes = [P, P, I, ctypes.c_int64, F, F, I, P, P, P, P]
    L.pkv_bm_create.restype = I
    L.pkv_bm_create.argtypes = [I, I, ctypes.POINTER(P)]
    L.pkv_bm_destroy.restype = None
    L.pkv_bm_destroy.argtypes = [P]
    L.pkv_bm_allocate.restype = I
    L.pkv_bm_allocate.argtypes = [P, P, I, P]
    for name in ("pkv_bm_free", "pkv_bm_fork"):
        getattr(L, name).restype = I
        getattr(L, name).argtypes = [P, P, I]
    L.pkv_bm_cow.restype = I
    L.pkv_bm_cow.argtypes = [P, P, I, P, P, ctypes.POINTER(I)]
    L.pkv_bm_set_fill.restype = I
    L.pkv_bm_set_fill.argtypes = [P, P, P, I]
    L.pkv_bm_stats.restype = I
    L.pkv_bm_stats.argtypes = [P, ctypes.POINTER(BmStats)]
    L.pkv_bm_refcounts.restype = I
    L.pkv_bm_refcounts.argtypes = [P, P, I]
    L.pkv_copy_blocks.restype = I
    L.pkv_copy_blocks.argtypes = [P, P, I, I, P, I, P, P]
    L.pkv_decode_workspace_size.restype = Z
    L.pkv_decode_workspace_size.argtypes = [I, I, I, I, I]
    L.pkv_set_decode_workers.restype = I
    L.pkv_set_decode_workers.argtypes = [I]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_status_string.argtypes = [I]
    return L


def pkv_status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(t, name, dtype=None, host_ok=False):
    """host_ok: a pinned host tensor is accepted as well (the GPU reads or
    writes it in place over its link to the host; pinned memory has one
    address for the host and the GPU)."""
    if t is None:
        return
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" +
                         (" or a pinned host tensor" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len) -> int:
    return int(lib().pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                               max_context_len))


def pkv_set_decode_workers(max_workers: int) -> None:
    st = lib().pkv_set_decode_workers(int(max_workers))
    if st != PKV_OK:
        raise PkvError(st, "pkv_set_decode_workers")


def pkv_quantize_blocks(k_fp16, v_fp16, k_codes, v_codes, k_scales, v_scales,
                        block_ids=None, dev_status=None, stream=None) -> None:
    """Quantize the (block, kv head) tiles of fp16 pools [NB][Hkv][16][d]."""
    _invoke(*_quantize("pkv_quantize_blocks", k_fp16, v_fp16, k_codes, v_codes, k_scales,
                       v_scales, block_ids, dev_status, stream))


def pkv_quantize_blocks_fp8(k_fp16, v_fp16, k_codes, v_codes, k_scales, v_scales,
                            block_ids=None, dev_status=None, stream=None) -> None:
    """FP8 (E4M3, uint8 code pools) quantization of the tiles of fp16 pools."""
    _invoke(*_quantize("pkv_quantize_blocks_fp8", k_fp16, v_fp16, k_codes, v_codes, k_scales,
                       v_scales, block_ids, dev_status, stream))


def _invoke(fn_name, args):
    st = getattr(lib(), fn_name)(*args)
    if st != PKV_OK:
        raise PkvError(st, fn_name)


class PreparedCall:
    """One call of the C ABI with its arguments checked and marshalled once.

    Calling the object issues the same call again: the same buffers (by
    address; their contents may change between calls, as a serving loop
    updates its query, block tables and context lengths in place), the same
    sizes and the stream that was current (or given) at preparation.  The
    buffers must stay alive and must not be reallocated while the object is
    used (the object holds references to the tensors it was prepared with,
    so they are not freed while it lives).  It saves the per-call argument
    checks of the plain functions, about ten microseconds of host time per
    call."""

    __slots__ = ("_fn", "_args", "_name", "_keep")

    def __init__(self, fn_name, args, keep=()):
        self._fn = getattr(lib(), fn_name)
        self._args = tuple(args)
        self._name = fn_name
        self._keep = tuple(keep)

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != PKV_OK:
            raise PkvError(st, self._name)


def prepare_quantize_blocks(k_fp16, v_fp16, k_codes, v_codes, k_scales, v_scales,
                            block_ids=None, dev_status=None, stream=None) -> PreparedCall:
    """``pkv_quantize_blocks`` with its arguments marshalled once."""
    return PreparedCall(*_quantize("pkv_quantize_blocks", k_fp16, v_fp16, k_codes, v_codes,
                                   k_scales, v_scales, block_ids, dev_status, stream),
                        keep=(k_fp16, v_fp16, k_codes, v_codes, k_scales, v_scales, block_ids,
                              dev_status))


def prepare_quantize_blocks_fp8(k_fp16, v_fp16, k_codes, v_codes, k_scales, v_scales,
                                block_ids=None, dev_status=None, stream=None) -> PreparedCall:
    """``pkv_quantize_blocks_fp8`` with its arguments marshalled once."""
    return PreparedCall(*_quantize("pkv_quantize_blocks_fp8", k_fp16, v_fp16, k_codes, v_codes,
                                   k_scales, v_scales, block_ids, dev_status, stream),
                        keep=(k_fp16, v_fp16, k_codes, v_codes, k_scales, v_scales, block_ids,
                              dev_status))


def _quantize(fn_name, k_fp16, v_fp16, k_codes, v_codes, k_scales, v_scales, block_ids,
              dev_status, stream):
    """Checks and marshals a quantize call: (C function name, arguments)."""
    import torch
    code_t = torch.uint8 if fn_name.endswith("fp8") else torch.int8
    _check(k_fp16, "k_fp16", torch.float16)
    _check(v_fp16, "v_fp16", torch.float16)
    _check(k_codes, "k_codes", code_t)
    _check(v_codes, "v_codes", code_t)
    _check(k_scales, "k_scales", torch.float32)
    _check(v_scales, "v_scales", torch.float32)
    _check(block_ids, "block_ids", torch.int32, host_ok=True)
    _check(dev_status, "dev_status", torch.int32)
    nb, hkv, bs, d = k_fp16.shape
    nids = 0 if block_ids is None else block_ids.numel()
    return fn_name, [_ptr(k_fp16), _ptr(v_fp16), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales),
                     _ptr(v_scales), _ptr(block_ids), nids, nb, hkv, d, bs, _ptr(dev_status),
                     _stream(stream)]


def _decode(fn_name, out, query, kp, vp, ks, vs, block_tables, context_lens,
            max_context_len, softmax_scale, workspace, dev_status, stream):
    """Checks and marshals a decode call: (C function name, arguments)."""
    import torch
    # the per-step inputs and the output may live in pinned host memory
    _check(out, "out", torch.float32, host_ok=True)
    _check(query, "query", torch.float16, host_ok=True)
    _check(block_tables, "block_tables", torch.int32, host_ok=True)
    _check(context_lens, "context_lens", torch.int32, host_ok=True)
    _check(workspace, "workspace")
    _check(dev_status, "dev_status", torch.int32)
    if ks is None:
        _check(kp, "k_cache", torch.float16)
        _check(vp, "v_cache", torch.float16)
    else:
        code_t = torch.uint8 if fn_name.endswith("fp8") else torch.int8
        _check(kp, "k_codes", code_t)
        _check(vp, "v_codes", code_t)
        _check(ks, "k_scales", torch.float32)
        _check(vs, "v_scales", torch.float32)
    n, hq, d = query.shape
    nb, hkv, bs, _ = kp.shape
    mb = block_tables.shape[1] if block_tables.dim() == 2 else 0
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [_ptr(out), _ptr(query), _ptr(kp), _ptr(vp)]
    if ks is not None:
        args += [_ptr(ks), _ptr(vs)]
    args += [nb, _ptr(block_tables), mb, _ptr(context_lens), int(max_context_len), n, hq, hkv,
             d, bs, float(softmax_scale), _ptr(workspace), ws_bytes, _ptr(dev_status),
             _stream(stream)]
    return fn_name, args


def pkv_paged_decode_fp16(out, query, k_cache, v_cache, block_tables, context_lens,
                          max_context_len, softmax_scale, workspace, dev_status=None,
                          stream=None) -> None:
    """out[N][Hq][d] fp32 = decode attention of query over fp16 pools."""
    _invoke(*_decode("pkv_paged_decode_fp16", out, query, k_cache, v_cache, None, None,
                     block_tables, context_lens, max_context_len, softmax_scale, workspace,
                     dev_status, stream))


def pkv_paged_decode_int8(out, query, k_codes, v_codes, k_scales, v_scales, block_tables,
                          context_lens, max_context_len, softmax_scale, workspace,
                          dev_status=None, stream=None) -> None:
    """out[N][Hq][d] fp32 = decode attention of query over INT8 pools + scales."""
    _invoke(*_decode("pkv_paged_decode_int8", out, query, k_codes, v_codes, k_scales, v_scales,
                     block_tables, context_lens, max_context_len, softmax_scale, workspace,
                     dev_status, stream))


def pkv_paged_decode_fp8(out, query, k_codes, v_codes, k_scales, v_scales, block_tables,
                         context_lens, max_context_len, softmax_scale, workspace,
                         dev_status=None, stream=None) -> None:
    """out[N][Hq][d] fp32 = decode attention of query over FP8 (E4M3) pools."""
    _invoke(*_decode("pkv_paged_decode_fp8", out, query, k_codes, v_codes, k_scales, v_scales,
                     block_tables, context_lens, max_context_len, softmax_scale, workspace,
                     dev_status, stream))


def prepare_paged_decode_fp16(out, query, k_cache, v_cache, block_tables, context_lens,
                              max_context_len, softmax_scale, workspace, dev_status=None,
                              stream=None) -> PreparedCall:
    """``pkv_paged_decode_fp16`` with its arguments marshalled once."""
    return PreparedCall(*_decode("pkv_paged_decode_fp16", out, query, k_cache, v_cache, None,
                                 None, block_tables, context_lens, max_context_len,
                                 softmax_scale, workspace, dev_status, stream),
                        keep=(out, query, k_cache, v_cache, block_tables, context_lens,
                              workspace, dev_status))


def prepare_paged_decode_int8(out, query, k_codes, v_codes, k_scales, v_scales, block_tables,
                              context_lens, max_context_len, softmax_scale, workspace,
                              dev_status=None, stream=None) -> PreparedCall:
    """``pkv_paged_decode_int8`` with its arguments marshalled once."""
    return PreparedCall(*_decode("pkv_paged_decode_int8", out, query, k_codes, v_codes,
                                 k_scales, v_scales, block_tables, context_lens,
                                 max_context_len, softmax_scale, workspace, dev_status, stream),
                        keep=(out, query, k_codes, v_codes, k_scales, v_scales, block_tables,
                              context_lens, workspace, dev_status))


def prepare_paged_decode_fp8(out, query, k_codes, v_codes, k_scales, v_scales, block_tables,
                             context_lens, max_context_len, softmax_scale, workspace,
                             dev_status=None, stream=None) -> PreparedCall:
    """``pkv_paged_decode_fp8`` with its arguments marshalled once."""
    return PreparedCall(*_decode("pkv_paged_decode_fp8", out, query, k_codes, v_codes,
                                 k_scales, v_scales, block_tables, context_lens,
                                 max_context_len, softmax_scale, workspace, dev_status, stream),
                        keep=(out, query, k_codes, v_codes, k_scales, v_scales, block_tables,
                              context_lens, workspace, dev_status))


def decode_workspace(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len, device=None):
    """A uint8 CUDA tensor big enough to serve as a decode workspace."""
    import torch
    nbytes = pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                       max_context_len)
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device or "cuda")


def pkv_paged_decode_int8_static_workspace(out, query, k_codes, v_codes, k_scales, v_scales,
                                           block_tables, context_lens, max_context_len,
                                           softmax_scale, dev_status=None, stream=None) -> None:
    """INT8 decode for callers that cannot allocate: the scratch is a fixed
    array inside the library (PKV_STATIC_WORKSPACE_BYTES per device).  Calls
    that may overlap on the GPU must not use it concurrently."""
    import torch
    _check(out, "out", torch.float32)
    _check(query, "query", torch.float16)
    _check(k_codes, "k_codes", torch.int8)
    _check(v_codes, "v_codes", torch.int8)
    _check(k_scales, "k_scales", torch.float32)
    _check(v_scales, "v_scales", torch.float32)
    _check(block_tables, "block_tables", torch.int32)
    _check(context_lens, "context_lens", torch.int32)
    _check(dev_status, "dev_status", torch.int32)
    n, hq, d = query.shape
    nb, hkv, bs, _ = k_codes.shape
    mb = block_tables.shape[1] if block_tables.dim() == 2 else 0
    st = lib().pkv_paged_decode_int8_static_workspace(
        _ptr(out), _ptr(query), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales),
        nb, _ptr(block_tables), mb, _ptr(context_lens), int(max_context_len), n, hq, hkv, d, bs,
        float(softmax_scale), _ptr(dev_status), _stream(stream))
    if st != PKV_OK:
        raise PkvError(st, "pkv_paged_decode_int8_static_workspace")


def _append(fn_name, k_cache, v_cache, codes, k_new, v_new, block_tables, positions,
            dev_status, stream):
    import torch
    _check(k_cache, "k_cache", torch.float16)
    _check(v_cache, "v_cache", torch.float16)
    _check(k_new, "k_new", torch.float16)
    _check(v_new, "v_new", torch.float16)
    _check(block_tables, "block_tables", torch.int32)
    _check(positions, "positions", torch.int32)
    _check(dev_status, "dev_status", torch.int32)
    nb, hkv, bs, d = k_cache.shape
    n = positions.numel()
    mb = block_tables.shape[1] if block_tables is not None and block_tables.dim() == 2 else 0
    args = [_ptr(k_cache), _ptr(v_cache)]
    if codes is not None:
        kc, vc, ks, vs = codes
        code_t = torch.uint8 if fn_name.endswith("fp8") else torch.int8
        _check(kc, "k_codes", code_t)
        _check(vc, "v_codes", code_t)
        _check(ks, "k_scales", torch.float32)
        _check(vs, "v_scales", torch.float32)
        args += [_ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs)]
    args += [nb, _ptr(k_new), _ptr(v_new), _ptr(block_tables), mb, _ptr(positions), n, hkv, d,
             bs, _ptr(dev_status), _stream(stream)]
    st = getattr(lib(), fn_name)(*args)
    if st != PKV_OK:
        raise PkvError(st, fn_name)


def pkv_append_fp16(k_cache, v_cache, k_new, v_new, block_tables, positions, dev_status=None,
                    stream=None) -> None:
    """Write k_new/v_new [N][Hkv][d] at token positions[s] of each sequence
    (slot positions[s] % 16 of block block_tables[s][positions[s] // 16])."""
    _append("pkv_append_fp16", k_cache, v_cache, None, k_new, v_new, block_tables, positions,
            dev_status, stream)


def pkv_append_int8(k_cache, v_cache, k_codes, v_codes, k_scales, v_scales, k_new, v_new,
                    block_tables, positions, dev_status=None, stream=None) -> None:
    """pkv_append_fp16, then re-quantize every (block, kv head) tile written."""
    _append("pkv_append_int8", k_cache, v_cache, (k_codes, v_codes, k_scales, v_scales), k_new,
            v_new, block_tables, positions, dev_status, stream)


def pkv_append_fp8(k_cache, v_cache, k_codes, v_codes, k_scales, v_scales, k_new, v_new,
                   block_tables, positions, dev_status=None, stream=None) -> None:
    """pkv_append_fp16, then re-quantize every written tile to FP8 (E4M3)."""
    _append("pkv_append_fp8", k_cache, v_cache, (k_codes, v_codes, k_scales, v_scales), k_new,
            v_new, block_tables, positions, dev_status, stream)


def pkv_evict_select(refcnt, last_used, current_tick, k, evict_ids, num_evicted, scores=None,
                     alpha=EVICT_ALPHA, beta=EVICT_BETA, stream=None) -> None:
    """Score every block (refcnt int32 [NB], last_used int64 [NB]) and write
    the min(k, candidates) most evictable ids, ascending, to evict_ids[:n]
    (-1 after), n to num_evicted[0] and the fp32 scores to ``scores``."""
    import torch
    _check(refcnt, "refcnt", torch.int32)
    _check(last_used, "last_used", torch.int64)
    _check(evict_ids, "evict_ids", torch.int32)
    _check(num_evicted, "num_evicted", torch.int32)
    _check(scores, "scores", torch.float32)
    nb = refcnt.numel()
    if last_used.numel() != nb or (scores is not None and scores.numel() != nb):
        raise ValueError("refcnt, last_used and scores must have one entry per block")
    if evict_ids is not None and evict_ids.numel() < k:
        raise ValueError("evict_ids must hold k entries")
    st = lib().pkv_evict_select(_ptr(refcnt), _ptr(last_used), nb, int(current_tick),
                                float(alpha), float(beta), int(k), _ptr(scores),
                                _ptr(evict_ids), _ptr(num_evicted), _stream(stream))
    if st != PKV_OK:
        raise PkvError(st, "pkv_evict_select")


def evict_count(num_blocks: int, percent: int = 15) -> int:
    """Blocks to evict when a fixed percentage of the scored blocks goes:
    floor(num_blocks * percent / 100) in integer arithmetic."""
    if num_blocks < 0 or not 0 <= percent <= 100:
        raise ValueError("bad block count or percentage")
    return (int(num_blocks) * int(percent)) // 100


def _np_i32(x):
    import numpy as np
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32).reshape(-1))


class BlockManager:
    """The library's host block manager (``pkv_bm_*``).  Ids are numpy int32
    arrays; a failing call raises PkvError and changes nothing."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        h = ctypes.c_void_p()
        st = lib().pkv_bm_create(int(num_blocks), int(block_size), ctypes.byref(h))
        if st != PKV_OK:
            raise PkvError(st, "pkv_bm_create")
        self._h = h
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self):
        if getattr(self, "_h", None):
            lib().pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _call(self, name, *args):
        st = getattr(lib(), name)(self._h, *args)
        if st != PKV_OK:
            raise PkvError(st, name)

    def allocate(self, hashes):
        """hashes: an int (that many blocks, no hash) or a sequence of uint64
        prefix hashes (0 = none).  Returns the block ids."""
        import numpy as np
        if isinstance(hashes, int):
            n, hp = hashes, None
        else:
            hp = np.ascontiguousarray(np.asarray(hashes, dtype=np.uint64).reshape(-1))
            n = hp.size
        out = np.empty(n, np.int32)
        self._call("pkv_bm_allocate", None if hp is None else hp.ctypes.data, n,
                   out.ctypes.data)
        return out

    def free(self, ids):
        a = _np_i32(ids)
        self._call("pkv_bm_free", a.ctypes.data, a.size)

    def fork(self, ids):
        a = _np_i32(ids)
        self._call("pkv_bm_fork", a.ctypes.data, a.size)

    def cow(self, ids):
        """Returns (blocks to write, (source, copy) pairs int32 [k][2])."""
        import numpy as np
        a = _np_i32(ids)
        out = np.empty(a.size, np.int32)
        pairs = np.empty((a.size, 2), np.int32)
        k = ctypes.c_int(0)
        self._call("pkv_bm_cow", a.ctypes.data, a.size, out.ctypes.data, pairs.ctypes.data,
                   ctypes.byref(k))
        return out, pairs[:k.value].copy()

    def set_fill(self, ids, tokens):
        a, t = _np_i32(ids), _np_i32(tokens)
        if a.size != t.size:
            raise ValueError("ids and tokens differ in length")
        self._call("pkv_bm_set_fill", a.ctypes.data, t.ctypes.data, a.size)

    def stats(self) -> dict:
        st = BmStats()
        self._call("pkv_bm_stats", ctypes.byref(st))
        return {"free": st.free_blocks, "used": st.used_blocks, "shared": st.shared_blocks,
                "logical": st.logical_blocks, "tokens": st.tokens,
                "internal_fragmentation": st.internal_fragmentation,
                "sharing_saving": st.sharing_saving}

    def refcounts(self):
        import numpy as np
        out = np.empty(self.num_blocks, np.int32)
        self._call("pkv_bm_refcounts", out.ctypes.data, self.num_blocks)
        return out


def pkv_copy_blocks(pools, pairs, dev_status=None, stream=None) -> None:
    """Copy block pairs[i][0] to block pairs[i][1] in every pool (CUDA
    tensors shaped [num_blocks, ...], contiguous); pairs: int32 [n][2] CUDA."""
    import torch
    _check(pairs, "pairs", torch.int32)
    _check(dev_status, "dev_status", torch.int32)
    nb = pools[0].shape[0]
    ptrs = (ctypes.c_void_p * len(pools))()
    sizes = (ctypes.c_int64 * len(pools))()
    for i, t in enumerate(pools):
        _check(t, f"pools[{i}]")
        if t.shape[0] != nb:
            raise ValueError("all pools must have the same number of blocks")
        ptrs[i] = t.data_ptr()
        sizes[i] = (t.numel() // nb) * t.element_size()
    st = lib().pkv_copy_blocks(ptrs, sizes, len(pools), nb, _ptr(pairs),
                               0 if pairs is None else pairs.shape[0], _ptr(dev_status),
                               _stream(stream))
    if st != PKV_OK:
        raise PkvError(st, "pkv_copy_blocks")

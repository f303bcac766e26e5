"""CPU oracle for paged decode attention and the per-(block, kv-head) INT8 quantizer.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, links or
runs it, and it shares no code with that path: the two meet only through the
seeded inputs of ``pkv_workloads``.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64 attention, fp32
quantizer); this module only builds it with gcc and marshals numpy arrays.
Every function cites the passage it follows:

* ``decode_fp16`` / ``decode_int8`` -- gather through the block table
  ("PagedAttention & KV-Cache Memory Management", section 2.1), dense softmax
  attention with GQA ("paged-attention-runtime" summary, CORE CAPABILITIES 2
  and 4; PagedKV-Fusion README, Architecture, component B), INT8 values =
  code * per-(block, kv-head) scale (PagedKV-Fusion README, Overview and the
  Memory footprint table).
* ``quantize`` -- symmetric per-(block, head) INT8 (PagedKV-Fusion README,
  Overview component B; Architecture "per-block,head symmetric INT8"), with
  the absmax/127 scale and round-half-to-even reading.
* ``kv_pool_mib`` -- the storage arithmetic of the Memory footprint table.
* ``quantize_fp8`` / ``decode_fp8`` / ``e4m3_*`` -- per-block scaled FP8
  (OCP E4M3) keys and values ("PagedAttention & KV-Cache Memory Management",
  section 5.1), scale = amax / 448, decoded exactly.
* ``append_fp16`` / ``append_int8`` -- the write of one new token per
  sequence at slot table[s][t / B] * B + t % B ("PagedAttention & KV-Cache
  Memory Management", section 2.1 and the prefill step of its kernel
  mechanics; section 3.3.2, each step adding only its new tokens); the INT8 cache then
  re-quantizes every tile it wrote with ``quantize``.
* ``evict_scores`` / ``evict_select`` -- the least-reference-count + age
  score of "PagedAttention & KV-Cache Memory Management", section 4.3.1
  (alpha 0.7, beta 0.3), in fp32, and the choice of the k most evictable
  blocks (PagedKV-Fusion README: score every physical block, return the
  eviction ids).

* ``block_manager.BlockManagerModel`` -- the block manager (free list,
  reference counts, prefix sharing, copy-on-write, fragmentation figures) of
  the "paged-attention-runtime" summary (CORE CAPABILITIES 1) and of
  "PagedAttention & KV-Cache Memory Management" (the prefix-sharing allocator,
  section 4.1.1), as a plain Python model.

All functions here are pinned by tests in ``tests/test_oracle_pins.py``,
``tests/test_oracle_append_evict.py`` and ``tests/test_oracle_block_manager.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

BAD_BLOCK = 1
BAD_CTX = 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", "-fexcess-precision=standard",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.pkv_oracle_half_to_double.restype = ctypes.c_double
        lib.pkv_oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.pkv_oracle_decode.restype = ctypes.c_int
        lib.pkv_oracle_decode.argtypes = [
            P, P, ctypes.c_int, P, P, P, P, P, P,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
            ctypes.c_int, P]
        lib.pkv_oracle_quantize.restype = ctypes.c_int64
        lib.pkv_oracle_quantize.argtypes = [
            P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
            ctypes.c_int, ctypes.c_int]
        lib.pkv_oracle_quantize_fp8.restype = ctypes.c_int64
        lib.pkv_oracle_quantize_fp8.argtypes = lib.pkv_oracle_quantize.argtypes
        lib.pkv_oracle_e4m3_to_double.restype = ctypes.c_double
        lib.pkv_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.pkv_oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.pkv_oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.pkv_oracle_append.restype = ctypes.c_int64
        lib.pkv_oracle_append.argtypes = [
            P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int64, P, P]
        lib.pkv_oracle_evict_scores.restype = ctypes.c_int64
        lib.pkv_oracle_evict_scores.argtypes = [
            P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_float]
        lib.pkv_oracle_evict_select.restype = ctypes.c_int64
        lib.pkv_oracle_evict_select.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int64]
        lib.pkv_oracle_max_threads.restype = ctypes.c_int
        lib.pkv_oracle_max_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(bits: int) -> float:
    """Exact value of one IEEE binary16 bit pattern (plain bit decoding)."""
    return _load().pkv_oracle_half_to_double(int(bits) & 0xFFFF)


def max_threads() -> int:
    return _load().pkv_oracle_max_threads()


def _decode(kind, query, kpool, vpool, kscale, vscale, block_tables,
            context_lens, num_kv_heads, block_size, max_context_len,
            softmax_scale, num_threads, return_flags):
    lib = _load()
    q = _c(query, np.float16)
    n, hq, d = q.shape
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    if kind == 0:
        kp, vp = _c(kpool, np.float16), _c(vpool, np.float16)
        ks = vs = None
    else:
        cdt = np.int8 if kind == 1 else np.uint8
        kp, vp = _c(kpool, cdt), _c(vpool, cdt)
        ks, vs = _c(kscale, np.float32), _c(vscale, np.float32)
    nb = kp.shape[0]
    assert kp.shape == (nb, num_kv_heads, block_size, d) and vp.shape == kp.shape
    mb = bt.shape[1] if bt.ndim == 2 else 0
    if max_context_len is None:
        max_context_len = mb * block_size
    out = np.zeros((n, hq, d), dtype=np.float64)
    flags = np.zeros((n, hq), dtype=np.uint32)
    rc = lib.pkv_oracle_decode(
        _ptr(out), _ptr(q), kind, _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs),
        _ptr(bt), _ptr(ctx), n, hq, num_kv_heads, d, block_size, mb, nb,
        int(max_context_len), float(softmax_scale), int(num_threads), _ptr(flags))
    if rc != 0:
        raise ValueError("oracle rejected the decode arguments")
    return (out, flags) if return_flags else out


def decode_fp16(query, k_pool, v_pool, block_tables, context_lens, *,
                num_kv_heads, softmax_scale, block_size=16,
                max_context_len=None, num_threads=0, return_flags=False):
    """fp64 paged decode attention over fp16 K/V pools.

    query [N][Hq][d] fp16; pools [NB][Hkv][B][d] fp16; block_tables [N][MB]
    int32; context_lens [N] int32.  Returns out [N][Hq][d] float64 (and the
    per-(seq, head) flags when ``return_flags``).
    """
    return _decode(0, query, k_pool, v_pool, None, None, block_tables,
                   context_lens, num_kv_heads, block_size, max_context_len,
                   softmax_scale, num_threads, return_flags)


def decode_int8(query, k_codes, v_codes, k_scales, v_scales, block_tables,
                context_lens, *, num_kv_heads, softmax_scale, block_size=16,
                max_context_len=None, num_threads=0, return_flags=False):
    """fp64 paged decode attention over INT8 pools, value = code * scale."""
    return _decode(1, query, k_codes, v_codes, k_scales, v_scales, block_tables,
                   context_lens, num_kv_heads, block_size, max_context_len,
                   softmax_scale, num_threads, return_flags)


def quantize(pool, block_ids=None, code_pool=None, scales=None, inplace=False):
    """Symmetric per-(block, kv-head) INT8 quantization of an fp16 pool.

    pool [NB][Hkv][B][d] fp16.  block_ids: optional int32 ids (duplicates
    allowed); None means every block.  Returns (codes int8 like pool,
    scales float32 [NB][Hkv]); tiles not named by block_ids keep the values of
    ``code_pool`` / ``scales`` when given, else zeros.  With ``inplace`` the
    given (contiguous) ``code_pool`` and ``scales`` arrays are written.
    """
    lib = _load()
    x = _c(pool, np.float16)
    nb, hkv, bs, d = x.shape
    if inplace:
        codes, sc = code_pool, scales
        assert codes.flags.c_contiguous and codes.dtype == np.int8 and codes.shape == x.shape
        assert sc.flags.c_contiguous and sc.dtype == np.float32 and sc.shape == (nb, hkv)
    else:
        codes = np.zeros(x.shape, np.int8) if code_pool is None else _c(code_pool, np.int8).copy()
        sc = np.zeros((nb, hkv), np.float32) if scales is None else _c(scales, np.float32).copy()
    ids = None if block_ids is None else _c(block_ids, np.int32).reshape(-1)
    nids = 0 if ids is None else ids.size
    bad = lib.pkv_oracle_quantize(_ptr(codes), _ptr(sc), _ptr(x), _ptr(ids), nids,
                                  nb, hkv, bs, d)
    if bad < 0:
        raise ValueError("oracle rejected the quantize arguments")
    return codes, sc


def kv_pool_mib(num_blocks, num_heads, head_dim, kind, block_size=16):
    """MiB held by the K and V pools of one layer.

    kind "fp16": two pools of 2-byte values.  kind "int8": two pools of 1-byte
    codes plus one fp32 scale per (block, head) for K and one for V -- the
    granularity that the Memory footprint table of the PagedKV-Fusion README
    implies.
    """
    elems = num_blocks * num_heads * block_size * head_dim
    if kind == "fp16":
        nbytes = 2 * elems * 2
    elif kind == "int8":
        nbytes = 2 * elems * 1 + 2 * num_blocks * num_heads * 4
    else:
        raise ValueError(kind)
    return nbytes / float(1 << 20)


def append_fp16(k_pool, v_pool, k_new, v_new, block_tables, positions, *, inplace=False):
    """Write one new token per sequence into fp16 K/V pools.

    pools [NB][Hkv][B][d] fp16; k_new, v_new [N][Hkv][d] fp16; block_tables
    [N][MB] int32; positions [N] int32 (token index of the new token, < 0 =
    no token).  Returns (k_pool, v_pool, flags [N] uint32, written [N] int32
    = physical block written or -1).  With ``inplace`` the given contiguous
    fp16 pools are written.
    """
    lib = _load()
    if inplace:
        kp, vp = k_pool, v_pool
        for a in (kp, vp):
            assert a.flags.c_contiguous and a.dtype == np.float16
    else:
        kp, vp = _c(k_pool, np.float16).copy(), _c(v_pool, np.float16).copy()
    nb, hkv, bs, d = kp.shape
    assert vp.shape == kp.shape
    kn, vn = _c(k_new, np.float16), _c(v_new, np.float16)
    bt = _c(block_tables, np.int32)
    pos = _c(positions, np.int32).reshape(-1)
    n = pos.size
    assert kn.shape == (n, hkv, d) and vn.shape == kn.shape
    mb = bt.shape[1] if bt.ndim == 2 else 0
    assert bt.shape[0] == n or n == 0
    flags = np.zeros(n, np.uint32)
    written = np.full(n, -1, np.int32)
    rc = lib.pkv_oracle_append(_ptr(kp), _ptr(vp), _ptr(kn), _ptr(vn), _ptr(bt), _ptr(pos),
                               n, hkv, d, bs, mb, nb, _ptr(flags), _ptr(written))
    if rc < 0:
        raise ValueError("oracle rejected the append arguments")
    return kp, vp, flags, written


def append_int8(k_pool, v_pool, k_codes, v_codes, k_scales, v_scales, k_new, v_new,
                block_tables, positions, *, inplace=False):
    """Append into the fp16 pools, then re-quantize every written tile.

    Returns (k_pool, v_pool, k_codes, v_codes, k_scales, v_scales, flags):
    the fp16 pools after ``append_fp16`` and the INT8 pools in which the
    (written block, every kv head) tiles are the ``quantize`` of the new fp16
    tiles; all other tiles keep their codes and scales.
    """
    kp, vp, flags, written = append_fp16(k_pool, v_pool, k_new, v_new, block_tables,
                                         positions, inplace=inplace)
    ids = written[written >= 0]
    if inplace:
        quantize(kp, block_ids=ids, code_pool=k_codes, scales=k_scales, inplace=True)
        quantize(vp, block_ids=ids, code_pool=v_codes, scales=v_scales, inplace=True)
        kc, ks, vc, vs = k_codes, k_scales, v_codes, v_scales
    else:
        kc, ks = quantize(kp, block_ids=ids, code_pool=k_codes, scales=k_scales)
        vc, vs = quantize(vp, block_ids=ids, code_pool=v_codes, scales=v_scales)
    return kp, vp, kc, vc, ks, vs, flags


def append_fp8(k_pool, v_pool, k_codes, v_codes, k_scales, v_scales, k_new, v_new,
               block_tables, positions):
    """``append_fp16``, then ``quantize_fp8`` of every written tile (other
    tiles keep their codes and scales)."""
    kp, vp, flags, written = append_fp16(k_pool, v_pool, k_new, v_new, block_tables, positions)
    ids = written[written >= 0]
    kc, ks = quantize_fp8(kp, block_ids=ids, code_pool=k_codes, scales=k_scales)
    vc, vs = quantize_fp8(vp, block_ids=ids, code_pool=v_codes, scales=v_scales)
    return kp, vp, kc, vc, ks, vs, flags


EVICT_ALPHA = 0.7  # weights of the least-reference-count + age score
EVICT_BETA = 0.3


def evict_scores(refcnt, last_used, current_tick, alpha=EVICT_ALPHA, beta=EVICT_BETA):
    """fp32 eviction score of every block; -inf for free (refcnt <= 0) blocks.

    Returns (scores float32 [NB], number of candidate blocks).
    """
    lib = _load()
    rc = _c(refcnt, np.int32).reshape(-1)
    lu = _c(last_used, np.int64).reshape(-1)
    assert rc.size == lu.size
    scores = np.empty(rc.size, np.float32)
    cand = lib.pkv_oracle_evict_scores(_ptr(scores), _ptr(rc), _ptr(lu), rc.size,
                                       int(current_tick), float(alpha), float(beta))
    return scores, int(cand)


def evict_select(refcnt, last_used, current_tick, k, alpha=EVICT_ALPHA, beta=EVICT_BETA):
    """The min(k, candidates) most evictable blocks, in ascending id order.

    Returns (ids int32 [n], scores float32 [NB]).
    """
    lib = _load()
    scores, _ = evict_scores(refcnt, last_used, current_tick, alpha, beta)
    rc = _c(refcnt, np.int32).reshape(-1)
    ids = np.empty(max(int(k), 0) + 1, np.int32)
    n = lib.pkv_oracle_evict_select(_ptr(ids), _ptr(scores), _ptr(rc), rc.size, int(k))
    if n < 0:
        raise ValueError("oracle rejected the eviction arguments")
    return ids[:n].copy(), scores


def decode_fp8(query, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, *,
               num_kv_heads, softmax_scale, block_size=16, max_context_len=None,
               num_threads=0, return_flags=False):
    """fp64 paged decode attention over FP8 (E4M3 bytes) pools,
    value = e4m3(code) * scale ("PagedAttention & KV-Cache Memory
    Management", section 5.1)."""
    return _decode(2, query, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens,
                   num_kv_heads, block_size, max_context_len, softmax_scale, num_threads,
                   return_flags)


def e4m3_to_double(code: int) -> float:
    return _load().pkv_oracle_e4m3_to_double(int(code) & 0xFF)


def e4m3_from_float(y: float) -> int:
    """Nearest finite E4M3 code of a non-NaN fp32 value (ties to even,
    saturating at +-448)."""
    return int(_load().pkv_oracle_e4m3_from_float(float(y)))


def quantize_fp8(pool, block_ids=None, code_pool=None, scales=None, inplace=False):
    """Per-(block, kv-head) FP8 E4M3 quantization of an fp16 pool: scale =
    fp32 amax / 448, code = E4M3 of the fp32 quotient x / scale (a NaN
    quotient gives 0).  Arguments and results as ``quantize`` with uint8
    codes."""
    lib = _load()
    x = _c(pool, np.float16)
    nb, hkv, bs, d = x.shape
    if inplace:
        codes, sc = code_pool, scales
        assert codes.flags.c_contiguous and codes.dtype == np.uint8 and codes.shape == x.shape
        assert sc.flags.c_contiguous and sc.dtype == np.float32 and sc.shape == (nb, hkv)
    else:
        codes = np.zeros(x.shape, np.uint8) if code_pool is None else _c(code_pool, np.uint8).copy()
        sc = np.zeros((nb, hkv), np.float32) if scales is None else _c(scales, np.float32).copy()
    ids = None if block_ids is None else _c(block_ids, np.int32).reshape(-1)
    nids = 0 if ids is None else ids.size
    bad = lib.pkv_oracle_quantize_fp8(_ptr(codes), _ptr(sc), _ptr(x), _ptr(ids), nids,
                                      nb, hkv, bs, d)
    if bad < 0:
        raise ValueError("oracle rejected the quantize arguments")
    return codes, sc

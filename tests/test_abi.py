"""The C-ABI library builds, loads and exports every declared call; host-side
argument checks return the documented status codes without touching a GPU.

Nothing here launches a kernel or makes a CUDA call: every case below is
rejected (or is a no-op) before the library reaches the CUDA runtime.
"""
import ctypes
import os
import re

import pytest

import paged_kv_cache_234_gb300 as pkv
from paged_kv_cache_234_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def L():
    pkv_build.build()
    return pkv.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pkv_quantize_blocks", "pkv_paged_decode_fp16", "pkv_paged_decode_int8"):
        assert required in names
    assert set(names) == set(pkv.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_c_program_uses_the_abi(L):
    # include/pkv.h compiled as C99 and libpkv.so linked by the system linker:
    # the host-only calls of tests/c_abi/abi_smoke.c (no GPU needed)
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    exe = os.path.join(pkv_build.BUILD_DIR, "abi_smoke")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.dirname(HEADER), os.path.join(here, "c_abi", "abi_smoke.c"),
                        "-L", pkv_build.BUILD_DIR, "-lpkv", "-Wl,-rpath," + pkv_build.BUILD_DIR,
                        "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "C ABI checks passed" in r.stdout, r.stdout + r.stderr


def test_status_strings(L):
    for code in range(6):
        assert pkv.pkv_status_string(code)
    assert pkv.pkv_status_string(0) == "ok"
    assert pkv.pkv_status_string(99) == "unknown status"


def test_workspace_size_arithmetic(L):
    # per worker: two partial records of min(item heads, group) heads x
    # (d + 4) floats, an item holding 8 query heads, or 16 when a kv head has
    # more than 8; at most 4096 workers and never more than the pages.
    def expect(workers, heads, d):
        return workers * 2 * heads * (d + 4) * 4
    assert pkv.pkv_decode_workspace_size(64, 32, 8, 128, 2048) == expect(4096, 4, 128)
    assert pkv.pkv_decode_workspace_size(2, 8, 2, 64, 37) == expect(2 * 2 * 3, 4, 64)
    assert pkv.pkv_decode_workspace_size(8, 8, 8, 128, 512) == expect(2048, 1, 128)
    assert pkv.pkv_decode_workspace_size(1, 32, 1, 128, 16) == expect(2, 16, 128)
    assert pkv.pkv_decode_workspace_size(3, 12, 1, 64, 16) == expect(3, 12, 64)
    assert pkv.pkv_decode_workspace_size(4, 8, 3, 128, 16) == 0      # heads not divisible
    assert pkv.pkv_decode_workspace_size(4, 8, 2, 96, 16) == 0       # unsupported head_dim
    assert pkv.pkv_decode_workspace_size(0, 8, 2, 64, 0) == 0


FAKE = 0x10000  # an aligned, never-dereferenced address


def _decode(L, int8=False, **kw):
    a = dict(out=FAKE, query=FAKE, k=FAKE, v=FAKE, ks=FAKE, vs=FAKE, num_blocks=16,
             tables=FAKE, mb=4, lens=FAKE, max_ctx=64, n=2, hq=8, hkv=2, d=64, bs=16,
             scale=0.125, ws=FAKE, ws_bytes=1 << 30, status=None, stream=None)
    a.update(kw)
    head = [a["out"], a["query"], a["k"], a["v"]]
    if int8:
        head += [a["ks"], a["vs"]]
    args = head + [a["num_blocks"], a["tables"], a["mb"], a["lens"], a["max_ctx"], a["n"],
                   a["hq"], a["hkv"], a["d"], a["bs"], a["scale"], a["ws"], a["ws_bytes"],
                   a["status"], a["stream"]]
    fn = L.pkv_paged_decode_int8 if int8 else L.pkv_paged_decode_fp16
    return fn(*args)


@pytest.mark.parametrize("int8", [False, True])
def test_decode_host_validation(L, int8):
    assert _decode(L, int8, out=None) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, int8, tables=None) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, int8, hq=7) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, int8, n=-1) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, int8, scale=float("nan")) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(L, int8, d=96) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(L, int8, bs=32) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(L, int8, n=9000) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(L, int8, k=FAKE + 4) == pkv.PKV_ERR_MISALIGNED
    assert _decode(L, int8, out=FAKE + 8) == pkv.PKV_ERR_MISALIGNED
    assert _decode(L, int8, ws_bytes=100) == pkv.PKV_ERR_WORKSPACE
    assert _decode(L, int8, ws=None) == pkv.PKV_ERR_WORKSPACE
    assert _decode(L, int8, n=0) == pkv.PKV_OK  # nothing to do, nothing launched
    if int8:
        assert _decode(L, int8, ks=None) == pkv.PKV_ERR_INVALID_ARG
        assert _decode(L, int8, vs=FAKE + 2) == pkv.PKV_ERR_MISALIGNED


def test_fp8_entry_points_host_validation(L):
    # decode: same argument rules as INT8
    a = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, FAKE, 4, FAKE, 64, 2, 8, 2, 64, 16, 0.125,
         FAKE, 1 << 30, None, None]
    def dec(i=None, v=None):
        b = list(a)
        if i is not None:
            b[i] = v
        return L.pkv_paged_decode_fp8(*b)
    assert dec(0, None) == pkv.PKV_ERR_INVALID_ARG          # out
    assert dec(4, None) == pkv.PKV_ERR_INVALID_ARG          # k_scales
    assert dec(14, 96) == pkv.PKV_ERR_UNSUPPORTED           # head_dim
    assert dec(2, FAKE + 4) == pkv.PKV_ERR_MISALIGNED       # k_codes
    assert dec(18, 100) == pkv.PKV_ERR_WORKSPACE
    assert dec(11, 0) == pkv.PKV_OK                         # no sequences, nothing launched
    # quantize
    q = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 16, 2, 64, 16, None, None]
    def qz(i=None, v=None):
        b = list(q)
        if i is not None:
            b[i] = v
        return L.pkv_quantize_blocks_fp8(*b)
    assert qz(2, None) == pkv.PKV_ERR_INVALID_ARG
    assert qz(10, 96) == pkv.PKV_ERR_UNSUPPORTED
    assert qz(3, FAKE + 1) == pkv.PKV_ERR_MISALIGNED
    assert qz(6, FAKE) == pkv.PKV_OK                        # empty id list
    # append
    ap = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, FAKE, FAKE, FAKE, 4, FAKE, 2, 2, 64, 16, None,
          None]
    def app(i=None, v=None):
        b = list(ap)
        if i is not None:
            b[i] = v
        return L.pkv_append_fp8(*b)
    assert app(4, None) == pkv.PKV_ERR_INVALID_ARG
    assert app(3, FAKE + 8) == pkv.PKV_ERR_MISALIGNED
    assert app(12, 0) == pkv.PKV_OK


def test_block_manager_null_handle_and_arguments(L):
    assert L.pkv_bm_create(4, 16, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_bm_allocate(None, None, 1, FAKE) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_bm_free(None, FAKE, 1) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_bm_stats(None, None) == pkv.PKV_ERR_INVALID_ARG
    bm = pkv.BlockManager(4)
    assert L.pkv_bm_allocate(bm._h, None, -1, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_bm_allocate(bm._h, None, 2, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_bm_refcounts(bm._h, None, 4) == pkv.PKV_ERR_INVALID_ARG
    bm.close()
    L.pkv_bm_destroy(None)  # a no-op


def test_quantize_host_validation(L):
    def q(**kw):
        a = dict(k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE, ids=None, nids=0,
                 nb=16, hkv=2, d=64, bs=16, status=None, stream=None)
        a.update(kw)
        return L.pkv_quantize_blocks(a["k"], a["v"], a["kc"], a["vc"], a["ks"], a["vs"],
                                     a["ids"], a["nids"], a["nb"], a["hkv"], a["d"], a["bs"],
                                     a["status"], a["stream"])
    assert q(k=None) == pkv.PKV_ERR_INVALID_ARG
    assert q(nb=0) == pkv.PKV_ERR_INVALID_ARG
    assert q(nids=-1) == pkv.PKV_ERR_INVALID_ARG
    assert q(d=96) == pkv.PKV_ERR_UNSUPPORTED
    assert q(bs=8) == pkv.PKV_ERR_UNSUPPORTED
    assert q(kc=FAKE + 1) == pkv.PKV_ERR_MISALIGNED
    assert q(ids=FAKE, nids=0) == pkv.PKV_OK  # empty id list: nothing launched


def test_append_host_validation(L):
    def a(int8=False, **kw):
        x = dict(k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE, nb=16, kn=FAKE, vn=FAKE,
                 tables=FAKE, mb=4, pos=FAKE, n=2, hkv=2, d=64, bs=16, status=None, stream=None)
        x.update(kw)
        head = [x["k"], x["v"]]
        if int8:
            head += [x["kc"], x["vc"], x["ks"], x["vs"]]
        args = head + [x["nb"], x["kn"], x["vn"], x["tables"], x["mb"], x["pos"], x["n"],
                       x["hkv"], x["d"], x["bs"], x["status"], x["stream"]]
        return (L.pkv_append_int8 if int8 else L.pkv_append_fp16)(*args)
    for int8 in (False, True):
        assert a(int8, k=None) == pkv.PKV_ERR_INVALID_ARG
        assert a(int8, pos=None) == pkv.PKV_ERR_INVALID_ARG
        assert a(int8, tables=None) == pkv.PKV_ERR_INVALID_ARG
        assert a(int8, nb=0) == pkv.PKV_ERR_INVALID_ARG
        assert a(int8, n=-1) == pkv.PKV_ERR_INVALID_ARG
        assert a(int8, d=96) == pkv.PKV_ERR_UNSUPPORTED
        assert a(int8, bs=8) == pkv.PKV_ERR_UNSUPPORTED
        assert a(int8, kn=FAKE + 8) == pkv.PKV_ERR_MISALIGNED
        assert a(int8, pos=FAKE + 2) == pkv.PKV_ERR_MISALIGNED
        assert a(int8, n=0) == pkv.PKV_OK  # nothing launched
    assert a(True, ks=None) == pkv.PKV_ERR_INVALID_ARG
    assert a(True, vc=FAKE + 4) == pkv.PKV_ERR_MISALIGNED


def test_evict_host_validation(L):
    def e(**kw):
        x = dict(ref=FAKE, last=FAKE, nb=1024, tick=10, alpha=0.7, beta=0.3, k=5, scores=None,
                 ids=FAKE, count=FAKE, stream=None)
        x.update(kw)
        return L.pkv_evict_select(x["ref"], x["last"], x["nb"], x["tick"], x["alpha"],
                                  x["beta"], x["k"], x["scores"], x["ids"], x["count"],
                                  x["stream"])
    assert e(k=-1) == pkv.PKV_ERR_INVALID_ARG
    assert e(nb=-1) == pkv.PKV_ERR_INVALID_ARG
    assert e(count=None) == pkv.PKV_ERR_INVALID_ARG
    assert e(ref=None) == pkv.PKV_ERR_INVALID_ARG
    assert e(ids=None) == pkv.PKV_ERR_INVALID_ARG
    assert e(alpha=float("nan")) == pkv.PKV_ERR_INVALID_ARG
    assert e(beta=float("inf")) == pkv.PKV_ERR_INVALID_ARG
    assert e(last=FAKE + 4) == pkv.PKV_ERR_MISALIGNED
    assert e(scores=FAKE + 2) == pkv.PKV_ERR_MISALIGNED


def test_copy_blocks_host_validation(L):
    P2 = ctypes.c_void_p * 2
    S2 = ctypes.c_int64 * 2
    def c(pools=(FAKE, FAKE), sizes=(4096, 32), n=2, nb=16, pairs=FAKE, npairs=3):
        return L.pkv_copy_blocks(P2(*pools), S2(*sizes), n, nb, pairs, npairs, None, None)
    assert c(n=0) == pkv.PKV_ERR_INVALID_ARG
    assert c(nb=0) == pkv.PKV_ERR_INVALID_ARG
    assert c(npairs=-1) == pkv.PKV_ERR_INVALID_ARG
    assert c(pairs=None) == pkv.PKV_ERR_INVALID_ARG
    assert c(pools=(FAKE, None)) == pkv.PKV_ERR_INVALID_ARG
    assert c(sizes=(4096, 0)) == pkv.PKV_ERR_INVALID_ARG
    assert c(sizes=(4096, 30)) == pkv.PKV_ERR_MISALIGNED
    assert c(pools=(FAKE + 2, FAKE)) == pkv.PKV_ERR_MISALIGNED
    assert c(n=9) == pkv.PKV_ERR_UNSUPPORTED
    assert c(npairs=0) == pkv.PKV_OK  # nothing launched


# The PagedKV-Fusion README's end-to-end demos evict 15 % of the scored
# blocks: 173 of 1155 (CPU reference) and 85 of 568 (CUDA run).
def test_evict_count_matches_the_pages_examples():
    assert pkv.evict_count(1155) == 173
    assert pkv.evict_count(568) == 85
    assert pkv.evict_count(0) == 0 and pkv.evict_count(100, 100) == 100


def test_set_decode_workers_rejects_negative(L):
    assert L.pkv_set_decode_workers(-1) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_set_decode_workers(0) == pkv.PKV_OK


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_234_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "pkv_oracle" not in text, f

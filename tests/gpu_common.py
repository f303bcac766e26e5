"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding on seeded inputs and compare with the CPU oracle."""
import numpy as np
import torch

import oracle
import paged_kv_cache_234_gb300 as pkv
from paged_kv_cache_234_gb300 import build as pkv_build

# Tolerances of the decode outputs against the fp64 oracle on identical inputs.
MAX_ABS = 2e-3
REL_L2 = 1e-3

_built = False


def ensure_built():
    global _built
    if not _built:
        pkv_build.build()
        pkv.lib()
        _built = True


class persistent_workers:
    """Within the block, decode calls use the persistent-worker partition
    (split-context pieces merged by the reduce kernel) even for batches that
    would take the one-item-per-cluster launch: a worker cap set through
    pkv_set_decode_workers selects the persistent partition."""

    def __init__(self, cap=4096):
        self.cap = cap

    def __enter__(self):
        ensure_built()
        pkv.pkv_set_decode_workers(self.cap)
        return self

    def __exit__(self, *exc):
        pkv.pkv_set_decode_workers(0)
        return False


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def oracle_codes(w, fp8=False):
    """INT8 (or FP8) pools + scales from the oracle quantizer (used blocks only)."""
    q = oracle.quantize_fp8 if fp8 else oracle.quantize
    kc, ks = q(w.k_pool, block_ids=w.used_block_ids)
    vc, vs = q(w.v_pool, block_ids=w.used_block_ids)
    return kc, vc, ks, vs


def gpu_decode(w, variant, codes=None, max_context_len=None, tables=None, lens=None,
               stream=None):
    """Run one decode call; returns (out as float64 numpy, device status word)."""
    ensure_built()
    n, hq, d = w.query.shape
    mcl = w.max_context_len if max_context_len is None else max_context_len
    q = dev(w.query)
    bt = dev(w.block_tables if tables is None else tables)
    cl = dev(w.context_lens if lens is None else lens)
    out = torch.full((n, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, mcl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if variant == "fp16":
        pkv.pkv_paged_decode_fp16(out, q, dev(w.k_pool), dev(w.v_pool), bt, cl, mcl,
                                  w.softmax_scale, ws, status, stream=stream)
    else:
        kc, vc, ks, vs = codes if codes is not None else oracle_codes(w, variant == "fp8")
        fn = pkv.pkv_paged_decode_fp8 if variant == "fp8" else pkv.pkv_paged_decode_int8
        fn(out, q, dev(kc), dev(vc), dev(ks), dev(vs), bt, cl, mcl, w.softmax_scale, ws, status,
           stream=stream)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), int(status.item())


def oracle_decode(w, variant, codes=None, max_context_len=None, tables=None, lens=None):
    mcl = w.max_context_len if max_context_len is None else max_context_len
    bt = w.block_tables if tables is None else tables
    cl = w.context_lens if lens is None else lens
    if variant == "fp16":
        return oracle.decode_fp16(w.query, w.k_pool, w.v_pool, bt, cl,
                                  num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                                  max_context_len=mcl, return_flags=True)
    kc, vc, ks, vs = codes if codes is not None else oracle_codes(w, variant == "fp8")
    fn = oracle.decode_fp8 if variant == "fp8" else oracle.decode_int8
    return fn(w.query, kc, vc, ks, vs, bt, cl, num_kv_heads=w.num_kv_heads,
              softmax_scale=w.softmax_scale, max_context_len=mcl, return_flags=True)


def assert_close(got, ref, what=""):
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / denom if denom > 0 else float(np.linalg.norm(got))
    assert max_abs <= MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {MAX_ABS}"
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    return max_abs, rel

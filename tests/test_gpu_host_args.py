"""Per-step arguments in pinned host memory.

The decode calls' query, block tables, context lengths and output, and the
quantizer's block ids, may be pinned host tensors: pinned memory has one
address for the host and the GPU, so the kernels read and write them in place
over the GPU's link to the host, with no copy operation.  The results must be
bit for bit those of the same calls with device tensors, and match the
oracle.  The KV pools, scales and workspace stay in device memory.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import assert_close, dev, ensure_built, oracle_codes, oracle_decode

pytestmark = pytest.mark.gpu


def pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


@pytest.mark.parametrize("variant", ["fp16", "int8"])
@pytest.mark.parametrize("case", ["cluster", "persistent"])
def test_decode_with_host_resident_step_arguments(variant, case):
    ensure_built()
    if case == "cluster":   # a small batch: one item per cluster
        w = W.random_case(401, num_seqs=5, num_heads=8, num_kv_heads=2, head_dim=128,
                          context_lens=[1, 40, 300, 17, 512])
    else:                   # the persistent workers + reduce
        w = W.random_case(402, num_seqs=24, num_heads=32, num_kv_heads=8, head_dim=128,
                          max_ctx=1200)
    n, hq, d = w.query.shape
    mcl = w.max_context_len
    codes = None if variant == "fp16" else oracle_codes(w)
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, mcl)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if variant == "fp16":
        pools = (dev(w.k_pool), dev(w.v_pool))
        call = pkv.pkv_paged_decode_fp16
    else:
        pools = tuple(dev(x) for x in codes)
        call = pkv.pkv_paged_decode_int8
    out_d = torch.empty((n, hq, d), dtype=torch.float32, device="cuda")
    call(out_d, dev(w.query), *pools, dev(w.block_tables), dev(w.context_lens), mcl,
         w.softmax_scale, ws, st)
    out_h = torch.full((n, hq, d), float("nan"), dtype=torch.float32).pin_memory()
    call(out_h, pinned(w.query), *pools, pinned(w.block_tables), pinned(w.context_lens), mcl,
         w.softmax_scale, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out_h.numpy()
    assert np.array_equal(got.view(np.uint32), out_d.cpu().numpy().view(np.uint32))
    ref, _ = oracle_decode(w, variant, codes)
    assert_close(got.astype(np.float64), ref, f"host arguments {variant}/{case}")


def test_quantize_with_host_resident_block_ids():
    ensure_built()
    w = W.random_case(403, num_seqs=6, num_heads=8, num_kv_heads=2, head_dim=64, max_ctx=200)
    kf, vf = dev(w.k_pool), dev(w.v_pool)
    kc = torch.zeros(w.k_pool.shape, dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros(w.k_pool.shape[:2], dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, pinned(w.used_block_ids))
    rkc, rks = oracle.quantize(w.k_pool, block_ids=w.used_block_ids)
    rvc, rvs = oracle.quantize(w.v_pool, block_ids=w.used_block_ids)
    torch.cuda.synchronize()
    assert np.array_equal(kc.cpu().numpy(), rkc) and np.array_equal(vc.cpu().numpy(), rvc)
    assert np.array_equal(ks.cpu().numpy(), rks) and np.array_equal(vs.cpu().numpy(), rvs)


def test_pageable_host_tensors_are_refused():
    ensure_built()
    w = W.random_case(404, num_seqs=2, num_heads=8, num_kv_heads=2, head_dim=64,
                      context_lens=[20, 3])
    n, hq, d = w.query.shape
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, w.max_context_len)
    out = torch.empty((n, hq, d), dtype=torch.float32)   # pageable: not accepted
    with pytest.raises(ValueError):
        pkv.pkv_paged_decode_fp16(out, dev(w.query), dev(w.k_pool), dev(w.v_pool),
                                  dev(w.block_tables), dev(w.context_lens), w.max_context_len,
                                  w.softmax_scale, ws)

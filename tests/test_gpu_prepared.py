"""Prepared calls: arguments checked and marshalled once, the C call issued again.

A PreparedCall must give bit for bit what the plain binding call gives on the
same buffers, and must follow changes made in place to those buffers between
calls (a serving loop rewrites its query, block tables and context lengths
every step): after such an update it matches the plain call and the oracle on
the updated inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import assert_close, dev, ensure_built, oracle_codes, oracle_decode

pytestmark = pytest.mark.gpu


def _case(case, seed):
    if case == "cluster":   # a small batch: one item per cluster
        return W.random_case(seed, num_seqs=5, num_heads=8, num_kv_heads=2, head_dim=128,
                             context_lens=[1, 40, 300, 17, 512])
    return W.random_case(seed, num_seqs=24, num_heads=32, num_kv_heads=8, head_dim=128,
                         max_ctx=1200)


@pytest.mark.parametrize("variant", ["fp16", "int8", "fp8"])
@pytest.mark.parametrize("case", ["cluster", "persistent"])
def test_prepared_decode_matches_and_follows_in_place_updates(variant, case):
    ensure_built()
    w = _case(case, 501)
    n, hq, d = w.query.shape
    mcl = w.max_context_len
    codes = None if variant == "fp16" else oracle_codes(w, variant == "fp8")
    pools = (dev(w.k_pool), dev(w.v_pool)) if codes is None else tuple(dev(x) for x in codes)
    plain = {"fp16": pkv.pkv_paged_decode_fp16, "int8": pkv.pkv_paged_decode_int8,
             "fp8": pkv.pkv_paged_decode_fp8}[variant]
    prep = {"fp16": pkv.prepare_paged_decode_fp16, "int8": pkv.prepare_paged_decode_int8,
            "fp8": pkv.prepare_paged_decode_fp8}[variant]
    q, bt, cl = dev(w.query), dev(w.block_tables), dev(w.context_lens)
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, mcl)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_p = torch.full((n, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    out_q = torch.full_like(out_p, float("nan"))
    call = prep(out_p, q, *pools, bt, cl, mcl, w.softmax_scale, ws, st)
    call()
    plain(out_q, q, *pools, bt, cl, mcl, w.softmax_scale, ws, st)
    torch.cuda.synchronize()
    assert torch.equal(out_p.view(torch.int32), out_q.view(torch.int32))

    # the next step: new queries and shorter contexts, written in place
    rng = np.random.default_rng(502)
    w.query[:] = rng.standard_normal(w.query.shape).astype(np.float16)
    w.context_lens[:] = np.maximum(w.context_lens - rng.integers(0, 20, n), 0).astype(np.int32)
    q.copy_(torch.from_numpy(w.query))
    cl.copy_(torch.from_numpy(w.context_lens))
    call()
    plain(out_q, q, *pools, bt, cl, mcl, w.softmax_scale, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out_p.view(torch.int32), out_q.view(torch.int32))
    ref, _ = oracle_decode(w, variant, codes)
    assert_close(out_p.cpu().numpy().astype(np.float64), ref, f"prepared {variant}/{case}")


@pytest.mark.parametrize("fp8", [False, True])
def test_prepared_quantize_matches_plain_call(fp8):
    ensure_built()
    w = W.random_case(503, num_seqs=6, num_heads=8, num_kv_heads=2, head_dim=64, max_ctx=200)
    kf, vf = dev(w.k_pool), dev(w.v_pool)
    cdt = torch.uint8 if fp8 else torch.int8
    outs = []
    for prepared in (True, False):
        kc = torch.zeros(w.k_pool.shape, dtype=cdt, device="cuda")
        vc = torch.zeros_like(kc)
        ks = torch.zeros(w.k_pool.shape[:2], dtype=torch.float32, device="cuda")
        vs = torch.zeros_like(ks)
        ids = dev(w.used_block_ids)
        if prepared:
            prep = pkv.prepare_quantize_blocks_fp8 if fp8 else pkv.prepare_quantize_blocks
            prep(kf, vf, kc, vc, ks, vs, ids)()
        else:
            (pkv.pkv_quantize_blocks_fp8 if fp8 else pkv.pkv_quantize_blocks)(
                kf, vf, kc, vc, ks, vs, ids)
        outs.append([t.cpu().numpy() for t in (kc, vc, ks, vs)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    if not fp8:
        rkc, rks = oracle.quantize(w.k_pool, block_ids=w.used_block_ids)
        assert np.array_equal(outs[0][0], rkc) and np.array_equal(outs[0][2], rks)


def test_prepared_call_reports_errors_when_called():
    # sizes are checked by the library at each call: a workspace too small
    # for the persistent launch is refused when the prepared call runs
    ensure_built()
    w = _case("persistent", 505)
    n, hq, d = w.query.shape
    out = torch.empty((n, hq, d), dtype=torch.float32, device="cuda")
    q, kp, vp = dev(w.query), dev(w.k_pool), dev(w.v_pool)
    bt, cl = dev(w.block_tables), dev(w.context_lens)
    tiny_ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    call = pkv.prepare_paged_decode_fp16(out, q, kp, vp, bt, cl, w.max_context_len,
                                         w.softmax_scale, tiny_ws)
    with pytest.raises(pkv.PkvError) as e:
        call()
    assert e.value.status == pkv.PKV_ERR_WORKSPACE


@pytest.mark.parametrize("case", ["cluster", "persistent"])
def test_prepared_decode_with_host_resident_step_arguments(case):
    # query, block tables, context lengths and output in pinned host memory,
    # read and written in place by the kernels: the same bits as device tensors
    ensure_built()
    w = _case(case, 506)
    n, hq, d = w.query.shape
    mcl = w.max_context_len
    codes = tuple(dev(x) for x in oracle_codes(w))
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, mcl)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    q_h, bt_h, cl_h = pin(w.query), pin(w.block_tables), pin(w.context_lens)
    out_h = torch.full((n, hq, d), float("nan"), dtype=torch.float32).pin_memory()
    out_d = torch.full((n, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    host = pkv.prepare_paged_decode_int8(out_h, q_h, *codes, bt_h, cl_h, mcl, w.softmax_scale, ws)
    devc = pkv.prepare_paged_decode_int8(out_d, dev(w.query), *codes, dev(w.block_tables),
                                         dev(w.context_lens), mcl, w.softmax_scale, ws)
    host()
    devc()
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int32), out_d.cpu().view(torch.int32))

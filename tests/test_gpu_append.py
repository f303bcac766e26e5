"""Token append on the GPU against the CPU oracle: fp16 pools bit-exact, INT8
codes and scales of the re-quantized tiles bit-exact, everything else left
untouched, and a whole decode step (append, then attention over the new
context) within the decode tolerance of the oracle's fp64 result."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import assert_close, dev, ensure_built, oracle_codes

pytestmark = pytest.mark.gpu


def gpu_append(kp, vp, kn, vn, tables, pos, codes=None, fp8=False):
    """Run one append on device copies; returns device tensors and the status."""
    ensure_built()
    kd, vd = dev(kp), dev(vp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (dev(kn), dev(vn), dev(tables), dev(pos))
    if codes is None:
        pkv.pkv_append_fp16(kd, vd, *args, dev_status=status)
        dc = None
    else:
        dc = tuple(dev(c) for c in codes)
        fn = pkv.pkv_append_fp8 if fp8 else pkv.pkv_append_int8
        fn(kd, vd, *dc, *args, dev_status=status)
    torch.cuda.synchronize()
    return kd, vd, dc, int(status.item())


def same_bits(gpu_t, ref):
    g = gpu_t.cpu().numpy()
    if g.dtype == np.float16:
        return np.array_equal(g.view(np.uint16), np.ascontiguousarray(ref).view(np.uint16))
    if g.dtype == np.float32:
        return np.array_equal(g.view(np.uint32), np.ascontiguousarray(ref).view(np.uint32))
    return np.array_equal(g, ref)


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (32, 8, 128), (14, 2, 64), (8, 8, 128)])
def test_append_fp16_and_int8_bit_exact(hq, hkv, d):
    lens = [1, 15, 16, 17, 0, 33, 255, 256, 257, 48]
    w = W.random_case(500 + d + hq, num_seqs=len(lens), num_heads=hq, num_kv_heads=hkv,
                      head_dim=d, context_lens=lens)
    kn, vn, pos = W.append_tokens(w, 21)
    rk, rv, flags, _ = oracle.append_fp16(w.k_pool, w.v_pool, kn, vn, w.block_tables, pos)
    assert not flags.any()
    kd, vd, _, st = gpu_append(w.k_pool, w.v_pool, kn, vn, w.block_tables, pos)
    assert st == 0 and same_bits(kd, rk) and same_bits(vd, rv)

    for fp8 in (False, True):
        codes = oracle_codes(w, fp8)
        app = oracle.append_fp8 if fp8 else oracle.append_int8
        ref = app(w.k_pool, w.v_pool, *codes, kn, vn, w.block_tables, pos)
        kd, vd, dc, st = gpu_append(w.k_pool, w.v_pool, kn, vn, w.block_tables, pos, codes,
                                    fp8=fp8)
        assert st == 0
        assert same_bits(kd, ref[0]) and same_bits(vd, ref[1])
        for got, want in zip(dc, (ref[2], ref[3], ref[4], ref[5])):
            assert same_bits(got, want)


@pytest.mark.parametrize("d", [64, 128])
def test_append_edge_positions_and_status(d):
    rng = np.random.default_rng(d)
    n, hkv, nb = 7, 2, 10
    tables = np.array([[0, 1], [2, 3], [4, 5], [6, -1], [7, 99], [3, 2], [8, 9]], np.int32)
    pos = np.array([-1, 16, 15, 32, 20, 31, 0], np.int32)
    kp = rng.standard_normal((nb, hkv, 16, d)).astype(np.float16)
    vp = rng.standard_normal((nb, hkv, 16, d)).astype(np.float16)
    kn = rng.standard_normal((n, hkv, d)).astype(np.float16)
    vn = rng.standard_normal((n, hkv, d)).astype(np.float16)
    codes = (np.full(kp.shape, 5, np.int8), np.full(kp.shape, -5, np.int8),
             np.full((nb, hkv), 2.0, np.float32), np.full((nb, hkv), 3.0, np.float32))
    ref = oracle.append_int8(kp, vp, *codes, kn, vn, tables, pos)
    assert ref[6].tolist() == [0, 0, 0, oracle.BAD_CTX, oracle.BAD_BLOCK, 0, 0]
    for int8 in (False, True):
        kd, vd, dc, st = gpu_append(kp, vp, kn, vn, tables, pos, codes if int8 else None)
        assert st == pkv.PKV_DEV_BAD_CTX | pkv.PKV_DEV_BAD_BLOCK
        assert same_bits(kd, ref[0]) and same_bits(vd, ref[1])
        if int8:
            for got, want in zip(dc, ref[2:6]):
                assert same_bits(got, want)


@pytest.mark.parametrize("name", ["c5a_64x2048", "c5b_256_ragged"])
def test_full_size_append_int8_then_decode(name):
    # the whole decode step at full size: append the newest token of every
    # sequence (fused tail re-quantize), then INT8 decode over the new context
    w = W.make(name)
    kn, vn, pos = W.append_tokens(w, 99)
    tails = w.tail_block_ids()
    codes = oracle_codes(w)
    kd, vd = dev(w.k_pool), dev(w.v_pool)
    kd0 = kd.clone()
    dc = tuple(dev(c) for c in codes)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_append_int8(kd, vd, *dc, dev(kn), dev(vn), dev(w.block_tables), dev(pos),
                        dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # reference: the oracle's append on the tail tiles only (the rest of the
    # pool is unchanged on both sides, checked on the device below)
    ref = oracle.append_int8(w.k_pool, w.v_pool, *codes, kn, vn, w.block_tables, pos,
                             inplace=False)
    tix = torch.from_numpy(tails.astype(np.int64)).cuda()
    assert same_bits(kd[tix], ref[0][tails]) and same_bits(vd[tix], ref[1][tails])
    for got, want in zip(dc, ref[2:6]):
        assert same_bits(got[tix], want[tails])
    untouched = torch.ones(w.num_blocks, dtype=torch.bool, device="cuda")
    untouched[tix] = False
    assert torch.equal(kd[untouched].view(torch.int16), kd0[untouched].view(torch.int16))
    del kd0

    n, hq, d = w.query.shape
    out = torch.full((n, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, w.max_context_len)
    pkv.pkv_paged_decode_int8(out, dev(w.query), *dc, dev(w.block_tables),
                              dev(w.context_lens), w.max_context_len, w.softmax_scale, ws,
                              status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = oracle.decode_int8(w.query, ref[2], ref[3], ref[4], ref[5], w.block_tables,
                              w.context_lens, num_kv_heads=w.num_kv_heads,
                              softmax_scale=w.softmax_scale)
    assert_close(out.cpu().numpy().astype(np.float64), want, f"{name} append+decode")


def test_append_fp16_then_decode_sees_the_new_token():
    w = W.random_case(77, num_seqs=6, num_heads=32, num_kv_heads=8, head_dim=128,
                      context_lens=[1, 16, 17, 100, 512, 33])
    kn, vn, pos = W.append_tokens(w, 5)
    kd, vd, _, st = gpu_append(w.k_pool, w.v_pool, kn, vn, w.block_tables, pos)
    assert st == 0
    n, hq, d = w.query.shape
    out = torch.empty((n, hq, d), dtype=torch.float32, device="cuda")
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, w.max_context_len)
    pkv.pkv_paged_decode_fp16(out, dev(w.query), kd, vd, dev(w.block_tables),
                              dev(w.context_lens), w.max_context_len, w.softmax_scale, ws)
    torch.cuda.synchronize()
    rk, rv, _, _ = oracle.append_fp16(w.k_pool, w.v_pool, kn, vn, w.block_tables, pos)
    want = oracle.decode_fp16(w.query, rk, rv, w.block_tables, w.context_lens,
                              num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale)
    assert_close(out.cpu().numpy().astype(np.float64), want, "fp16 append+decode")
    # a one-token context returns the appended V row
    for h in range(hq):
        np.testing.assert_allclose(out[0, h].cpu().numpy(),
                                   vn[0, h // (hq // w.num_kv_heads)].astype(np.float32),
                                   rtol=0, atol=1e-6)

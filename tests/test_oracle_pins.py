"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test names what it pins and which plausible mistake it would catch.  The
oracle is then trusted as the reference for the CUDA parity tests.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import pkv_workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------
# fp16 decoding: every one of the 65536 bit patterns against numpy's own
# binary16 -> binary64 conversion (a library routine).  Catches a wrong
# exponent bias, a subnormal mistake or a sign slip.
def test_half_decoding_matches_numpy_for_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# --------------------------------------------------------------------------
# Memory arithmetic printed by the PagedKV-Fusion README (Memory footprint
# table).  Pins the layout reading: one fp32 scale for K and one for V per
# (block, head); two pools.
def test_memory_footprint_matches_printed_table():
    rows = _read_golden("memory_footprint.txt")
    assert len(rows) == 3
    for nb, h, d, fp16_mib, int8_mib in rows:
        assert oracle.kv_pool_mib(int(nb), int(h), int(d), "fp16") == float(fp16_mib)
        assert oracle.kv_pool_mib(int(nb), int(h), int(d), "int8") == float(int8_mib)


# --------------------------------------------------------------------------
# Worked example with a closed-form answer.  Block size 2, head_dim 2, four q
# heads over two kv heads (GQA 2), a non-identity block table, softmax scale
# 0.5 and a NaN padding slot.  Catches: a dropped softmax scale, the h % Hkv
# head mapping, a wrong slot (t % B) or block (t / B) index, a missing mask.
def _worked_case():
    nan = np.nan
    B, d = 2, 2
    # physical pool [3 blocks][2 kv heads][2 slots][2]
    k = np.full((3, 2, B, d), nan)
    v = np.full((3, 2, B, d), nan)
    # logical tokens 0,1 -> physical block 1; token 2 -> physical block 0 slot 0
    # kv head 0
    k[1, 0, 0] = [0.0, 2.0];  v[1, 0, 0] = [1.0, 0.0]
    k[1, 0, 1] = [2.0, 0.0];  v[1, 0, 1] = [0.0, 1.0]
    k[0, 0, 0] = [4.0, -2.0]; v[0, 0, 0] = [1.0, 1.0]
    # kv head 1: keys reversed, different values
    k[1, 1, 0] = [4.0, 0.0];  v[1, 1, 0] = [2.0, 0.0]
    k[1, 1, 1] = [2.0, 0.0];  v[1, 1, 1] = [0.0, 2.0]
    k[0, 1, 0] = [0.0, 0.0];  v[0, 1, 0] = [-2.0, 4.0]
    q = np.array([[[1.0, 0.0], [0.0, 1.0], [1.0, 0.0], [0.0, 0.0]]])
    table = np.array([[1, 0]], dtype=np.int32)
    ctx = np.array([3], dtype=np.int32)
    return q, k, v, table, ctx


def _softmax_combo(z, vals):
    w = [math.exp(x) for x in z]
    s = sum(w)
    return [sum(wi * vi[j] for wi, vi in zip(w, vals)) / s for j in range(2)]


def test_worked_example_closed_form():
    q, k, v, table, ctx = _worked_case()
    out = oracle.decode_fp16(q.astype(np.float16), k.astype(np.float16), v.astype(np.float16),
                             table, ctx, num_kv_heads=2, softmax_scale=0.5, block_size=2)
    v0 = [[1, 0], [0, 1], [1, 1]]
    v1 = [[2, 0], [0, 2], [-2, 4]]
    expect = [
        _softmax_combo([0.0, 1.0, 2.0], v0),    # head 0 -> kv 0, z = 0.5*(0, 2, 4)
        _softmax_combo([1.0, 0.0, -1.0], v0),   # head 1 -> kv 0, z = 0.5*(2, 0, -2)
        _softmax_combo([2.0, 1.0, 0.0], v1),    # head 2 -> kv 1, z = 0.5*(4, 2, 0)
        [0.0, 2.0],                             # head 3 -> kv 1, q = 0: mean of V
    ]
    np.testing.assert_allclose(out[0], np.array(expect), rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# Identity block table == contiguous dense attention, computed by torch's
# scaled_dot_product_attention in fp64 with its own GQA expansion (a library
# routine).  Ragged contexts (not multiples of 16) with NaN padding slots.
def _identity_case(seed, n, hq, hkv, d, ctx, kind="fp16"):
    rng = np.random.default_rng(seed)
    B = 16
    nblk = [(c + B - 1) // B for c in ctx]
    mb = max(nblk + [1])
    nb = sum(nblk) + 1
    kpool = np.full((nb, hkv, B, d), np.nan)
    vpool = np.full((nb, hkv, B, d), np.nan)
    table = np.full((n, mb), -1, np.int32)
    dense_k, dense_v = [], []
    off = 0
    for s in range(n):
        kd = rng.standard_normal((hkv, max(ctx[s], 1), d))
        vd = rng.standard_normal((hkv, max(ctx[s], 1), d))
        if kind == "int8":
            kd = np.clip(np.round(kd * 40), -127, 127)
            vd = np.clip(np.round(vd * 40), -127, 127)
        else:
            kd = kd.astype(np.float16).astype(np.float64)
            vd = vd.astype(np.float16).astype(np.float64)
        kd, vd = kd[:, :ctx[s]], vd[:, :ctx[s]]
        dense_k.append(kd)
        dense_v.append(vd)
        for j in range(nblk[s]):
            table[s, j] = off + j
            t0, t1 = j * B, min(ctx[s], (j + 1) * B)
            kpool[off + j, :, : t1 - t0] = kd[:, t0:t1]
            vpool[off + j, :, : t1 - t0] = vd[:, t0:t1]
        off += nblk[s]
    q = rng.standard_normal((n, hq, d)).astype(np.float16)
    return q, kpool, vpool, table, np.array(ctx, np.int32), dense_k, dense_v


def _sdpa(q, dense_k, dense_v, scale):
    outs = []
    for s in range(q.shape[0]):
        qs = torch.from_numpy(q[s].astype(np.float64))[None, :, None, :]
        ks = torch.from_numpy(dense_k[s])[None]
        vs = torch.from_numpy(dense_v[s])[None]
        if ks.shape[2] == 0:
            outs.append(np.zeros(q.shape[1:]))
            continue
        o = torch.nn.functional.scaled_dot_product_attention(
            qs, ks, vs, scale=scale, enable_gqa=True)
        outs.append(o[0, :, 0, :].numpy())
    return np.stack(outs)


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (8, 8, 128), (14, 2, 64), (16, 1, 32)])
def test_identity_table_equals_contiguous_sdpa_fp16(hq, hkv, d):
    ctx = [1, 15, 16, 17, 37, 64]
    q, kp, vp, table, lens, dk, dv = _identity_case(7 + hq + d, len(ctx), hq, hkv, d, ctx)
    scale = 1.0 / math.sqrt(d)
    got = oracle.decode_fp16(q, kp.astype(np.float16), vp.astype(np.float16), table, lens,
                             num_kv_heads=hkv, softmax_scale=scale)
    ref = _sdpa(q, dk, dv, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_identity_table_equals_contiguous_sdpa_int8_with_scales():
    # K and V scales differ per tile and are powers of two, so code * scale is
    # exact and the dense reference can be formed without the oracle's rule.
    hq, hkv, d = 8, 2, 64
    ctx = [5, 16, 40]
    q, kc, vc, table, lens, dk, dv = _identity_case(99, len(ctx), hq, hkv, d, ctx, "int8")
    nb = kc.shape[0]
    ks = (2.0 ** -(np.arange(nb * hkv) % 3 + 1)).reshape(nb, hkv).astype(np.float32)
    vs = (2.0 ** -(np.arange(nb * hkv) % 4 + 2)).reshape(nb, hkv).astype(np.float32)
    kcodes = np.nan_to_num(kc, nan=0.0).astype(np.int8)
    vcodes = np.nan_to_num(vc, nan=0.0).astype(np.int8)
    dk_s, dv_s = [], []
    for s in range(len(ctx)):
        ks_tok = np.concatenate([np.repeat(ks[table[s, j]][:, None], 16, 1)
                                 for j in range((ctx[s] + 15) // 16)], 1)[:, :ctx[s], None]
        vs_tok = np.concatenate([np.repeat(vs[table[s, j]][:, None], 16, 1)
                                 for j in range((ctx[s] + 15) // 16)], 1)[:, :ctx[s], None]
        dk_s.append(dk[s] * ks_tok)
        dv_s.append(dv[s] * vs_tok)
    scale = 0.125
    got = oracle.decode_int8(q, kcodes, vcodes, ks, vs, table, lens,
                             num_kv_heads=hkv, softmax_scale=scale)
    ref = _sdpa(q, dk_s, dv_s, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Invariants of paging itself.
def test_physical_placement_is_irrelevant_bit_exact():
    w = W.make("c1_tiny")
    base = oracle.decode_fp16(w.query, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                              num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale)
    perm = np.random.default_rng(5).permutation(w.num_blocks).astype(np.int32)
    kp = np.empty_like(w.k_pool); vp = np.empty_like(w.v_pool)
    kp[perm] = w.k_pool; vp[perm] = w.v_pool
    table = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    moved = oracle.decode_fp16(w.query, kp, vp, table, w.context_lens,
                               num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale)
    assert np.array_equal(base, moved)


def test_single_token_context_returns_that_value_exactly():
    w = W.random_case(11, num_seqs=3, num_heads=4, num_kv_heads=2, head_dim=64,
                      context_lens=[1, 1, 1])
    out = oracle.decode_fp16(w.query, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                             num_kv_heads=2, softmax_scale=w.softmax_scale)
    for s in range(3):
        blk = w.block_tables[s, 0]
        for h in range(4):
            assert np.array_equal(out[s, h], w.v_pool[blk, h // 2, 0].astype(np.float64))


def test_constant_value_rows_return_that_value():
    w = W.random_case(12, num_seqs=4, num_heads=8, num_kv_heads=2, head_dim=128,
                      context_lens=[3, 16, 33, 100])
    c = np.random.default_rng(1).standard_normal(128).astype(np.float16)
    vp = w.v_pool.copy()
    vp[w.used_block_ids] = c
    out = oracle.decode_fp16(w.query, w.k_pool, vp, w.block_tables, w.context_lens,
                             num_kv_heads=2, softmax_scale=w.softmax_scale)
    np.testing.assert_allclose(out, np.broadcast_to(c.astype(np.float64), out.shape),
                               rtol=0, atol=1e-13)


def test_zero_query_gives_mean_of_values():
    hq, hkv, d = 4, 2, 64
    ctx = [7, 16, 50]
    q, kp, vp, table, lens, dk, dv = _identity_case(3, 3, hq, hkv, d, ctx)
    q[:] = 0
    out = oracle.decode_fp16(q, kp.astype(np.float16), vp.astype(np.float16), table, lens,
                             num_kv_heads=hkv, softmax_scale=0.3)
    for s in range(3):
        mean = dv[s].mean(axis=1)  # [hkv][d]
        np.testing.assert_allclose(out[s], np.repeat(mean, hq // hkv, axis=0), rtol=0, atol=1e-13)


def test_brute_force_python_on_tiny_config():
    w = W.make("c1_tiny")
    out = oracle.decode_fp16(w.query, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                             num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale)
    g = w.num_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        for h in range(w.num_heads):
            qv = [float(x) for x in w.query[s, h]]
            rows = []
            for t in range(int(w.context_lens[s])):
                blk = int(w.block_tables[s, t // 16])
                kk = [float(x) for x in w.k_pool[blk, h // g, t % 16]]
                vv = [float(x) for x in w.v_pool[blk, h // g, t % 16]]
                rows.append((w.softmax_scale * sum(a * b for a, b in zip(qv, kk)), vv))
            m = max(z for z, _ in rows)
            ws = [math.exp(z - m) for z, _ in rows]
            tot = sum(ws)
            ref = [sum(wt * vv[i] for wt, (_, vv) in zip(ws, rows)) / tot for i in range(w.head_dim)]
            np.testing.assert_allclose(out[s, h], ref, rtol=0, atol=1e-12)


def test_invalid_inputs_give_zeros_and_flags():
    w = W.random_case(13, num_seqs=4, num_heads=4, num_kv_heads=2, head_dim=64,
                      context_lens=[20, 0, 40, 10])
    table = w.block_tables.copy()
    table[2, 1] = w.num_blocks + 5          # out-of-pool id inside the context
    lens = w.context_lens.copy()
    lens[3] = 10_000                        # longer than the table can hold
    out, flags = oracle.decode_fp16(w.query, w.k_pool, w.v_pool, table, lens,
                                    num_kv_heads=2, softmax_scale=w.softmax_scale,
                                    return_flags=True)
    assert np.all(out[1] == 0) and np.all(flags[1] == 0)
    assert np.all(out[2] == 0) and np.all(flags[2] == oracle.BAD_BLOCK)
    assert np.all(out[3] == 0) and np.all(flags[3] == oracle.BAD_CTX)
    assert np.all(flags[0] == 0) and np.all(np.isfinite(out[0])) and np.any(out[0] != 0)


# --------------------------------------------------------------------------
# Quantizer.  Worked ties: a tile whose max |x| is 127 has scale exactly 1.0,
# one whose max is 254 has scale 2.0 and one whose max is 63.5 has scale 0.5,
# so x / scale is exact and the rounding rule alone decides the code.
# Catches: round-half-away-from-zero, truncation, a 127.5 or 128 divisor.
TIE_CASES = [
    (127.0, [(2.5, 2), (3.5, 4), (-2.5, -2), (0.5, 0), (1.5, 2), (-0.5, 0),
             (126.5, 126), (-3.5, -4), (-127.0, -127)]),
    (254.0, [(5.0, 2), (7.0, 4), (-5.0, -2), (1.0, 0), (3.0, 2), (253.0, 126)]),
    (63.5, [(0.25, 0), (0.75, 2), (-0.75, -2), (1.25, 2), (63.25, 126)]),
]


@pytest.mark.parametrize("amax,pairs", TIE_CASES)
def test_quantize_ties_round_half_to_even(amax, pairs):
    tile = np.zeros((1, 1, 16, 64), np.float16)
    flat = tile.reshape(-1)
    flat[0] = amax
    for i, (x, _) in enumerate(pairs):
        flat[1 + i] = x
    codes, scales = oracle.quantize(tile)
    assert scales[0, 0] == np.float32(amax / 127.0)
    c = codes.reshape(-1)
    assert c[0] == 127
    for i, (_, want) in enumerate(pairs):
        assert c[1 + i] == want, (pairs[i], c[1 + i])
    assert np.all(c[1 + len(pairs):] == 0)


@pytest.mark.parametrize("heavy", [False, True])
def test_quantize_error_bound_and_extremes(heavy):
    rng = np.random.default_rng(21 + heavy)
    x = rng.standard_normal((64, 4, 16, 128)).astype(np.float32)
    if heavy:
        idx = rng.choice(x.size, size=x.size // 1000, replace=False)
        x.reshape(-1)[idx] *= 10
    x = x.astype(np.float16)
    codes, scales = oracle.quantize(x)
    xf = x.astype(np.float64)
    amax = np.abs(xf).max(axis=(2, 3))
    # scale is the fp32 quotient of the fp32 absmax by 127
    assert np.array_equal(scales, (amax.astype(np.float32) / np.float32(127)).astype(np.float32))
    deq = codes.astype(np.float64) * scales[:, :, None, None].astype(np.float64)
    err = np.abs(xf - deq)
    # scale/2, plus one fp32 ulp of the quotient x/scale (|x/scale| <= 127 <
    # 2^7, so an ulp is at most 2^-16): x/scale is rounded to fp32 before the
    # half-even rounding, which can carry 63.49999 to 63.5 and then to 64.
    bound = scales[:, :, None, None].astype(np.float64) * (0.5 + 2.0 ** -16)
    assert np.all(err <= bound)
    assert codes.min() >= -127 and codes.max() <= 127
    # the element holding max |x| maps to +-127
    flat = xf.reshape(64, 4, -1)
    arg = np.abs(flat).argmax(axis=2)
    top = np.take_along_axis(codes.reshape(64, 4, -1), arg[..., None], 2)[..., 0]
    sign = np.sign(np.take_along_axis(flat, arg[..., None], 2)[..., 0])
    assert np.array_equal(top, (127 * sign).astype(np.int8))


def test_quantize_zero_nan_inf_tiles():
    x = np.zeros((3, 1, 16, 64), np.float16)
    x[1, 0, 0, :8] = [1.0, -2.0, np.nan, 0.5, np.nan, 3.0, -3.0, 0.0]
    x[2, 0, 0, 0] = np.inf
    x[2, 0, 0, 1] = 5.0
    codes, scales = oracle.quantize(x)
    assert scales[0, 0] == 0 and np.all(codes[0] == 0)         # all-zero tile
    assert scales[1, 0] == np.float32(3.0) / np.float32(127)   # NaN ignored in the max
    c1 = codes[1, 0, 0, :8]
    assert c1[2] == 0 and c1[4] == 0 and c1[5] == 127 and c1[6] == -127
    assert np.isinf(scales[2, 0]) and np.all(codes[2] == 0)    # inf scale: all codes 0


def test_quantize_block_ids_subset_duplicates_and_bad_ids():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((10, 2, 16, 64)).astype(np.float16)
    full_c, full_s = oracle.quantize(x)
    ids = np.array([7, 2, 7, -1, 10, 2], np.int32)
    c, s = oracle.quantize(x, block_ids=ids)
    for b in range(10):
        if b in (2, 7):
            assert np.array_equal(c[b], full_c[b]) and np.array_equal(s[b], full_s[b])
        else:
            assert np.all(c[b] == 0) and np.all(s[b] == 0)

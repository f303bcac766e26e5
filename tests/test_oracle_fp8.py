"""Pins of the oracle's FP8 (OCP E4M3) functions: decoding and rounding
against torch's float8_e4m3fn conversion (a library routine), saturation,
the quantizer's error bound, and FP8 decode attention against torch SDPA."""
import math

import numpy as np
import pytest
import torch

import oracle


def torch_e4m3(values):
    t = torch.tensor(np.asarray(values, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


# Every byte decodes to torch's value (NaN exactly at 0x7F and 0xFF).
# Catches a wrong bias, a subnormal slip, a mantissa width error.
def test_every_code_decodes_like_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got).sum() == 2
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok].astype(np.float64))
    assert oracle.e4m3_to_double(0x7E) == 448.0 and oracle.e4m3_to_double(1) == 2.0 ** -9


# Round to nearest with ties to even on the E4M3 grid, as torch does, on
# every finite value, every midpoint between neighbours (the ties), the
# fp32 numbers either side of each midpoint, and random values.
def test_rounding_matches_torch():
    mags = sorted({oracle.e4m3_to_double(c) for c in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(mags, mags[1:])]
    vals = list(mags) + mids
    for m in mids:
        f = np.float32(m)
        vals += [float(np.nextafter(f, np.float32(0))), float(np.nextafter(f, np.float32(np.inf)))]
    rng = np.random.default_rng(0)
    vals += list(rng.uniform(-464, 464, 4000)) + list(rng.uniform(-0.02, 0.02, 2000))
    vals = np.asarray(vals, np.float32)
    vals = np.concatenate([vals, -vals])
    vals = vals[np.abs(vals) <= 464]
    ref = torch_e4m3(vals)
    got = np.array([oracle.e4m3_from_float(float(v)) for v in vals], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:5]]


# The encoder against a brute-force search over all finite codes (nearest
# value, ties to the code with an even last bit) on a dense sweep.
def test_rounding_matches_brute_force_search():
    lut = np.array([oracle.e4m3_to_double(c) for c in range(0x7F)])
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(0, 470, 3000), rng.uniform(0, 0.05, 2000),
                           (lut[:-1] + lut[1:]) / 2, lut]).astype(np.float32)
    for v in vals:
        err = np.abs(lut - float(v))
        best = np.flatnonzero(err == err.min())
        want = best[0] if best.size == 1 else [b for b in best if b % 2 == 0][0]
        assert oracle.e4m3_from_float(float(v)) == want, float(v)


def test_saturation_beyond_the_largest_finite_value():
    for v in (448.0, 449.0, 463.99, 464.0, 470.0, 1e6, 3.0e38):
        assert oracle.e4m3_from_float(v) == 0x7E
        assert oracle.e4m3_from_float(-v) == 0xFE


# The quantizer: scale = fp32(amax) / 448; each value within half a grid step
# (at its magnitude) of code * scale; the absmax element reaches +-448; zero,
# NaN and inf tiles as for INT8.
@pytest.mark.parametrize("heavy", [False, True])
def test_quantize_fp8_error_bound(heavy):
    rng = np.random.default_rng(5 + heavy)
    x = rng.standard_normal((24, 2, 16, 64)).astype(np.float32)
    if heavy:
        x.reshape(-1)[rng.choice(x.size, 40, replace=False)] *= 30
    x = x.astype(np.float16)
    codes, sc = oracle.quantize_fp8(x)
    xd = x.astype(np.float64)
    for b in range(x.shape[0]):
        for h in range(x.shape[1]):
            amax = np.float32(np.abs(xd[b, h]).max())
            assert sc[b, h] == amax / np.float32(448)
            y = xd[b, h] / float(sc[b, h])
            deq = np.vectorize(oracle.e4m3_to_double)(codes[b, h])
            step = np.where(np.abs(y) >= 2.0 ** -6,
                            2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 1e-300))) - 3),
                            2.0 ** -9)
            assert np.all(np.abs(deq - y) <= step / 2 * (1 + 2.0 ** -20))
            assert np.any((codes[b, h] & 0x7F) == 0x7E)


def test_quantize_fp8_zero_nan_inf_tiles():
    x = np.zeros((3, 1, 16, 64), np.float16)
    x[1, 0, 0, :5] = np.nan
    x[1, 0, 1, 0] = 2.0
    x[2, 0, 3, 7] = np.inf
    x[2, 0, 4, 0] = 1.0
    codes, sc = oracle.quantize_fp8(x)
    assert sc[0, 0] == 0 and not codes[0].any()
    assert sc[1, 0] == np.float32(2.0) / np.float32(448)
    assert not codes[1, 0, 0, :5].any() and codes[1, 0, 1, 0] == 0x7E
    assert np.isinf(sc[2, 0]) and not codes[2].any()


# FP8 decode with power-of-two scales (exact dequantization) through an
# identity block table equals torch's fp64 SDPA over the dense values.
def test_fp8_decode_identity_table_equals_sdpa():
    rng = np.random.default_rng(11)
    n, hq, hkv, d, ctx = 3, 8, 2, 64, [1, 23, 48]
    nblk = [(c + 15) // 16 for c in ctx]
    nb = sum(nblk)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    kc = rng.choice(finite, (nb, hkv, 16, d)).astype(np.uint8)
    vc = rng.choice(finite, (nb, hkv, 16, d)).astype(np.uint8)
    ks = (2.0 ** rng.integers(-4, 2, (nb, hkv))).astype(np.float32)
    vs = (2.0 ** rng.integers(-4, 2, (nb, hkv))).astype(np.float32)
    table = np.full((n, max(nblk)), -1, np.int32)
    off = 0
    for s in range(n):
        table[s, :nblk[s]] = np.arange(off, off + nblk[s])
        off += nblk[s]
    q = rng.standard_normal((n, hq, d)).astype(np.float16)
    lut = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    got = oracle.decode_fp8(q, kc, vc, ks, vs, table, np.array(ctx, np.int32), num_kv_heads=hkv,
                            softmax_scale=1 / math.sqrt(d))
    for s in range(n):
        blks = table[s, :nblk[s]]
        kd = (lut[kc[blks]] * ks[blks][:, :, None, None]).transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :ctx[s]]
        vd = (lut[vc[blks]] * vs[blks][:, :, None, None]).transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :ctx[s]]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[s].astype(np.float64))[None, :, None, :], torch.from_numpy(kd)[None],
            torch.from_numpy(vd)[None], scale=1 / math.sqrt(d), enable_gqa=True)[0, :, 0, :].numpy()
        np.testing.assert_allclose(got[s], ref, rtol=0, atol=1e-12)

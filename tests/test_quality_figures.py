"""Quantization quality of the INT8 path against the PagedKV-Fusion README's
printed figures (Results, "Quantization quality vs FP32"): RMSE and max-abs
error of the INT8-KV attention output against full precision, and the
output's standard deviation, for Gaussian unit-variance K and V.

The README does not print the shape; a context of 48 tokens reproduces its
output std 0.233 (for N(0,1) scores the std of a softmax-weighted mean of N
unit-variance rows falls like 1/sqrt(N)).  On that probe the oracle's INT8
path must land on the printed RMSE within 15 % and the printed std within
5 % -- a check of the quantizer reading (absmax / 127, round half to even)
against the pages' own measurement.  The heavy-tailed row is reported only:
its printed output std (7.02) cannot come from N(0,1) values.  CPU only."""
import os

import numpy as np

import oracle
import pkv_workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quality_figures.txt")


def printed():
    rows = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            name, rmse, mx, sd = line.split()
            rows[name] = (float(rmse), float(mx), float(sd))
    return rows


def quality(w, quantize, decode):
    ref = oracle.decode_fp16(w.query, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                             num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale)
    kc, ks = quantize(w.k_pool, block_ids=w.used_block_ids)
    vc, vs = quantize(w.v_pool, block_ids=w.used_block_ids)
    got = decode(w.query, kc, vc, ks, vs, w.block_tables, w.context_lens,
                 num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale)
    err = got - ref
    return float(np.sqrt((err ** 2).mean())), float(np.abs(err).max()), float(ref.std())


def test_gaussian_probe_matches_the_printed_int8_quality():
    rmse_p, max_p, std_p = printed()["gaussian"]
    w = W.random_case(48, num_seqs=16, num_heads=8, num_kv_heads=8, head_dim=128,
                      context_lens=[48] * 16)
    rmse, mx, sd = quality(w, oracle.quantize, oracle.decode_int8)
    assert abs(sd - std_p) <= 0.05 * std_p, sd
    assert abs(rmse - rmse_p) <= 0.15 * rmse_p, rmse
    assert 0.5 * max_p <= mx <= 1.5 * max_p, mx
    # FP8 (3 mantissa bits) on the same probe: reported, coarser than INT8 here
    rmse8, _, _ = quality(w, oracle.quantize_fp8, oracle.decode_fp8)
    assert rmse < rmse8 < 10 * rmse

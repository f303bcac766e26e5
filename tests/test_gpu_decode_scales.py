"""Decode parity across the magnitudes of K, V and q.

The per-(block, kv head) scales exist so that one cache can hold K and V of
any magnitude ("PagedKV-Fusion" README, Overview, component B;
"PagedAttention & KV-Cache Memory Management" section 5.1, Quantization
Pipeline & Block-Granular Layout), so the kernels must hold the decode
tolerance (max-abs 2e-3, rel-L2 1e-3 against the fp64 oracle on identical
inputs) whatever that magnitude: K and V scaled by 2^-12 ... 2^4, one block
of every sequence with V a hundred times larger than the rest (scales that
differ within one item), and queries with standard deviation 10 (peaked
softmax).  The same inputs are split over forced worker counts as well, so
the scale handling is checked across partial records.
"""
import pytest

import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import assert_close, ensure_built, gpu_decode, oracle_codes, oracle_decode

pytestmark = pytest.mark.gpu

VARIANTS = ["fp16", "int8", "fp8"]
MAGNITUDES = {
    "v2^-12": dict(v_mult=2.0 ** -12),
    "v2^-8": dict(v_mult=2.0 ** -8),
    "v2^-4": dict(v_mult=2.0 ** -4),
    "v2^4": dict(v_mult=2.0 ** 4),
    "k2^-12": dict(k_mult=2.0 ** -12),
    "k2^-8": dict(k_mult=2.0 ** -8),
    "k2^-4": dict(k_mult=2.0 ** -4),
    "k2^4": dict(k_mult=2.0 ** 4),
    "kv2^-12": dict(k_mult=2.0 ** -12, v_mult=2.0 ** -12),
    "hot-block-x100": dict(v_hot_mult=100.0),
    "hot-block-x100-v2^-8": dict(v_hot_mult=100.0, v_mult=2.0 ** -8),
    "q-sd10": dict(q_std=10.0),
    "q-sd10-k2^-4-v2^-12": dict(q_std=10.0, k_mult=2.0 ** -4, v_mult=2.0 ** -12),
}
LENS = [1, 17, 300, 777, 1024, 2000]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("mag", list(MAGNITUDES), ids=list(MAGNITUDES))
def test_magnitudes_match_oracle(variant, mag):
    w = W.random_case(300 + list(MAGNITUDES).index(mag), num_seqs=len(LENS), num_heads=8,
                      num_kv_heads=2, head_dim=128, context_lens=LENS, **MAGNITUDES[mag])
    codes = None if variant == "fp16" else oracle_codes(w, variant == "fp8")
    got, st = gpu_decode(w, variant, codes)
    ref, flags = oracle_decode(w, variant, codes)
    assert st == 0 and not flags.any()
    assert_close(got, ref, f"{mag}/{variant}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("mag", ["v2^-12", "hot-block-x100-v2^-8", "q-sd10"])
def test_magnitudes_head_dim_64_group_7(variant, mag):
    w = W.random_case(320 + list(MAGNITUDES).index(mag), num_seqs=5, num_heads=14,
                      num_kv_heads=2, head_dim=64, context_lens=[1, 40, 512, 700, 1100],
                      **MAGNITUDES[mag])
    codes = None if variant == "fp16" else oracle_codes(w, variant == "fp8")
    got, st = gpu_decode(w, variant, codes)
    ref, flags = oracle_decode(w, variant, codes)
    assert st == 0 and not flags.any()
    assert_close(got, ref, f"d64/{mag}/{variant}")


@pytest.mark.parametrize("variant", ["int8", "fp8"])
@pytest.mark.parametrize("workers", [1, 2, 7, 13, 64])
def test_scale_spread_over_forced_splits(variant, workers):
    # blocks of one item with V scales 100x apart, cut into pieces that start
    # at different pages: every piece's record and the merge keep the scales
    w = W.random_case(340, num_seqs=4, num_heads=8, num_kv_heads=2, head_dim=128,
                      context_lens=[2000, 333, 1024, 48], v_hot_mult=100.0, v_mult=2.0 ** -8)
    codes = oracle_codes(w, variant == "fp8")
    ensure_built()
    try:
        pkv.pkv_set_decode_workers(workers)
        got, st = gpu_decode(w, variant, codes)
    finally:
        pkv.pkv_set_decode_workers(0)
    ref, _ = oracle_decode(w, variant, codes)
    assert st == 0
    assert_close(got, ref, f"workers={workers}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("mag", ["hot-block-x100-v2^-8", "q-sd10-k2^-4-v2^-12", "v2^4"])
@pytest.mark.parametrize("hq,hkv", [(32, 2), (64, 1)])
def test_magnitudes_two_groups_per_item(variant, mag, hq, hkv):
    # 16 and 64 query heads per kv head: work items of two groups of 8 share
    # every page, and the V-scale reference rescales both groups' accumulators
    w = W.random_case(360 + list(MAGNITUDES).index(mag) + hq, num_seqs=4, num_heads=hq,
                      num_kv_heads=hkv, head_dim=128, context_lens=[1, 300, 777, 2000],
                      **MAGNITUDES[mag])
    codes = None if variant == "fp16" else oracle_codes(w, variant == "fp8")
    got, st = gpu_decode(w, variant, codes)
    ref, flags = oracle_decode(w, variant, codes)
    assert st == 0 and not flags.any()
    assert_close(got, ref, f"g{hq // hkv}/{mag}/{variant}")


@pytest.mark.parametrize("variant", ["int8", "fp8"])
@pytest.mark.parametrize("workers", [1, 7, 64])
def test_two_groups_scale_spread_over_forced_splits(variant, workers):
    # records of 16 heads merged by the reduce, V scales 100x apart
    w = W.random_case(370, num_seqs=3, num_heads=32, num_kv_heads=2, head_dim=128,
                      context_lens=[2000, 333, 48], v_hot_mult=100.0, v_mult=2.0 ** -8)
    codes = oracle_codes(w, variant == "fp8")
    ensure_built()
    try:
        pkv.pkv_set_decode_workers(workers)
        got, st = gpu_decode(w, variant, codes)
    finally:
        pkv.pkv_set_decode_workers(0)
    ref, _ = oracle_decode(w, variant, codes)
    assert st == 0
    assert_close(got, ref, f"two groups, workers={workers}")

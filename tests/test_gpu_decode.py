"""Paged decode attention on the GPU against the fp64 CPU oracle.

Every case compares the CUDA output element by element with the oracle on the
same seeded inputs: max-abs <= 2e-3 and rel-L2 <= 1e-3.  The full-size
configurations run in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import (assert_close, dev, ensure_built, gpu_decode, oracle_codes,
                        oracle_decode, persistent_workers)

pytestmark = pytest.mark.gpu

VARIANTS = ["fp16", "int8", "fp8"]
_cache = {}


def workload(name, variant):
    if name not in _cache:
        _cache.clear()  # one configuration at a time (the full-size pools are large)
        _cache[name] = (W.make(name), {})
    w, codes = _cache[name]
    if variant != "fp16" and variant not in codes:
        codes[variant] = oracle_codes(w, variant == "fp8")
    return w, codes.get(variant)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", W.CONFIG_NAMES)
def test_configs_match_oracle(name, variant):
    w, codes = workload(name, variant)
    got, st = gpu_decode(w, variant, codes)
    ref, flags = oracle_decode(w, variant, codes)
    assert st == 0 and not flags.any()
    assert_close(got, ref, f"{name}/{variant}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("workers", [1, 2, 7, 13, 64, 0])
def test_split_count_sweep(variant, workers):
    # the same batch split over 1..many workers: every split merges to the
    # oracle's answer, and to each other within float rounding
    w = W.random_case(40, num_seqs=6, num_heads=8, num_kv_heads=2, head_dim=128,
                      context_lens=[300, 1, 77, 512, 16, 250])
    codes = oracle_codes(w, variant == "fp8")
    ensure_built()
    try:
        pkv.pkv_set_decode_workers(workers)
        got, st = gpu_decode(w, variant, codes)
    finally:
        pkv.pkv_set_decode_workers(0)
    base, _ = gpu_decode(w, variant, codes)
    ref, _ = oracle_decode(w, variant, codes)
    assert st == 0
    assert_close(got, ref, f"workers={workers}")
    # every split merges to the same answer up to float rounding: the
    # probabilities reach PV as fp32 values (an exact f16 high + low pair), so
    # only the exp2 of differences taken against split-dependent running maxima
    # and the order of fp32 additions differ
    diff = float(np.max(np.abs(got - base)))
    print(f"\nsplit {variant} workers={workers}: max |diff| vs automatic {diff:.3e}")
    assert diff <= 1e-6


@pytest.mark.parametrize("mode", ["auto", "persistent"])
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (8, 2, 64), (14, 2, 64), (32, 8, 128),
                                      (16, 1, 128), (24, 2, 64), (4, 4, 64), (40, 2, 128),
                                      (32, 1, 64), (9, 1, 128)])
def test_group_sizes_and_edge_lengths(variant, hq, hkv, d, mode):
    # "auto": these small batches take the one-item-per-cluster launch;
    # "persistent": the same batch through the persistent workers + reduce
    lens = [1, 15, 16, 17, 0, 33, 255, 256, 257]
    w = W.random_case(7 * hq + d, num_seqs=len(lens), num_heads=hq, num_kv_heads=hkv,
                      head_dim=d, context_lens=lens)
    codes = oracle_codes(w, variant == "fp8")
    if mode == "persistent":
        with persistent_workers():
            got, st = gpu_decode(w, variant, codes)
    else:
        got, st = gpu_decode(w, variant, codes)
    ref, flags = oracle_decode(w, variant, codes)
    assert st == 0 and not flags.any()
    assert_close(got, ref, f"{hq}/{hkv}/{d}")
    assert np.all(got[4] == 0)  # empty context


@pytest.mark.parametrize("mode", ["auto", "persistent"])
@pytest.mark.parametrize("variant", VARIANTS)
def test_bad_block_id_and_bad_length_give_zeros_and_status(variant, mode):
    w = W.random_case(55, num_seqs=5, num_heads=8, num_kv_heads=2, head_dim=64,
                      context_lens=[40, 100, 64, 5, 70])
    codes = oracle_codes(w, variant == "fp8")
    tables = w.block_tables.copy()
    tables[1, 3] = w.num_blocks + 1000   # out of the pool, inside the context
    tables[4, 2] = -7
    lens = w.context_lens.copy()
    lens[2] = 10_000                     # beyond max_context_len
    if mode == "persistent":
        with persistent_workers():
            got, st = gpu_decode(w, variant, codes, max_context_len=100, tables=tables,
                                 lens=lens)
    else:
        got, st = gpu_decode(w, variant, codes, max_context_len=100, tables=tables, lens=lens)
    ref, flags = oracle_decode(w, variant, codes, max_context_len=100, tables=tables, lens=lens)
    assert st == pkv.PKV_DEV_BAD_BLOCK | pkv.PKV_DEV_BAD_CTX
    for s in (1, 2, 4):
        assert np.all(got[s] == 0) and np.all(ref[s] == 0)
    assert_close(got, ref, "bad inputs")


@pytest.mark.parametrize("variant", VARIANTS)
def test_side_stream_and_determinism(variant):
    w = W.random_case(66, num_seqs=12, num_heads=32, num_kv_heads=8, head_dim=128, max_ctx=700)
    codes = oracle_codes(w, variant == "fp8")
    s = torch.cuda.Stream()
    a, _ = gpu_decode(w, variant, codes, stream=s)
    b, _ = gpu_decode(w, variant, codes, stream=s)
    c, _ = gpu_decode(w, variant, codes)
    assert np.array_equal(a, b) and np.array_equal(a, c)
    ref, _ = oracle_decode(w, variant, codes)
    assert_close(a, ref, "side stream")


def test_all_empty_contexts_write_zeros():
    w = W.random_case(77, num_seqs=3, num_heads=8, num_kv_heads=2, head_dim=128,
                      context_lens=[0, 0, 0])
    got, st = gpu_decode(w, "fp16", max_context_len=0)
    assert st == 0 and np.all(got == 0)
    with persistent_workers():
        got, st = gpu_decode(w, "fp16", max_context_len=0)
    assert st == 0 and np.all(got == 0)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["c1_tiny", "c2_8x512", "c4_qwen2_b8"])
def test_small_configs_both_launches_agree(name, variant):
    # the one-item-per-cluster launch and the persistent workers + reduce give
    # the oracle's answer and agree with each other to float rounding
    w, codes = workload(name, variant)
    got, st = gpu_decode(w, variant, codes)
    with persistent_workers():
        alt, st2 = gpu_decode(w, variant, codes)
    ref, _ = oracle_decode(w, variant, codes)
    assert st == 0 and st2 == 0
    assert_close(got, ref, f"{name}/{variant} cluster")
    assert_close(alt, ref, f"{name}/{variant} persistent")
    assert float(np.max(np.abs(got - alt))) <= 1e-6

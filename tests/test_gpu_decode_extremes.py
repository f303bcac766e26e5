"""Paged decode at the extremes of its work decomposition, against the oracle.

* One long sequence among short ones: its single work item is spread over
  dozens of workers, so the split-context reduce merges more than 32 pieces
  of one item (the path that reads the pieces' maxima 32 at a time).
* A few long items over the whole grid (one worker per eight pages): more
  than eight pieces per item on average, merged by the reduce that gives
  each task up to eight CTAs whose warps each take chunks of eight pieces
  (the last CTA to finish combines the CTAs' partials in a fixed order, so
  repeated calls give the same bits); with a maximum context far above the
  real ones, most workers hold no pages at all, and with many tasks fewer
  CTAs share a task and they loop over the tasks.
* The largest batch the decode accepts (8192 sequences): the per-sequence
  tables fill the most shared memory and are built in many passes.
* A quantize + decode step captured once in a CUDA graph and replayed on new
  inputs gives the same bits as the same calls made directly.
"""
import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import (assert_close, dev, ensure_built, gpu_decode, oracle_codes,
                        oracle_decode)

pytestmark = pytest.mark.gpu

VARIANTS = ["fp16", "int8", "fp8"]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("workers", [0, 40])
def test_one_long_item_over_many_workers(variant, workers):
    # 16 items (one kv head): with at most four workers per item the grid has
    # 64 workers, and the 2048-page item takes ~63 of them (40 when capped)
    lens = [32768] + [16] * 15
    w = W.random_case(91, num_seqs=len(lens), num_heads=8, num_kv_heads=1, head_dim=128,
                      context_lens=lens)
    codes = oracle_codes(w, variant == "fp8")
    ensure_built()
    try:
        pkv.pkv_set_decode_workers(workers)
        got, st = gpu_decode(w, variant, codes)
    finally:
        pkv.pkv_set_decode_workers(0)
    ref, flags = oracle_decode(w, variant, codes)
    assert st == 0 and not flags.any()
    assert_close(got, ref, f"long item, workers={workers}")


MANY_PIECES = [
    # (query heads, kv heads, head_dim, context lengths, maximum context)
    (32, 8, 128, [32768], None),         # 8 items of 2048 pages, ~256 pieces each
    (16, 1, 64, [16384, 3, 0], None),    # two groups of 8 query heads per item
    (8, 1, 128, [2048, 0, 0, 0], 16384),  # most workers empty: the bound is 8x the pages
    (8, 1, 128, [300] * 16, 16384),     # 128 tasks: fewer CTAs per task
    (8, 1, 64, [300] * 48, 16384),      # 384 tasks, more than one wave: CTAs loop
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("case", range(len(MANY_PIECES)))
def test_items_over_many_pieces(variant, case):
    hq, hkv, d, lens, mcl = MANY_PIECES[case]
    w = W.random_case(95 + case, num_seqs=len(lens), num_heads=hq, num_kv_heads=hkv,
                      head_dim=d, context_lens=lens)
    codes = oracle_codes(w, variant == "fp8")
    tables = w.block_tables
    if mcl is not None:  # table rows wide enough for the maximum (block 0 past the ends)
        tables = np.zeros((len(lens), mcl // 16), dtype=np.int32)
        tables[:, :w.block_tables.shape[1]] = w.block_tables
    got, st = gpu_decode(w, variant, codes, max_context_len=mcl, tables=tables)
    ref, flags = oracle_decode(w, variant, codes, max_context_len=mcl, tables=tables)
    assert st == 0 and not flags.any()
    assert_close(got, ref, f"many pieces, case {case}")
    # the partials are combined in a fixed order, whichever CTA arrives last
    again, st = gpu_decode(w, variant, codes, max_context_len=mcl, tables=tables)
    assert st == 0 and np.array_equal(again.view(np.uint64), got.view(np.uint64))
    assert np.all(got[w.context_lens == 0] == 0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_bad_block_ids_in_items_over_many_pieces(variant):
    # ~190 pieces per long item, merged by several CTAs: a bad id in a middle
    # piece (sequence 0) and in the first piece (sequence 2) zeroes exactly
    # those sequences' outputs and sets the status flag
    lens = [16384, 300, 16384]
    w = W.random_case(98, num_seqs=3, num_heads=8, num_kv_heads=1, head_dim=128,
                      context_lens=lens)
    codes = oracle_codes(w, variant == "fp8")
    tables = w.block_tables.copy()
    tables[0, 700] = w.num_blocks + 5
    tables[2, 3] = -5
    got, st = gpu_decode(w, variant, codes, tables=tables)
    ref, flags = oracle_decode(w, variant, codes, tables=tables)
    assert st == pkv.PKV_DEV_BAD_BLOCK
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert np.all(ref[0] == 0) and np.all(ref[2] == 0)
    assert_close(got, ref, "bad ids over many pieces")


@pytest.mark.parametrize("variant", VARIANTS)
def test_largest_batch_of_sequences(variant):
    w = W.random_case(92, num_seqs=8192, num_heads=8, num_kv_heads=2, head_dim=64, max_ctx=40)
    codes = oracle_codes(w, variant == "fp8")
    got, st = gpu_decode(w, variant, codes)
    ref, flags = oracle_decode(w, variant, codes)
    assert st == 0 and not flags.any()
    assert_close(got, ref, "8192 sequences")
    assert np.all(got[w.context_lens == 0] == 0)


def test_quantize_and_decode_replayed_from_a_cuda_graph():
    ensure_built()
    w = W.random_case(93, num_seqs=24, num_heads=32, num_kv_heads=8, head_dim=128, max_ctx=600)
    n, hq, d = w.query.shape
    kf, vf = dev(w.k_pool), dev(w.v_pool)
    kc = torch.zeros(w.k_pool.shape, dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros(w.k_pool.shape[:2], dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, dev(w.used_block_ids))
    tails = dev(w.tail_block_ids())
    q, bt, cl = dev(w.query), dev(w.block_tables), dev(w.context_lens)
    out = torch.zeros((n, hq, d), dtype=torch.float32, device="cuda")
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, w.max_context_len)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, tails, status)
        pkv.pkv_paged_decode_int8(out, q, kc, vc, ks, vs, bt, cl, w.max_context_len,
                                  w.softmax_scale, ws, status)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # first call outside the capture: per-device set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    rng = np.random.default_rng(5)
    for _ in range(2):
        # new query and new tail-block contents, then replay
        q.copy_(torch.from_numpy(rng.standard_normal(w.query.shape).astype(np.float16)))
        for b in w.tail_block_ids():
            kf[int(b)].copy_(torch.from_numpy(
                rng.standard_normal(w.k_pool.shape[1:]).astype(np.float16)))
        g.replay()
        torch.cuda.synchronize()
        replayed = out.clone()
        kc_r = kc.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(kc_r, kc)
        assert torch.equal(replayed, out)
    assert int(status.item()) == 0
    # and the result is the oracle's for the final pools
    wq = dataclasses.replace(w, query=q.cpu().numpy(), k_pool=kf.cpu().numpy())
    codes = oracle_codes(wq)
    ref, _ = oracle_decode(wq, "int8", codes)
    assert_close(out.cpu().numpy().astype(np.float64), ref, "graph replay")

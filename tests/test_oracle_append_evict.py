"""Pins of the oracle's append and eviction functions to facts outside the oracle.

Append: the write is the inverse of the block-table gather ("PagedAttention &
KV-Cache Memory Management", section 2.1), so appending a sequence token by
token and then reading the pool back through the table must give the token
stream, and attention over it must equal dense attention computed by torch.

Eviction: the least-reference-count + age score of the same page (section
4.3.1), checked with exact rational arithmetic where alpha and beta are
binary fractions, and against two textbook special cases: equal reference
counts reduce it to least-recently-used, equal ages to least-reference-count.
"""
import math
from fractions import Fraction
from itertools import combinations

import numpy as np
import pytest
import torch

import oracle
import pkv_workloads as W

B = 16


def _pool(nb, hkv, d):
    return np.full((nb, hkv, B, d), np.nan, np.float16)


def _gather(pool, table_row, ctx):
    """Dense [Hkv][ctx][d] rows read with numpy indexing: block t // B, slot t % B."""
    t = np.arange(ctx)
    blk = table_row[t // B]
    return np.transpose(pool[blk, :, t % B, :], (1, 0, 2))


# --------------------------------------------------------------------------
# Token-by-token append into a shuffled pool, then a gather, returns the
# stream; every slot that was not written keeps its bit pattern.  Catches a
# swapped block/slot index, a row written to the wrong kv head, a write that
# spills into a neighbouring slot.
def test_append_token_by_token_then_gather_returns_the_stream():
    rng = np.random.default_rng(5)
    n, hkv, d = 3, 2, 8
    lens = [37, 16, 1]
    nb = 12
    perm = rng.permutation(nb).astype(np.int32)
    table = np.full((n, 3), -1, np.int32)
    off = 0
    for s, c in enumerate(lens):
        k = (c + B - 1) // B
        table[s, :k] = perm[off:off + k]
        off += k
    kp, vp = _pool(nb, hkv, d), _pool(nb, hkv, d)
    kp[perm[off:]] = 7.0                       # blocks no table uses
    k0, v0 = kp.copy(), vp.copy()
    stream_k = rng.standard_normal((n, max(lens), hkv, d)).astype(np.float16)
    stream_v = rng.standard_normal((n, max(lens), hkv, d)).astype(np.float16)
    for t in range(max(lens)):
        pos = np.array([t if t < c else -1 for c in lens], np.int32)
        kp, vp, flags, written = oracle.append_fp16(kp, vp, stream_k[:, t], stream_v[:, t],
                                                    table, pos)
        assert not flags.any()
        assert np.array_equal(written >= 0, pos >= 0)
    for s, c in enumerate(lens):
        assert np.array_equal(_gather(kp, table[s], c), np.transpose(stream_k[s, :c], (1, 0, 2)))
        assert np.array_equal(_gather(vp, table[s], c), np.transpose(stream_v[s, :c], (1, 0, 2)))
    # untouched slots: compare bit patterns (NaN == NaN there)
    touched = np.zeros((nb, B), bool)
    for s, c in enumerate(lens):
        for t in range(c):
            touched[table[s, t // B], t % B] = True
    mask = ~touched[:, None, :, None] & np.ones(kp.shape, bool)
    assert np.array_equal(kp.view(np.uint16)[mask], k0.view(np.uint16)[mask])
    assert np.array_equal(vp.view(np.uint16)[mask], v0.view(np.uint16)[mask])


# --------------------------------------------------------------------------
# Append the last token of each sequence, then decode: equals torch's fp64
# scaled_dot_product_attention over the dense stream with the new token at
# its end (a library routine, GQA expanded by torch).
@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (14, 2, 64), (32, 8, 128)])
def test_append_then_decode_equals_dense_sdpa(hq, hkv, d):
    w = W.random_case(300 + hq, num_seqs=5, num_heads=hq, num_kv_heads=hkv, head_dim=d,
                      context_lens=[1, 16, 17, 40, 64])
    kn, vn, pos = W.append_tokens(w, 17)
    kp, vp, flags, _ = oracle.append_fp16(w.k_pool, w.v_pool, kn, vn, w.block_tables, pos)
    assert not flags.any()
    got = oracle.decode_fp16(w.query, kp, vp, w.block_tables, w.context_lens,
                             num_kv_heads=hkv, softmax_scale=w.softmax_scale)
    for s, c in enumerate(w.context_lens.tolist()):
        dk = _gather(w.k_pool, w.block_tables[s], c - 1).astype(np.float64)
        dv = _gather(w.v_pool, w.block_tables[s], c - 1).astype(np.float64)
        dk = np.concatenate([dk, kn[s][:, None, :].astype(np.float64)], axis=1)
        dv = np.concatenate([dv, vn[s][:, None, :].astype(np.float64)], axis=1)
        q = torch.from_numpy(w.query[s].astype(np.float64))[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, torch.from_numpy(dk)[None], torch.from_numpy(dv)[None],
            scale=w.softmax_scale, enable_gqa=True)[0, :, 0, :].numpy()
        np.testing.assert_allclose(got[s], ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Edge cases: no token (position < 0), first and last slot of a block, a
# position past the table, a table entry outside the pool.  Flagged or
# skipped sequences write nothing.
def test_append_edge_positions_and_bad_inputs():
    rng = np.random.default_rng(9)
    n, hkv, d, nb = 6, 2, 8, 8
    table = np.array([[0, 1], [2, 3], [4, 5], [6, -1], [7, 99], [3, 2]], np.int32)
    pos = np.array([-1, 16, 15, 32, 20, 31], np.int32)
    kp = rng.standard_normal((nb, hkv, B, d)).astype(np.float16)
    vp = rng.standard_normal((nb, hkv, B, d)).astype(np.float16)
    kn = rng.standard_normal((n, hkv, d)).astype(np.float16)
    vn = rng.standard_normal((n, hkv, d)).astype(np.float16)
    k1, v1, flags, written = oracle.append_fp16(kp, vp, kn, vn, table, pos)
    assert flags.tolist() == [0, 0, 0, oracle.BAD_CTX, oracle.BAD_BLOCK, 0]
    assert written.tolist() == [-1, 3, 4, -1, -1, 2]
    expect_k, expect_v = kp.copy(), vp.copy()
    for s, blk, slot in [(1, 3, 0), (2, 4, 15), (5, 2, 15)]:
        expect_k[blk, :, slot] = kn[s]
        expect_v[blk, :, slot] = vn[s]
    assert np.array_equal(k1, expect_k) and np.array_equal(v1, expect_v)


# --------------------------------------------------------------------------
# INT8 append: every written tile is re-quantized from its new fp16 content.
# Pinned by the quantizer's error bound (|x - code * scale| <= scale / 2 plus
# fp32 rounding) and the absmax element reaching +-127, on the new row too;
# tiles not written keep their codes and scales bit for bit.
def test_append_int8_requantizes_written_tiles_only():
    w = W.random_case(41, num_seqs=4, num_heads=8, num_kv_heads=2, head_dim=64,
                      context_lens=[5, 16, 33, 0])
    kc, ks = oracle.quantize(w.k_pool, block_ids=w.used_block_ids)
    vc, vs = oracle.quantize(w.v_pool, block_ids=w.used_block_ids)
    kn, vn, pos = W.append_tokens(w, 3)
    kn[0, 1, 5] = 40.0                        # new row holds the tile's absmax
    kp, vp, kc2, vc2, ks2, vs2, flags = oracle.append_int8(
        w.k_pool, w.v_pool, kc, vc, ks, vs, kn, vn, w.block_tables, pos)
    assert not flags.any()
    tails = set(w.tail_block_ids().tolist())
    for blk in range(w.num_blocks):
        for h in range(w.num_kv_heads):
            for pool, codes, sc, oldc, olds in ((kp, kc2, ks2, kc, ks), (vp, vc2, vs2, vc, vs)):
                if blk not in tails:
                    assert np.array_equal(codes[blk, h], oldc[blk, h])
                    assert sc[blk, h].view(np.uint32) == olds[blk, h].view(np.uint32)
                    continue
                x = pool[blk, h].astype(np.float64)
                ok = ~np.isnan(x)
                scale = float(sc[blk, h])
                assert scale == np.float32(np.nanmax(np.abs(x))) / np.float32(127)
                err = np.abs(x[ok] - codes[blk, h][ok] * scale)
                assert err.max() <= scale * (0.5 + 2.0 ** -16)
                assert np.abs(codes[blk, h]).max() == 127
    s0_blk = w.block_tables[0, 4 // B]
    assert kc2[s0_blk, 1, 4, 5] == 127        # 40 / (40 / 127) -> 127


# --------------------------------------------------------------------------
# Eviction score with binary-fraction weights (alpha 3/4, beta 1/4): every
# fp32 operation is exact for these small integers, so the score must equal
# the rational value of the formula.  Catches a flipped sign of either
# difference, a dropped term, max_refcnt taken over free blocks' zeros, or
# the weights swapped.
def test_evict_scores_exact_with_binary_weights():
    st = W.eviction_state(3000, 11, max_age=500)
    sc, cand = oracle.evict_scores(st.refcnt, st.last_used, st.current_tick, 0.75, 0.25)
    m = int(st.refcnt.max())
    assert cand == int((st.refcnt > 0).sum())
    for b in range(st.refcnt.size):
        r = int(st.refcnt[b])
        if r <= 0:
            assert sc[b] == -np.inf
            continue
        exact = Fraction(3, 4) * (m - r) + Fraction(1, 4) * (st.current_tick - int(st.last_used[b]))
        assert Fraction(float(sc[b])) == exact


# --------------------------------------------------------------------------
# Brute force on tiny pools: with binary weights the exact scores order the
# blocks, and the chosen set must be the best size-n subset under the order
# (larger score first, equal scores to the smaller id) -- found here by
# enumerating every subset.
@pytest.mark.parametrize("seed", range(6))
def test_evict_select_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    nb = 9
    ref = rng.integers(0, 4, size=nb).astype(np.int32)
    tick = 20
    last = (tick - rng.integers(0, 4, size=nb)).astype(np.int64)
    cand = [b for b in range(nb) if ref[b] > 0]
    m = max([int(r) for r in ref] + [0])
    exact = {b: Fraction(3, 4) * (m - int(ref[b])) + Fraction(1, 4) * (tick - int(last[b]))
             for b in cand}
    for k in range(nb + 2):
        got, _ = oracle.evict_select(ref, last, tick, k, 0.75, 0.25)
        n = min(k, len(cand))
        best = None
        for sub in combinations(cand, n):
            key = sorted(((-exact[b], b) for b in sub))
            # a subset is better when its sorted (score desc, id asc) list is smaller
            if best is None or key < best[0]:
                best = (key, sub)
        assert got.tolist() == sorted(best[1])


# --------------------------------------------------------------------------
# Equal reference counts: the score reduces to beta * age, so the choice is
# least-recently-used (smallest last_used, ties to the smaller id); equal
# ages reduce it to the smallest reference counts.  Pages' weights 0.7/0.3.
def test_evict_equal_refcounts_is_lru_and_equal_ages_is_lrc():
    rng = np.random.default_rng(2)
    nb, k = 4000, 600
    last = (50_000 - rng.integers(0, 3000, size=nb)).astype(np.int64)
    ref = np.full(nb, 2, np.int32)
    got, _ = oracle.evict_select(ref, last, 50_000, k)
    lru = np.lexsort((np.arange(nb), last))[:k]          # oldest first, then id
    assert got.tolist() == sorted(lru.tolist())
    ref = rng.integers(1, 9, size=nb).astype(np.int32)
    last = np.full(nb, 50_000, np.int64)
    got, _ = oracle.evict_select(ref, last, 50_000, k)
    lrc = np.lexsort((np.arange(nb), ref))[:k]
    assert got.tolist() == sorted(lrc.tolist())


# --------------------------------------------------------------------------
# Invariants: free blocks are never chosen, the count is min(k, candidates),
# ids ascend, and k = 0 or an all-free pool chooses nothing.
def test_evict_select_invariants():
    st = W.eviction_state(5000, 4)
    cand = int((st.refcnt > 0).sum())
    for k in (0, 1, 750, cand, cand + 10):
        ids, scores = oracle.evict_select(st.refcnt, st.last_used, st.current_tick, k)
        assert ids.size == min(k, cand)
        assert np.all(np.diff(ids) > 0)
        assert np.all(st.refcnt[ids] > 0)
        if 0 < ids.size < cand:
            rest = np.setdiff1d(np.nonzero(st.refcnt > 0)[0], ids)
            worst_in = scores[ids].min()
            assert worst_in >= scores[rest].max()
    ids, _ = oracle.evict_select(np.zeros(10, np.int32), np.zeros(10, np.int64), 5, 3)
    assert ids.size == 0


# --------------------------------------------------------------------------
# fp32 rounding of the pages' weights: 0.7 and 0.3 are not binary fractions,
# so each product is rounded once.  The score of refcnt gap 1 and age 0 is
# fp32(0.7) exactly; age 1 and gap 0 is fp32(0.3); gap 1 and age 1 is
# fp32(fp32(0.7) + fp32(0.3)) = 1 (the rounded sum).  Catches a score
# evaluated in fp64 or with a fused multiply-add.
def test_evict_scores_fp32_rounding_of_page_weights():
    ref = np.array([1, 2, 2, 1], np.int32)
    last = np.array([10, 10, 9, 9], np.int64)
    sc, _ = oracle.evict_scores(ref, last, 10)
    f = np.float32
    assert sc[0] == f(0.7) and sc[1] == 0.0 and sc[2] == f(0.3)
    assert sc[3] == f(f(0.7) + f(0.3))
    assert sc[0].view(np.uint32) == np.float32(0.7).view(np.uint32)
    assert math.isclose(float(sc[3]), 1.0, abs_tol=0)

"""Eviction scoring + choice of the blocks to evict on the GPU against the CPU
oracle: scores bit-exact (same fp32 operations), chosen ids and count exact,
over pool sizes from one block to the largest single cluster, with the pages'
weights and with special cases (all ties, all free, huge ticks, overflowing
weights)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import ensure_built

pytestmark = pytest.mark.gpu


def gpu_evict(refcnt, last_used, tick, k, alpha=0.7, beta=0.3):
    ensure_built()
    ref = torch.from_numpy(np.ascontiguousarray(refcnt, np.int32)).cuda()
    last = torch.from_numpy(np.ascontiguousarray(last_used, np.int64)).cuda()
    scores = torch.full((ref.numel(),), 12345.0, dtype=torch.float32, device="cuda")
    ids = torch.full((max(k, 1),), -7, dtype=torch.int32, device="cuda")
    count = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    pkv.pkv_evict_select(ref, last, tick, k, ids, count, scores, alpha, beta)
    torch.cuda.synchronize()
    n = int(count.item())
    return ids.cpu().numpy(), n, scores.cpu().numpy()


def check(refcnt, last_used, tick, k, alpha=0.7, beta=0.3):
    ids, n, scores = gpu_evict(refcnt, last_used, tick, k, alpha, beta)
    want, want_scores = oracle.evict_select(refcnt, last_used, tick, k, alpha, beta)
    assert np.array_equal(scores.view(np.uint32), want_scores.view(np.uint32))
    assert n == want.size
    assert np.array_equal(ids[:n], want)
    assert np.all(ids[n:k] == -1)
    return n


def max_pool_blocks():
    # the largest pool one launch takes: 16-CTA clusters where the device
    # schedules them, else 8; probed through the documented size limit
    ensure_built()
    ref = torch.zeros(16 * 49152 + 1, dtype=torch.int32, device="cuda")
    last = torch.zeros_like(ref, dtype=torch.int64)
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    for nb in (16 * 49152, 8 * 49152):
        try:
            pkv.pkv_evict_select(ref[:nb], last[:nb], 0, 0, None, count)
            torch.cuda.synchronize()
            return nb
        except pkv.PkvError as e:
            assert e.status == pkv.PKV_ERR_UNSUPPORTED
    raise AssertionError("no supported pool size")


@pytest.mark.parametrize("nb", [1, 7, 1000, 1024, 4096, 4097, 16384, 65536, 262144])
def test_pool_sizes_and_k(nb):
    st = W.eviction_state(nb, nb)
    cand = int((st.refcnt > 0).sum())
    for k in sorted({0, 1, pkv.evict_count(nb), max(cand - 1, 0), cand, cand + 3, nb + 5}):
        assert check(st.refcnt, st.last_used, st.current_tick, k) == min(k, cand)


def test_largest_pool_one_launch_takes():
    nb = max_pool_blocks()
    st = W.eviction_state(nb, 3)
    check(st.refcnt, st.last_used, st.current_tick, pkv.evict_count(nb))
    ensure_built()
    ref = torch.ones(nb + 1, dtype=torch.int32, device="cuda")
    last = torch.zeros(nb + 1, dtype=torch.int64, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_evict_select(ref, last, 0, 0, None, count)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED


def test_all_ties_take_the_smallest_ids():
    nb = 20000
    ref = np.full(nb, 3, np.int32)
    last = np.full(nb, 50, np.int64)
    for k in (1, 999, 12345):
        ids, n, _ = gpu_evict(ref, last, 60, k)
        assert n == k and np.array_equal(ids[:n], np.arange(k))


def test_all_free_and_mixed_free():
    nb = 9000
    ids, n, scores = gpu_evict(np.zeros(nb, np.int32), np.zeros(nb, np.int64), 5, 100)
    assert n == 0 and np.all(ids[:100] == -1) and np.all(scores == -np.inf)
    rng = np.random.default_rng(1)
    ref = rng.integers(-3, 3, size=nb).astype(np.int32)     # negatives count as free
    last = rng.integers(0, 100, size=nb).astype(np.int64)
    check(ref, last, 100, 500)


def test_large_ticks_negative_ages_and_extreme_weights():
    rng = np.random.default_rng(8)
    nb = 30000
    ref = rng.integers(1, 40, size=nb).astype(np.int32)
    tick = 3 * (1 << 40) + 17
    last = tick - rng.integers(-1000, 1 << 33, size=nb)       # some uses "in the future"
    check(ref, last.astype(np.int64), tick, 4000)
    check(ref, last.astype(np.int64), tick, 4000, alpha=0.0, beta=1.0)     # pure LRU
    check(ref, last.astype(np.int64), tick, 4000, alpha=1.0, beta=0.0)     # pure LRC
    check(ref, last.astype(np.int64), tick, 4000, alpha=-0.5, beta=0.25)   # negative weight
    # products overflow to +-inf; inf - inf is NaN and counts as -inf
    check(ref, last.astype(np.int64), tick, 4000, alpha=3e38, beta=-3e38)

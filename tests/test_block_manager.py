"""The library's native block manager (C++, host) against the block-manager
model of the oracle, operation by operation: same ids, same copy pairs, same
refusals, same counts and figures.  Host code only: runs without a GPU."""
import random

import numpy as np
import pytest

import paged_kv_cache_234_gb300 as pkv
from oracle.block_manager import NO_HASH, BlockManagerModel
from paged_kv_cache_234_gb300 import build as pkv_build


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv_build.build()
    pkv.lib()


def same_state(bm, model):
    assert np.array_equal(bm.refcounts(), np.asarray(model.refcnt, np.int32))
    a, b = bm.stats(), model.stats()
    for key in ("free", "used", "shared", "logical", "tokens"):
        assert a[key] == b[key], key
    for key in ("internal_fragmentation", "sharing_saving"):
        assert a[key] == pytest.approx(b[key], abs=1e-12), key


def refused(fn, *args):
    try:
        fn(*args)
    except pkv.PkvError as e:
        return e.status
    return None


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_model(seed):
    rng = random.Random(100 + seed)
    n_blocks = rng.choice([1, 7, 64, 200])
    bm, model = pkv.BlockManager(n_blocks), BlockManagerModel(n_blocks)
    seqs = []
    for step in range(2500):
        op = rng.random()
        if op < 0.3:
            hs = [rng.choice([NO_HASH, NO_HASH, rng.randrange(1, 9), rng.getrandbits(64) | 1])
                  for _ in range(rng.randrange(0, 7))]
            want = model.allocate(hs)
            if want is None:
                assert refused(bm.allocate, hs) == pkv.PKV_ERR_EXHAUSTED
            else:
                got = bm.allocate(hs)
                assert got.tolist() == want
                seqs.append(list(want))
        elif op < 0.45 and seqs:
            s = seqs.pop(rng.randrange(len(seqs)))
            assert model.free(s)
            bm.free(s)
        elif op < 0.55 and seqs:
            s = rng.choice(seqs)
            assert model.fork(s)
            bm.fork(s)
            seqs.append(list(s))
        elif op < 0.8 and seqs:
            s = rng.choice(seqs)
            idx = sorted(rng.sample(range(len(s)), rng.randrange(1, len(s) + 1))) if s else []
            ids = [s[i] for i in idx]
            want = model.cow_batch(ids)
            if want is None:
                assert refused(bm.cow, ids) == pkv.PKV_ERR_EXHAUSTED
            else:
                got, pairs = bm.cow(ids)
                assert got.tolist() == want[0]
                assert [tuple(p) for p in pairs.tolist()] == want[1]
                for i, b in zip(idx, want[0]):
                    s[i] = b
        elif op < 0.9 and seqs:
            s = rng.choice(seqs)
            toks = [rng.randrange(0, 17) for _ in s]
            assert model.set_fill(s, toks)
            bm.set_fill(s, toks)
        else:
            # refused calls change nothing on either side
            bad = [n_blocks + 3] if rng.random() < 0.5 else [-1]
            assert refused(bm.free, bad) == pkv.PKV_ERR_INVALID_ARG and not model.free(bad)
            assert refused(bm.fork, bad) == pkv.PKV_ERR_INVALID_ARG
            assert refused(bm.set_fill, [0], [17]) == pkv.PKV_ERR_INVALID_ARG
        if step % 50 == 0:
            same_state(bm, model)
    same_state(bm, model)
    bm.close()


def test_over_free_and_duplicate_ids():
    bm, model = pkv.BlockManager(8), BlockManagerModel(8)
    ids = bm.allocate(2)
    model.allocate([NO_HASH, NO_HASH])
    assert refused(bm.free, [ids[0], ids[0]]) == pkv.PKV_ERR_INVALID_ARG
    assert not model.free([int(ids[0]), int(ids[0])])
    bm.fork([ids[0]])
    model.fork([int(ids[0])])
    bm.free([ids[0], ids[0]])
    assert model.free([int(ids[0]), int(ids[0])])
    same_state(bm, model)
    # the same shared block written twice in one call: one copy, then the
    # original is exclusive
    bm.fork([ids[1]])
    model.fork([int(ids[1])])
    got, pairs = bm.cow([ids[1], ids[1]])
    want = model.cow_batch([int(ids[1]), int(ids[1])])
    assert got.tolist() == want[0] and [tuple(p) for p in pairs.tolist()] == want[1]
    same_state(bm, model)


def test_pages_figures_through_the_native_manager():
    # 3 sequences sharing a 4-block prompt: 66.7 % saved
    bm = pkv.BlockManager(32)
    for _ in range(3):
        assert bm.allocate([11, 12, 13, 14]).tolist() == [0, 1, 2, 3]
    assert round(100 * bm.stats()["sharing_saving"], 1) == 66.7
    # 8 beams over 70 tokens: 7 copies of the tail block on divergence
    bm = pkv.BlockManager(64)
    ids = bm.allocate(5)
    bm.set_fill(ids, [16, 16, 16, 16, 6])
    for _ in range(7):
        bm.fork(ids)
    copies = sum(bm.cow([ids[-1]])[1].shape[0] for _ in range(8))
    assert copies == 7 and bm.stats()["used"] == 12


def test_create_rejects_bad_sizes():
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(-1)
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(4, 0)
    bm = pkv.BlockManager(0)
    assert refused(bm.allocate, 1) == pkv.PKV_ERR_EXHAUSTED
    assert bm.allocate(0).size == 0


def test_threads_share_one_manager():
    # every call takes the manager's lock: eight threads allocating (some
    # blocks shared by prefix hash across threads), forking, copying on write
    # and freeing leave the manager consistent and, at the end, fully free
    import threading

    bm = pkv.BlockManager(4096)
    errors = []

    def worker(tid):
        rng = random.Random(1000 + tid)
        try:
            for _ in range(300):
                held = []
                n = rng.randint(1, 16)
                hashes = [rng.choice([NO_HASH, NO_HASH, 7 + rng.randrange(8)]) for _ in range(n)]
                ids = bm.allocate(hashes)
                fresh = [int(b) for b, h in zip(ids, hashes) if h == NO_HASH]
                assert len(set(fresh)) == len(fresh)
                held += [int(b) for b in ids]
                if rng.random() < 0.5:
                    f = [int(b) for b in ids[: rng.randint(1, n)]]
                    bm.fork(f)
                    held += f
                if rng.random() < 0.5:
                    k = rng.randint(1, len(held))
                    src = held[:k]
                    new, _ = bm.cow(src)
                    held = [int(b) for b in new] + held[k:]
                bm.free(held)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:3]
    st = bm.stats()
    assert st["free"] == 4096 and st["used"] == 0 and st["logical"] == 0
    assert not bm.refcounts().any()

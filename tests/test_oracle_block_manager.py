"""Pins of the block-manager model to the pages' figures and to invariants
that an independent record of the sequences' block lists must satisfy."""
import random

import pytest

from oracle.block_manager import NO_HASH, BlockManagerModel, blocks_for_tokens

KIB = 1024


# --------------------------------------------------------------------------
# "paged-attention-runtime" summary, STATUS: prefix sharing validated with a
# "66.7% reduction".  Three sequences with the same prompt hold one copy of
# its blocks: 1 - 1/3 of the logical blocks saved.  Catches a prefix cache
# that does not share, or shares without counting references.
def test_prefix_sharing_three_sequences_saves_two_thirds():
    bm = BlockManagerModel(64)
    prompt = [0x1001, 0x1002, 0x1003, 0x1004]
    ids = [bm.allocate(prompt) for _ in range(3)]
    assert ids[0] == ids[1] == ids[2] == [0, 1, 2, 3]
    st = bm.stats()
    assert (st["used"], st["logical"], st["shared"]) == (4, 12, 4)
    assert round(100 * st["sharing_saving"], 1) == 66.7


# --------------------------------------------------------------------------
# "PagedAttention & KV-Cache Memory Management", section 2.2: a 73-token
# prefill with B = 16 takes 5 pages and leaves part of the last one unused
# (the page prints 9 for the last page; 9 is its used slots, 7 are empty).
def test_seventy_three_tokens_take_five_pages():
    assert blocks_for_tokens(73) == 5
    bm = BlockManagerModel(16)
    ids = bm.allocate([NO_HASH] * blocks_for_tokens(73))
    assert bm.set_fill(ids, [16, 16, 16, 16, 9])
    st = bm.stats()
    assert st["tokens"] == 73 and st["used"] == 5
    assert st["internal_fragmentation"] == pytest.approx(7 / 80, abs=1e-15)


# --------------------------------------------------------------------------
# Same page, section 4.1.1: 8 beams over a 70-token context with 128 KB of KV
# per token: about 71 MiB without sharing, about 23 MiB with copy-on-write.
# The beams share the 5 blocks; when each beam writes its next token into the
# shared tail block, 7 beams get a copy and the last keeps the original: 12
# physical blocks instead of 40, and the page's token-level figure
# (70 + 7 x 16) x 128 KiB = 22.75 MiB.  Catches a CoW that copies for the
# last holder too, or forgets to drop the old reference.
def test_eight_beams_copy_on_write():
    bm = BlockManagerModel(64)
    ctx, beams = 70, 8
    ids = bm.allocate([NO_HASH] * blocks_for_tokens(ctx))
    bm.set_fill(ids, [16, 16, 16, 16, 6])
    for _ in range(beams - 1):
        assert bm.fork(ids)
    assert (bm.stats()["used"], bm.stats()["logical"]) == (5, 40)
    copies = 0
    for _ in range(beams):
        new, copied = bm.cow(ids[-1])
        copies += copied
        assert bm.fill[new] == 6
    assert copies == beams - 1
    assert bm.stats()["used"] == 12 and bm.stats()["logical"] == 40
    no_share_mib = beams * ctx * 128 * KIB / 2**20
    cow_mib = (ctx + copies * 16) * 128 * KIB / 2**20
    assert round(no_share_mib) == 70 and abs(no_share_mib - 71) < 1.5   # "≈ 71 MiB"
    assert cow_mib == 22.75 and round(cow_mib) == 23                     # "≈ 23 MiB"


# --------------------------------------------------------------------------
# Free-list order and all-or-nothing allocation: a fresh pool hands out
# 0, 1, 2, ...; a freed block is handed out next; a request that cannot be
# served changes nothing.
def test_free_list_order_and_exhaustion():
    bm = BlockManagerModel(4)
    assert bm.allocate([NO_HASH] * 3) == [0, 1, 2]
    assert bm.free([1])
    assert bm.allocate([NO_HASH]) == [1]
    before = (list(bm.refcnt), list(bm.free_list))
    assert bm.allocate([NO_HASH] * 2) is None
    assert (list(bm.refcnt), list(bm.free_list)) == before
    assert bm.allocate([NO_HASH]) == [3]
    assert bm.cow(3) == (3, False)
    assert bm.fork([3]) and bm.cow(3) is None  # shared, and no free block


# --------------------------------------------------------------------------
# Invariants under a random workload, checked against an independent record
# of every sequence's block list: each block's count is the number of list
# entries naming it; free and used blocks partition the pool; cached hashes
# point at used blocks registered under them; stats add up.
@pytest.mark.parametrize("seed", range(4))
def test_random_workload_invariants(seed):
    rng = random.Random(seed)
    bm = BlockManagerModel(96)
    seqs = []
    for _ in range(3000):
        op = rng.random()
        if op < 0.35:
            hs = [rng.choice([NO_HASH, NO_HASH, rng.randrange(1, 12)]) for _ in range(rng.randrange(1, 6))]
            got = bm.allocate(hs)
            if got is not None:
                seqs.append(list(got))
        elif op < 0.55 and seqs:
            s = seqs.pop(rng.randrange(len(seqs)))
            assert bm.free(s)
        elif op < 0.7 and seqs:
            s = rng.choice(seqs)
            assert bm.fork(s)
            seqs.append(list(s))
        elif op < 0.9 and seqs:
            s = rng.choice(seqs)
            i = rng.randrange(len(s))
            r = bm.cow(s[i])
            if r is not None:
                s[i] = r[0]
        elif seqs:
            s = rng.choice(seqs)
            bm.set_fill(s, [rng.randrange(0, 17) for _ in s])
        refs = [0] * bm.num_blocks
        for s in seqs:
            for b in s:
                refs[b] += 1
        assert refs == bm.refcnt
        free = set(bm.free_list)
        assert len(free) == len(bm.free_list)
        assert free == {b for b in range(bm.num_blocks) if bm.refcnt[b] == 0}
        for h, b in bm.cache.items():
            assert bm.refcnt[b] > 0 and bm.hash_of[b] == h
        st = bm.stats()
        assert st["free"] + st["used"] == bm.num_blocks
        assert st["logical"] == sum(len(s) for s in seqs)

"""Batched block copies (copy-on-write) on the GPU: every pool's bytes of each
source block land in its destination bit for bit and nothing else changes;
and a beam-search step through the block manager -- fork, copy-on-write of
the shared tail block, append, decode -- matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import assert_close, dev, ensure_built
from oracle.block_manager import BlockManagerModel

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hkv,d", [(8, 128), (2, 64), (1, 64)])
def test_copy_blocks_all_pools_bit_exact(hkv, d):
    ensure_built()
    rng = np.random.default_rng(hkv * 100 + d)
    nb = 300
    kf = rng.standard_normal((nb, hkv, 16, d)).astype(np.float16)
    vf = rng.standard_normal((nb, hkv, 16, d)).astype(np.float16)
    kc = rng.integers(-127, 128, (nb, hkv, 16, d), dtype=np.int8)
    ks = rng.random((nb, hkv)).astype(np.float32)  # 4-byte path when hkv % 4 != 0
    pools = [kf, vf, kc, ks]
    src = rng.choice(nb, 90, replace=False)
    dst = np.setdiff1d(np.arange(nb), src)[rng.permutation(nb - 90)[:90]]
    pairs = np.stack([src, dst], 1).astype(np.int32)
    pairs[5] = [7, 7]                      # no-op
    pairs[6] = [nb + 1, 3]                 # bad id: skipped, reported
    want = [p.copy() for p in pools]
    for s, t in pairs:
        if 0 <= s < nb and 0 <= t < nb and s != t:
            for w, p in zip(want, pools):
                w[t] = p[s]
    dpools = [dev(p) for p in pools]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_copy_blocks(dpools, dev(pairs), status)
    torch.cuda.synchronize()
    assert int(status.item()) == pkv.PKV_DEV_BAD_BLOCK
    for got, w in zip(dpools, want):
        g = got.cpu().numpy()
        assert np.array_equal(g.view(np.uint8), w.view(np.uint8))


def test_beam_fork_copy_on_write_append_decode():
    """Four beams share a 70-token prefix; each appends its own next token.
    The block manager gives the first three a copy of the shared tail block
    (the last keeps the original), the GPU copies it, appends each beam's
    token, and the decode of every beam equals the oracle's over its own
    dense history."""
    ensure_built()
    beams, ctx, hq, hkv, d = 4, 70, 32, 8, 128
    nb = 64
    base = W.random_case(5, num_seqs=1, num_heads=hq, num_kv_heads=hkv, head_dim=d,
                         context_lens=[ctx], extra_blocks=nb - 5, nan_padding=False)
    bm = pkv.BlockManager(base.num_blocks)
    model = BlockManagerModel(base.num_blocks)
    ids = bm.allocate(5)
    assert ids.tolist() == model.allocate([0] * 5)
    # the prompt's KV lives in blocks 0..4 of the pool (place it there)
    kp = base.k_pool.copy()
    vp = base.v_pool.copy()
    src_blocks = base.block_tables[0, :5]
    kp[ids] = base.k_pool[src_blocks]
    vp[ids] = base.v_pool[src_blocks]
    for _ in range(beams - 1):
        bm.fork(ids)
        model.fork(ids.tolist())
    tables = np.tile(ids, (beams, 1)).astype(np.int32)
    tail = int(ids[-1])
    pairs = []
    for b in range(beams):
        new, pr = bm.cow([tail])
        nm = model.cow_batch([tail])
        assert new.tolist() == nm[0] and [tuple(x) for x in pr.tolist()] == nm[1]
        tables[b, -1] = new[0]
        pairs += pr.tolist()
    assert len(pairs) == beams - 1
    kd, vd = dev(kp), dev(vp)
    pkv.pkv_copy_blocks([kd, vd], dev(np.asarray(pairs, np.int32)))
    rng = np.random.default_rng(9)
    kn = rng.standard_normal((beams, hkv, d)).astype(np.float16)
    vn = rng.standard_normal((beams, hkv, d)).astype(np.float16)
    pos = np.full(beams, ctx, np.int32)          # token 70: slot 6 of the tail block
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_append_fp16(kd, vd, dev(kn), dev(vn), dev(tables), dev(pos), status)
    q = rng.standard_normal((beams, hq, d)).astype(np.float16)
    lens = np.full(beams, ctx + 1, np.int32)
    out = torch.empty((beams, hq, d), dtype=torch.float32, device="cuda")
    ws = pkv.decode_workspace(beams, hq, hkv, d, ctx + 1)
    pkv.pkv_paged_decode_fp16(out, dev(q), kd, vd, dev(tables), dev(lens), ctx + 1,
                              1.0 / np.sqrt(d), ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # oracle: the same copies and appends on the host pools, then decode
    rk, rv = kp.copy(), vp.copy()
    for s, t in pairs:
        rk[t], rv[t] = rk[s], rv[s]
    rk, rv, flags, _ = oracle.append_fp16(rk, rv, kn, vn, tables, pos)
    assert not flags.any()
    want = oracle.decode_fp16(q, rk, rv, tables, lens, num_kv_heads=hkv,
                              softmax_scale=1.0 / np.sqrt(d))
    assert_close(out.cpu().numpy().astype(np.float64), want, "beams")
    # the beams differ only in their last token, and their shared prefix blocks are one copy
    assert len(set(tables[:, :-1].ravel().tolist())) == 4
    assert len(set(tables[:, -1].tolist())) == beams

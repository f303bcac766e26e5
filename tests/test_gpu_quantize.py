"""INT8 quantizer on the GPU: codes and scales bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import dev, ensure_built

pytestmark = pytest.mark.gpu


def gpu_quantize(k, v, block_ids=None, init_codes=None, init_scales=None):
    ensure_built()
    kd, vd = dev(k), dev(v)
    nb, hkv = k.shape[:2]
    if init_codes is None:
        kc = torch.zeros(k.shape, dtype=torch.int8, device="cuda")
        vc = torch.zeros(k.shape, dtype=torch.int8, device="cuda")
        ks = torch.zeros((nb, hkv), dtype=torch.float32, device="cuda")
        vs = torch.zeros((nb, hkv), dtype=torch.float32, device="cuda")
    else:
        kc, vc = dev(init_codes[0]), dev(init_codes[1])
        ks, vs = dev(init_scales[0]), dev(init_scales[1])
    ids = None if block_ids is None else dev(np.asarray(block_ids, np.int32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_quantize_blocks(kd, vd, kc, vc, ks, vs, ids, status)
    torch.cuda.synchronize()
    return (kc.cpu().numpy(), vc.cpu().numpy(), ks.cpu().numpy(), vs.cpu().numpy(),
            int(status.item()))


def assert_same(gpu, ref):
    assert np.array_equal(gpu[0], ref[0])
    assert np.array_equal(gpu[1].view(np.uint32), ref[1].view(np.uint32))


@pytest.mark.parametrize("name", ["c1_tiny", "c2_8x512", "c3_32x1024_heavy", "c4_qwen2_b8"])
def test_whole_pool_bit_exact(name):
    w = W.make(name)
    kc, vc, ks, vs, st = gpu_quantize(w.k_pool, w.v_pool)
    assert st == 0
    assert_same((kc, ks), oracle.quantize(w.k_pool))
    assert_same((vc, vs), oracle.quantize(w.v_pool))


@pytest.mark.parametrize("name", ["c5a_64x2048", "c5b_256_ragged"])
def test_full_size_used_blocks_bit_exact(name):
    w = W.make(name)
    ids = w.used_block_ids
    kc, vc, ks, vs, st = gpu_quantize(w.k_pool, w.v_pool, block_ids=ids)
    assert st == 0
    rk, rks = oracle.quantize(w.k_pool, block_ids=ids)
    rv, rvs = oracle.quantize(w.v_pool, block_ids=ids)
    assert_same((kc, ks), (rk, rks))
    assert_same((vc, vs), (rv, rvs))


@pytest.mark.parametrize("d", [64, 128])
def test_edge_tiles(d):
    rng = np.random.default_rng(d)
    x = (rng.standard_normal((12, 2, 16, d)) * 3).astype(np.float16)
    flat = x.reshape(12, 2, -1)
    flat[0, 0] = 0                                     # all zero
    flat[0, 1, :] = 0
    flat[0, 1, :9] = [127, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5, -3.5]  # ties at scale 1
    flat[1, 0, ::3] = np.nan                           # NaNs ignored in the max
    flat[1, 1, 5] = np.inf                             # inf: scale inf, codes 0
    flat[2, 0, :] = 65504.0                            # fp16 max
    flat[2, 1, :] = np.float16(6e-8)                   # subnormal fp16 only
    flat[3, 0, :] = -1.0
    flat[3, 0, 7] = 1.0
    flat[4, 1, :] = np.nan                             # all NaN
    kc, vc, ks, vs, st = gpu_quantize(x, x[::-1].copy())
    assert st == 0
    assert_same((kc, ks), oracle.quantize(x))
    assert_same((vc, vs), oracle.quantize(x[::-1].copy()))
    assert kc[0, 1, 0, 1] == 2 and kc[0, 1, 0, 2] == 4 and kc[0, 1, 0, 3] == -2


def test_block_ids_subset_duplicates_and_bad_ids():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((20, 4, 16, 128)).astype(np.float16)
    v = rng.standard_normal((20, 4, 16, 128)).astype(np.float16)
    sentinel_c = np.full(k.shape, 77, np.int8)
    sentinel_s = np.full((20, 4), 9.0, np.float32)
    ids = [3, 17, 3, -4, 25, 0, 17]
    kc, vc, ks, vs, st = gpu_quantize(k, v, block_ids=ids, init_codes=(sentinel_c, sentinel_c),
                                      init_scales=(sentinel_s, sentinel_s))
    assert st == pkv.PKV_DEV_BAD_BLOCK
    rk = oracle.quantize(k, block_ids=np.array(ids, np.int32), code_pool=sentinel_c,
                         scales=sentinel_s)
    rv = oracle.quantize(v, block_ids=np.array(ids, np.int32), code_pool=sentinel_c,
                         scales=sentinel_s)
    assert_same((kc, ks), rk)
    assert_same((vc, vs), rv)
    assert np.all(kc[5] == 77) and np.all(ks[5] == 9.0)

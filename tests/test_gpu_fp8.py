"""FP8 (OCP E4M3) quantizer and decode on the GPU against the CPU oracle:
codes and scales bit-exact (ties, saturation, NaN / inf / zero tiles), and
decode with NaN bytes in the padding slots of the code pools."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import assert_close, dev, ensure_built, gpu_decode, oracle_decode

pytestmark = pytest.mark.gpu


def gpu_quantize_fp8(k, v, block_ids=None):
    ensure_built()
    kd, vd = dev(k), dev(v)
    kc = torch.zeros(k.shape, dtype=torch.uint8, device="cuda")
    vc = torch.zeros(k.shape, dtype=torch.uint8, device="cuda")
    ks = torch.zeros(k.shape[:2], dtype=torch.float32, device="cuda")
    vs = torch.zeros(k.shape[:2], dtype=torch.float32, device="cuda")
    ids = None if block_ids is None else dev(np.asarray(block_ids, np.int32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_quantize_blocks_fp8(kd, vd, kc, vc, ks, vs, ids, status)
    torch.cuda.synchronize()
    return (kc.cpu().numpy(), vc.cpu().numpy(), ks.cpu().numpy(), vs.cpu().numpy(),
            int(status.item()))


def same(gc, gs, rc, rs):
    assert np.array_equal(gc, rc)
    assert np.array_equal(gs.view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("name", ["c1_tiny", "c2_8x512", "c3_32x1024_heavy", "c4_qwen2_b8"])
def test_quantize_fp8_whole_pool_bit_exact(name):
    w = W.make(name)
    kc, vc, ks, vs, st = gpu_quantize_fp8(w.k_pool, w.v_pool)
    assert st == 0
    same(kc, ks, *oracle.quantize_fp8(w.k_pool))
    same(vc, vs, *oracle.quantize_fp8(w.v_pool))


def test_quantize_fp8_full_size_used_blocks():
    w = W.make("c5a_64x2048")
    ids = w.used_block_ids
    kc, vc, ks, vs, st = gpu_quantize_fp8(w.k_pool, w.v_pool, ids)
    assert st == 0
    same(kc, ks, *oracle.quantize_fp8(w.k_pool, block_ids=ids))
    same(vc, vs, *oracle.quantize_fp8(w.v_pool, block_ids=ids))


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_fp8_ties_saturation_and_special_tiles(d):
    x = np.zeros((8, 2, 16, d), np.float16)
    flat = x.reshape(8, 2, -1)
    # scale 1 (amax 448): every midpoint between neighbouring E4M3 values
    # that fp16 holds exactly is a tie the rounding must send to even
    mags = sorted({oracle.e4m3_to_double(c) for c in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(mags, mags[1:])]
    vals = [v for v in mids if float(np.float16(v)) == v][: flat.shape[2] - 1]
    flat[0, 0, 0] = 448.0
    flat[0, 0, 1:1 + len(vals)] = vals
    flat[0, 1, 0] = -448.0
    flat[0, 1, 1:1 + len(vals)] = [-v for v in vals]
    flat[1, 0, ::3] = np.nan                            # NaN ignored in the max, code 0
    flat[1, 0, 1] = 3.0
    flat[1, 1, 5] = np.inf                              # scale inf, codes 0
    flat[2, 0, :] = 65504.0                             # fp16 max
    flat[2, 1, :] = np.float16(6e-8)                    # fp16 subnormals only
    flat[3, 0, 1::2] = 1e-3                             # E4M3 subnormal quotients
    flat[3, 0, 0] = 300.0
    flat[4] = np.random.default_rng(d).standard_normal(flat[4].shape) * 100
    kc, vc, ks, vs, st = gpu_quantize_fp8(x, x[::-1].copy())
    assert st == 0
    same(kc, ks, *oracle.quantize_fp8(x))
    same(vc, vs, *oracle.quantize_fp8(x[::-1].copy()))
    assert ks[0, 0] == 1.0 and kc[0, 0, 0, 0] == 0x7E


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (32, 8, 128), (14, 2, 64), (16, 1, 128)])
def test_fp8_decode_with_nan_bytes_in_padding(hq, hkv, d):
    lens = [1, 15, 16, 17, 0, 33, 255, 256, 257]
    w = W.random_case(800 + hq + d, num_seqs=len(lens), num_heads=hq, num_kv_heads=hkv,
                      head_dim=d, context_lens=lens)
    kc, ks = oracle.quantize_fp8(w.k_pool, block_ids=w.used_block_ids)
    vc, vs = oracle.quantize_fp8(w.v_pool, block_ids=w.used_block_ids)
    # bytes past each context end are NaN codes (0x7F / 0xFF): never used
    for s, c in enumerate(lens):
        if c % 16:
            blk = w.block_tables[s, (c - 1) // 16]
            kc[blk, :, c % 16:, ::2] = 0x7F
            vc[blk, :, c % 16:, 1::2] = 0xFF
    codes = (kc, vc, ks, vs)
    got, st = gpu_decode(w, "fp8", codes)
    ref, flags = oracle_decode(w, "fp8", codes)
    assert st == 0 and not flags.any()
    assert_close(got, ref, f"fp8 {hq}/{hkv}/{d}")
    assert np.all(got[4] == 0)

"""Quantization quality measured through the CUDA path.

The same figures as the CPU test beside this one (PagedKV-Fusion README,
Results, "Quantization quality vs FP32": RMSE and max-abs error of the
INT8-KV attention output against full precision, and the output's standard
deviation), but with the codes and scales from pkv_quantize_blocks /
pkv_quantize_blocks_fp8 and the outputs from pkv_paged_decode_int8 /
pkv_paged_decode_fp8 on the GPU, so that the kernels' own rounding is part of
the figure.  The reference is the fp64 oracle on the same fp16 data.

The figures are reported (printed, one line per workload and KV kind), not
gated against the README.  What is asserted is that the kernels add almost
nothing to the quantization error: the GPU path's RMSE is within 2 % of the
oracle's quantized path on the same codes.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import dev, ensure_built

pytestmark = pytest.mark.gpu

PROBES = {
    # the README's Gaussian row: ctx 48 reproduces its output std 0.233
    "gaussian_ctx48": lambda: W.random_case(48, num_seqs=16, num_heads=8, num_kv_heads=8,
                                            head_dim=128, context_lens=[48] * 16),
    "c2_8x512": lambda: W.make("c2_8x512"),
    "c3_32x1024_heavy": lambda: W.make("c3_32x1024_heavy"),
}


def _gpu_quantized_decode(w, fp8):
    n, hq, d = w.query.shape
    kf, vf = dev(w.k_pool), dev(w.v_pool)
    cdt = torch.uint8 if fp8 else torch.int8
    kc = torch.zeros(w.k_pool.shape, dtype=cdt, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros(w.k_pool.shape[:2], dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    ids = dev(w.used_block_ids)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    quant = pkv.pkv_quantize_blocks_fp8 if fp8 else pkv.pkv_quantize_blocks
    quant(kf, vf, kc, vc, ks, vs, ids, status)
    out = torch.empty((n, hq, d), dtype=torch.float32, device="cuda")
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, w.max_context_len)
    decode = pkv.pkv_paged_decode_fp8 if fp8 else pkv.pkv_paged_decode_int8
    decode(out, dev(w.query), kc, vc, ks, vs, dev(w.block_tables), dev(w.context_lens),
           w.max_context_len, w.softmax_scale, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return (out.cpu().numpy().astype(np.float64),
            tuple(t.cpu().numpy() for t in (kc, vc, ks, vs)))


@pytest.mark.parametrize("name", list(PROBES))
@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_quality_through_the_kernels(name, kind):
    ensure_built()
    w = PROBES[name]()
    fp8 = kind == "fp8"
    full = oracle.decode_fp16(w.query, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                              num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale)
    got, (kc, vc, ks, vs) = _gpu_quantized_decode(w, fp8)
    odec = oracle.decode_fp8 if fp8 else oracle.decode_int8
    oq = odec(w.query, kc, vc, ks, vs, w.block_tables, w.context_lens,
              num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale)
    err, oerr = got - full, oq - full
    rmse, mx = float(np.sqrt((err ** 2).mean())), float(np.abs(err).max())
    ormse, omx = float(np.sqrt((oerr ** 2).mean())), float(np.abs(oerr).max())
    print(f"\nquality {name} {kind}: kernel RMSE {rmse:.5f} max-abs {mx:.4f} | "
          f"oracle RMSE {ormse:.5f} max-abs {omx:.4f} | fp64 output std {full.std():.3f}")
    assert abs(rmse - ormse) <= 0.02 * ormse

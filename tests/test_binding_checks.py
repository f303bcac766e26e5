"""The Python binding checks its tensors before anything reaches the C ABI:
pools and workspaces must be CUDA tensors, per-step inputs CUDA or pinned host
tensors.  Runs without a GPU: plain CPU tensors are rejected with ValueError,
for the direct calls and the prepared ones alike, before the library is
called.
"""
import pytest
import torch

import paged_kv_cache_234_gb300 as pkv


def _inputs(code_dtype=torch.int8):
    n, hq, hkv, d, nb = 2, 8, 2, 64, 4
    return dict(
        out=torch.zeros(n, hq, d, dtype=torch.float32),
        query=torch.zeros(n, hq, d, dtype=torch.float16),
        k=torch.zeros(nb, hkv, 16, d, dtype=code_dtype),
        v=torch.zeros(nb, hkv, 16, d, dtype=code_dtype),
        ks=torch.zeros(nb, hkv, dtype=torch.float32),
        vs=torch.zeros(nb, hkv, dtype=torch.float32),
        bt=torch.zeros(n, 2, dtype=torch.int32),
        cl=torch.ones(n, dtype=torch.int32),
        ws=torch.zeros(1024, dtype=torch.uint8),
    )


CALLS = [
    ("decode_int8", lambda a: pkv.pkv_paged_decode_int8(
        a["out"], a["query"], a["k"], a["v"], a["ks"], a["vs"], a["bt"], a["cl"], 32, 0.125,
        a["ws"])),
    ("prepare_int8", lambda a: pkv.prepare_paged_decode_int8(
        a["out"], a["query"], a["k"], a["v"], a["ks"], a["vs"], a["bt"], a["cl"], 32, 0.125,
        a["ws"])),
    ("decode_fp16", lambda a: pkv.pkv_paged_decode_fp16(
        a["out"], a["query"], a["k"].half(), a["v"].half(), a["bt"], a["cl"], 32, 0.125,
        a["ws"])),
    ("decode_fp8", lambda a: pkv.pkv_paged_decode_fp8(
        a["out"], a["query"], a["k"].view(torch.uint8), a["v"].view(torch.uint8), a["ks"],
        a["vs"], a["bt"], a["cl"], 32, 0.125, a["ws"])),
    ("quantize", lambda a: pkv.pkv_quantize_blocks(
        a["k"].half(), a["v"].half(), a["k"], a["v"], a["ks"], a["vs"])),
]


@pytest.mark.parametrize("name,call", CALLS, ids=[c[0] for c in CALLS])
def test_cpu_tensors_are_rejected(name, call):
    with pytest.raises(ValueError, match="CUDA tensor"):
        call(_inputs())


"""The INT8 decode entry point that allocates nothing.

pkv_paged_decode_int8_static_workspace serves callers that cannot allocate
device memory themselves (their memory belongs to another allocator, or they
cannot accept the device synchronisation an allocation may cause): its
scratch is a fixed array inside the library.  Here it must give the same
outputs as pkv_paged_decode_int8 with a caller-provided workspace, bit for
bit (the same kernels with the same worker count run on the same inputs), on
two calls in a row (the second call reuses whatever the first left in the
shared array), match the oracle within the decode tolerance, and refuse a
call whose scratch would not fit.

This file is collected after every other test file, and its tests pass both
in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import assert_close, dev, ensure_built, oracle_codes, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("launch", ["auto", "persistent"])
def test_matches_the_workspace_entry_point_on_two_calls_in_a_row(launch):
    # "persistent": a worker cap selects the persistent workers + reduce,
    # whose split-context records live in the scratch array; "auto": this
    # batch's own choice (it fits one item per thread-block cluster, which
    # merges in shared memory and uses no scratch)
    ensure_built()
    if launch == "persistent":
        pkv.pkv_set_decode_workers(4096)
    try:
        _two_calls_in_a_row()
    finally:
        pkv.pkv_set_decode_workers(0)


def _two_calls_in_a_row():
    w = W.random_case(91, num_seqs=16, num_heads=32, num_kv_heads=8, head_dim=128, max_ctx=1500)
    codes = oracle_codes(w)
    kc, vc, ks, vs = (dev(x) for x in codes)
    n, hq, d = w.query.shape
    q, bt, cl = dev(w.query), dev(w.block_tables), dev(w.context_lens)
    mcl = w.max_context_len
    assert pkv.pkv_decode_workspace_size(n, hq, w.num_kv_heads, d, mcl) <= \
        pkv.PKV_STATIC_WORKSPACE_BYTES

    ref = torch.empty((n, hq, d), dtype=torch.float32, device="cuda")
    ws = pkv.decode_workspace(n, hq, w.num_kv_heads, d, mcl)
    pkv.pkv_paged_decode_int8(ref, q, kc, vc, ks, vs, bt, cl, mcl, w.softmax_scale, ws)
    torch.cuda.synchronize()
    ref_np = ref.cpu().numpy()
    want, _ = oracle_decode(w, "int8", codes)

    for _ in range(2):
        out = torch.full((n, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkv.pkv_paged_decode_int8_static_workspace(out, q, kc, vc, ks, vs, bt, cl, mcl,
                                                   w.softmax_scale, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref_np.view(np.uint32))
        assert_close(got.astype(np.float64), want, "static workspace")


def test_refuses_a_call_whose_scratch_does_not_fit():
    ensure_built()
    # 8 query heads per kv head, head_dim 128 and 4096 pages in flight need
    # 4096 workers x 2 x 8 x 132 x 4 bytes: more than the fixed array
    n, hq, hkv, d, mcl = 1, 64, 8, 128, 8192
    assert pkv.pkv_decode_workspace_size(n, hq, hkv, d, mcl) > pkv.PKV_STATIC_WORKSPACE_BYTES
    q = torch.zeros((n, hq, d), dtype=torch.float16, device="cuda")
    kc = torch.zeros((1, hkv, 16, d), dtype=torch.int8, device="cuda")
    ks = torch.ones((1, hkv), dtype=torch.float32, device="cuda")
    bt = torch.zeros((n, mcl // 16), dtype=torch.int32, device="cuda")
    cl = torch.full((n,), mcl, dtype=torch.int32, device="cuda")
    out = torch.zeros((n, hq, d), dtype=torch.float32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_decode_int8_static_workspace(out, q, kc, kc, ks, ks, bt, cl, mcl, 0.1)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 0)  # nothing was launched

"""The decode kernel's bounded-wait failure path.

Every wait of the decode kernel for a stage of copies is bounded; when one
runs out the kernel sets PKV_DEV_TIMEOUT in the caller's status word, lets
every copy the worker issued land (so that none still writes into shared
memory), and the worker returns: the call ends and the context stays usable
("PagedAttention & KV-Cache Memory Management", section 2.4 Failure Modes
& Recovery Strategies, and 3.3.4 Failure Recovery Path).

A copy that never lands cannot be made safely, so the debug build of the
library (PKV_DEBUG) takes the limit of the stage waits from a setting: at 0
a wait gives up at once, as if its limit had run out, while its copies are
still in flight.  The copies themselves do land, and the drain after the
timeout waits for them with its normal limit.  After the limit is restored,
the same call on the debug build and on the release build matches the
oracle again.  Both launches are covered: this batch's own one (one item per
thread-block cluster, where a warp that gave up still joins its cluster's
barrier and marks its records bad) and the persistent workers + reduce
(selected by a worker cap).
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import assert_close, dev, ensure_built, gpu_decode, oracle_codes, oracle_decode

pytestmark = pytest.mark.gpu


def _debug_int8(L, w, codes):
    n, hq, d = w.query.shape
    mcl = w.max_context_len
    q, bt, cl = dev(w.query), dev(w.block_tables), dev(w.context_lens)
    kc, vc, ks, vs = (dev(a) for a in codes)
    out = torch.full((n, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = L.pkv_decode_workspace_size(n, hq, w.num_kv_heads, d, mcl)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.pkv_paged_decode_int8(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                 ks.data_ptr(), vs.data_ptr(), w.num_blocks, bt.data_ptr(),
                                 w.max_blocks_per_seq, cl.data_ptr(), mcl, n, hq,
                                 w.num_kv_heads, d, 16, w.softmax_scale, ws.data_ptr(),
                                 ws.numel(), status.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()  # raises if the context were lost
    return rc, out.cpu().numpy().astype(np.float64), int(status.item())


@pytest.mark.parametrize("launch", ["auto", "persistent"])
def test_a_stage_wait_that_runs_out_sets_the_status_and_the_call_returns(launch):
    ensure_built()
    L = pkv.debug_lib()
    cap = 4096 if launch == "persistent" else 0
    w = W.random_case(93, num_seqs=16, num_heads=32, num_kv_heads=8, head_dim=128,
                      max_ctx=1500)
    codes = oracle_codes(w)
    ref, _ = oracle_decode(w, "int8", codes)
    try:
        assert L.pkv_set_decode_workers(cap) == 0
        assert L.pkv_debug_set_stage_wait_ns(0) == 0
        rc, _, st = _debug_int8(L, w, codes)
        assert rc == 0
        assert st & pkv.PKV_DEV_TIMEOUT, f"status {st:#x}: no stage wait ran out"
    finally:
        assert L.pkv_debug_set_stage_wait_ns(-1) == 0
    try:
        assert L.pkv_debug_flags(1) == 0  # the timed-out run stayed inside its buffers
        # the same call with the default limit, on the debug and the release build
        rc, got, st = _debug_int8(L, w, codes)
        assert rc == 0 and st == 0
        assert_close(got, ref, f"debug build after the timeout ({launch})")
    finally:
        L.pkv_set_decode_workers(0)
    pkv.pkv_set_decode_workers(cap)
    try:
        got, st = gpu_decode(w, "int8", codes)
    finally:
        pkv.pkv_set_decode_workers(0)
    assert st == 0
    assert_close(got, ref, f"release build after the timeout ({launch})")

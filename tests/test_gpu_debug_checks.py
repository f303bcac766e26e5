"""The decode and eviction kernels built with their debug checks (PKV_DEBUG).

Decode: every shared-memory address it forms stays inside the CTA's dynamic
shared memory and is aligned for its access, and every table index is in
range, on a spread of shapes -- head dims 64 and 128, group sizes 1 to 16,
ragged and edge lengths, one item split over many workers, 3000 sequences --
with the outputs still matching the oracle.  Eviction: each CTA's staged
slice fits its shared memory, the cluster fits the peer arrays and every
16-byte copy lands inside the slice, from 1 block to the largest pool one
launch takes, with the oracle's choice.  A failed check redirects or skips
the access and sets a flag, so these runs cannot fault.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_234_gb300 as pkv
import pkv_workloads as W
from gpu_common import assert_close, dev, oracle_codes, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    lib = pkv.debug_lib()
    lib.pkv_debug_flags(1)
    return lib


def debug_decode(L, w, variant, codes, workers=0):
    n, hq, d = w.query.shape
    mcl = w.max_context_len
    q, bt, cl = dev(w.query), dev(w.block_tables), dev(w.context_lens)
    out = torch.full((n, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = L.pkv_decode_workspace_size(n, hq, w.num_kv_heads, d, mcl)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    common = (w.num_blocks, bt.data_ptr(), w.max_blocks_per_seq, cl.data_ptr(), mcl, n, hq,
              w.num_kv_heads, d, 16, w.softmax_scale, ws.data_ptr(), ws.numel(),
              status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert L.pkv_set_decode_workers(workers) == 0
    try:
        if variant == "fp16":
            kf, vf = dev(w.k_pool), dev(w.v_pool)
            st = L.pkv_paged_decode_fp16(out.data_ptr(), q.data_ptr(), kf.data_ptr(),
                                         vf.data_ptr(), *common)
        else:
            kc, vc, ks, vs = (dev(a) for a in codes)
            fn = L.pkv_paged_decode_fp8 if variant == "fp8" else L.pkv_paged_decode_int8
            st = fn(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), ks.data_ptr(),
                    vs.data_ptr(), *common)
        torch.cuda.synchronize()
    finally:
        L.pkv_set_decode_workers(0)
    assert st == 0
    return out.cpu().numpy().astype(np.float64), int(status.item())


CASES = [
    ("c1", dict(seed=201, num_seqs=2, num_heads=8, num_kv_heads=2, head_dim=64,
                context_lens=[37, 16]), 0),
    ("edge-128", dict(seed=202, num_seqs=9, num_heads=32, num_kv_heads=8, head_dim=128,
                      context_lens=[1, 15, 16, 17, 0, 33, 255, 256, 257]), 0),
    ("group-16", dict(seed=203, num_seqs=5, num_heads=16, num_kv_heads=1, head_dim=128,
                      context_lens=[300, 1, 64, 129, 511]), 0),
    ("group-7-d64", dict(seed=204, num_seqs=6, num_heads=14, num_kv_heads=2, head_dim=64,
                         context_lens=[512, 7, 100, 33, 0, 250]), 0),
    ("group-1", dict(seed=205, num_seqs=8, num_heads=8, num_kv_heads=8, head_dim=128,
                     context_lens=[512] * 8), 0),
    ("long-item", dict(seed=206, num_seqs=16, num_heads=8, num_kv_heads=1, head_dim=128,
                       context_lens=[16384] + [16] * 15), 0),
    ("split-13", dict(seed=207, num_seqs=6, num_heads=8, num_kv_heads=2, head_dim=128,
                      context_lens=[300, 1, 77, 512, 16, 250]), 13),
    ("many-seqs", dict(seed=208, num_seqs=3000, num_heads=8, num_kv_heads=2, head_dim=64,
                       max_ctx=40), 0),
]


@pytest.mark.parametrize("variant", ["fp16", "int8", "fp8"])
@pytest.mark.parametrize("name,kw,workers", CASES, ids=[c[0] for c in CASES])
def test_debug_build_finds_no_out_of_range_access(L, name, kw, workers, variant):
    kw = dict(kw)
    w = W.random_case(kw.pop("seed"), **kw)
    codes = None if variant == "fp16" else oracle_codes(w, variant == "fp8")
    got, st = debug_decode(L, w, variant, codes, workers)
    flags = L.pkv_debug_flags(1)
    assert flags == 0, f"{name}/{variant}: debug check bits {flags:#x}"
    ref, oflags = oracle_decode(w, variant, codes)
    assert st == 0 and not oflags.any()
    assert_close(got, ref, f"{name}/{variant} (debug build)")


@pytest.mark.parametrize("num_blocks", [1, 100, 1024, 16384, 65536, 200_000, 16 * 49152])
def test_debug_build_eviction_stays_in_its_buffers(L, num_blocks):
    import oracle
    if num_blocks == 16 * 49152:
        # the largest pool one launch takes: 16-CTA clusters where the
        # device schedules them, else 8
        probe_ref = torch.zeros(num_blocks, dtype=torch.int32, device="cuda")
        probe_last = torch.zeros(num_blocks, dtype=torch.int64, device="cuda")
        cnt0 = torch.zeros(1, dtype=torch.int32, device="cuda")
        if L.pkv_evict_select(probe_ref.data_ptr(), probe_last.data_ptr(), num_blocks, 0, 0.7,
                              0.3, 0, None, None, cnt0.data_ptr(),
                              torch.cuda.current_stream().cuda_stream) == pkv.PKV_ERR_UNSUPPORTED:
            num_blocks = 8 * 49152
        torch.cuda.synchronize()
    k = pkv.evict_count(num_blocks) or 1
    st = W.eviction_state(num_blocks, 31)
    ref, last = dev(st.refcnt), dev(st.last_used)
    ids = torch.empty(max(k, 1), dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    sc = torch.empty(num_blocks, dtype=torch.float32, device="cuda")
    L.pkv_debug_evict_flags(1)
    rc = L.pkv_evict_select(ref.data_ptr(), last.data_ptr(), num_blocks, st.current_tick,
                            pkv.EVICT_ALPHA, pkv.EVICT_BETA, k, sc.data_ptr(), ids.data_ptr(),
                            cnt.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    flags = L.pkv_debug_evict_flags(1)
    assert flags == 0, f"eviction debug check bits {flags:#x}"
    want_ids, want_sc = oracle.evict_select(st.refcnt, st.last_used, st.current_tick, k)
    assert int(cnt.item()) == want_ids.size
    assert np.array_equal(ids.cpu().numpy()[: want_ids.size], want_ids)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), want_sc.view(np.uint32))

"""Benchmark of the paged decode hot path on GB300.

One step = one decode step of a 64-sequence batch with an INT8 KV cache:
  1. pkv_quantize_blocks on the batch's tail blocks (the blocks that hold each
     sequence's newest tokens, K and V),
  2. pkv_paged_decode_int8 over the whole batch (block-table gather, INT8
     dequant, QK^T, online softmax, PV, split-context reduce, GQA).
Workload: 64 seqs x ctx 2048, 32 q / 8 kv heads, head_dim 128, block 16, a
65536-block pool with seeded random placement (synthetic N(0,1) data).

Metric: KV GB/s = algorithmic bytes per step / step time (the bytes of K, V
and scales a step must read plus what the quantizer reads and writes), also
sequence-steps/s and p50 us/step.  Steps run back to back, as a stream runs
them, between one pair of CUDA events, issued as prepared calls (arguments
marshalled once, so that the host stays ahead of the GPU); the inputs are
larger than L2, so no flush separates them.  The same calls with the L2 flushed before each one and
an event pair around each are reported as a labelled extra
("flushed_per_call" and the variants' flushed_* keys).  The fp16-KV and
FP8-KV decodes of the same batch, the
token append that precedes a decode step (fp16, and INT8 with the fused tail
re-quantize), eviction scoring + choice of 15 % of the blocks at pools of
1024, 16384 and 65536 blocks, the copy-on-write block copies (64 and 4096
blocks of K and V) and the host block manager's throughput are timed
alongside and reported under "variants".

--impl reference times the CPU oracle (plain C, fp64 attention) on a bounded
sample of the same workload, as the reference arm.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import pkv_workloads as W  # noqa: E402

CONFIG = "c5a_64x2048"
METRIC = "paged decode attn: KV GB/s (% of HBM peak), seq-steps/s, p50 µs/step"
UNIT = "GB/s"
FLUSH_BYTES = 256 << 20  # > 129 MB L2: written, then another one read, between steps
# DRAM bytes per launch of the INT8 decode (decode + reduce kernels) on this
# workload from the ncu capture summarised in profiles/, with the hash of the
# kernel source it was taken on; the figure is dropped when the source changes.
TRAFFIC = {"decode_int8": (270069760 + 736256 + 5003008, "4d213eb79d7e8572")}  # decode + reduce kernels (read + write)


def _src_hash():
    """Hash of the decode kernel's source code, comments and blank lines left
    out (a comment edit does not change the counters)."""
    p = os.path.join(ROOT, "paged_kv_cache_234_gb300", "csrc", "pkv_decode.cu")
    code = []
    for line in open(p):
        line = line.split("//", 1)[0].rstrip()
        if line:
            code.append(line)
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def decode_bytes(ctx, num_kv_heads, head_dim, elem_bytes, with_scales):
    """Algorithmic bytes one decode call must read: K and V of every cached
    token of every kv head, plus one K and one V scale per (block, kv head)."""
    ctx = np.asarray(ctx, dtype=np.int64)
    b = int(ctx.sum()) * num_kv_heads * head_dim * 2 * elem_bytes
    if with_scales:
        b += int(((ctx + 15) // 16).sum()) * num_kv_heads * 2 * 4
    return b


def quantize_bytes(num_tiles, head_dim):
    """fp16 read + int8 written per value, one fp32 scale per tile (K and V)."""
    return num_tiles * 2 * (16 * head_dim * 3 + 4)


def append_bytes(num_tiles, head_dim, int8):
    """Per (sequence, kv head), K and V: the new fp16 row read and written;
    INT8 adds the 15 other fp16 rows read, 16 rows of codes and a scale written."""
    row = head_dim * 2
    if not int8:
        return num_tiles * 2 * 2 * row
    return num_tiles * 2 * (16 * row + row + 16 * head_dim + 4)


def evict_bytes(num_blocks, k):
    """refcnt (4 B) and last_used (8 B) read, the fp32 score written per block,
    k chosen ids and the count written."""
    return num_blocks * (4 + 8 + 4) + 4 * k + 4


EVICT_SIZES = (1024, 16384, 65536)  # the pages' pool sizes, then this workload's pool
COPY_PAIRS = (64, 4096)  # copy-on-write batches: one decode step's tails, a large fork


def block_manager_rate(num_blocks=65536, batch=128, seconds=1.0, model=False):
    """Blocks per second through allocate + copy-on-write + free cycles of
    `batch`-block requests (each block also forked once, so every
    copy-on-write copies) on the native manager, or on the oracle's model."""
    ids_per_cycle = 0
    if model:
        from oracle.block_manager import BlockManagerModel
        bm = BlockManagerModel(num_blocks)
        alloc = lambda: bm.allocate([0] * batch)
        fork, cow, free = bm.fork, bm.cow_batch, bm.free
    else:
        import paged_kv_cache_234_gb300 as pkv
        bm = pkv.BlockManager(num_blocks)
        alloc = lambda: bm.allocate(batch)
        fork, cow, free = bm.fork, (lambda ids: bm.cow(ids)), bm.free
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        a = alloc()
        fork(a)
        new, _ = cow(a)
        free(a)
        free(new)
        ids_per_cycle += batch
    return ids_per_cycle / (time.perf_counter() - t0)


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # the raw samples: PKV_CLOCKS_DIR if set, else the system temp folder
        folder = os.environ.get("PKV_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(folder, f"pkv_clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _subpool(w, seqs):
    """The sampled sequences' blocks gathered into a compact pool, with their
    tables renumbered (attention does not depend on physical placement)."""
    tab = w.block_tables[seqs]
    lens = w.context_lens[seqs]
    ids = np.unique(tab[tab >= 0]).astype(np.int32)
    local = np.full(w.num_blocks, -1, np.int32)
    local[ids] = np.arange(ids.size, dtype=np.int32)
    ltab = np.where(tab >= 0, local[np.maximum(tab, 0)], -1).astype(np.int32)
    tails = np.array([ltab[i, (c - 1) // 16] for i, c in enumerate(lens) if c > 0], np.int32)
    return (np.ascontiguousarray(w.k_pool[ids]), np.ascontiguousarray(w.v_pool[ids]), ltab,
            lens, tails)


def workload_desc(w, n_tails):
    """The benchmark workload as named in both arms' "config"."""
    n, hq, d = w.query.shape
    return (f"{CONFIG}: {n} seqs x ctx {w.max_context_len}, {hq} q / {w.num_kv_heads} kv heads, "
            f"head_dim {d}, block 16, pool {w.num_blocks} blocks; step = INT8 quantize of "
            f"{n_tails} tail blocks + INT8 decode")


def run_reference(args, ws, rank):
    """CPU oracle on a bounded sample of the workload (rank 0 only): each step
    quantizes the tail blocks of 8 of the 64 sequences and decodes those 8."""
    if rank != 0:
        return
    import oracle
    w = W.make(CONFIG)
    sample = 8
    seqs = np.arange(0, w.num_seqs, w.num_seqs // sample)[:sample]
    kp, vp, tab, lens, tails = _subpool(w, seqs)
    kc, ks = oracle.quantize(kp)   # the cache contents, not timed
    vc, vs = oracle.quantize(vp)
    threads = oracle.max_threads()
    step_b = (decode_bytes(lens, w.num_kv_heads, w.head_dim, 1, True)
              + quantize_bytes(len(tails) * w.num_kv_heads, w.head_dim))
    t_total = 0.0
    for it in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.quantize(kp, block_ids=tails, code_pool=kc, scales=ks, inplace=True)
        oracle.quantize(vp, block_ids=tails, code_pool=vc, scales=vs, inplace=True)
        oracle.decode_int8(w.query[seqs], kc, vc, ks, vs, tab, lens,
                           num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                           num_threads=threads)
        if it >= args.warmup:
            t_total += time.perf_counter() - t0
    value = step_b * args.steps / t_total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t_total / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w, len(w.tail_block_ids())),
                   "sample": f"CPU oracle on {sample} of {w.num_seqs} sequences per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{sample} of {w.num_seqs} sequences per step: INT8 "
                                   "quantize of their tail blocks + fp64 INT8 decode"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w, seconds=10.0):
    """Oracle INT8 decode on a bounded sample, timed on this host's cores:
    all threads (the reported value) and one thread (reported beside it)."""
    import oracle
    threads = oracle.max_threads()
    seqs = np.arange(4)
    kp, vp, tab, lens, _ = _subpool(w, seqs)
    kc, ks = oracle.quantize(kp)
    vc, vs = oracle.quantize(vp)
    nb = decode_bytes(lens, w.num_kv_heads, w.head_dim, 1, True)

    def rate(nthreads, secs):
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.decode_int8(w.query[seqs], kc, vc, ks, vs, tab, lens,
                               num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                               num_threads=nthreads)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= secs:
                return nb * reps / dt / 1e9, reps, dt

    value, reps, dt = rate(threads, seconds)
    single, reps1, dt1 = rate(1, seconds / 4)
    return {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"fp64 INT8 decode of 4 of {w.num_seqs} sequences, repeated {reps} times "
                      f"({dt:.1f} s)",
            "single_thread": {"value": single, "unit": UNIT,
                              "sample": f"the same, 1 thread, {reps1} times ({dt1:.1f} s)"}}


def run_profile(args):
    """Decode calls of one variant on the benchmark batch placed in a smaller
    pool (same bytes per call), for ncu captures that must stay small."""
    import torch
    import paged_kv_cache_234_gb300 as pkv
    from paged_kv_cache_234_gb300 import build as pkv_build
    pkv_build.build()
    if args.profile == "int8-small":
        w = W.make("c2_8x512")
    elif args.profile == "int8-d64":
        w = W.build("qwen2_512x2048", num_heads=14, num_kv_heads=2, head_dim=64,
                    num_blocks=65536 + 64, context_lens=[2048] * 512, seed=1007)
    elif args.profile == "int8-long":
        w = W.build("long_1x131072", num_heads=32, num_kv_heads=8, head_dim=128,
                    num_blocks=8192 + 64, context_lens=[131072], seed=1006)
    else:
        w = W.build(CONFIG + "_pool16k", num_heads=128 if args.profile == "int8-g16" else 32,
                    num_kv_heads=8, head_dim=128, num_blocks=16384, context_lens=[2048] * 64,
                    seed=1005)
    n, hq, d = w.query.shape
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kf, vf = dev(w.k_pool), dev(w.v_pool)
    q, bt, cl = dev(w.query), dev(w.block_tables), dev(w.context_lens)
    out = torch.empty((n, hq, d), dtype=torch.float32, device="cuda")
    ws_t = pkv.decode_workspace(n, hq, w.num_kv_heads, d, w.max_context_len)
    if args.profile == "quantize":
        kc = torch.zeros(w.k_pool.shape, dtype=torch.int8, device="cuda")
        vc = torch.zeros_like(kc)
        ks = torch.zeros(w.k_pool.shape[:2], dtype=torch.float32, device="cuda")
        vs = torch.zeros_like(ks)
        tails = dev(w.tail_block_ids())
        call = lambda: pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, tails)
    elif args.profile in ("int8", "fp8", "int8-small", "int8-g16", "int8-long", "int8-d64"):
        kc = torch.zeros(w.k_pool.shape, dtype=torch.int8, device="cuda")
        vc = torch.zeros_like(kc)
        ks = torch.zeros(w.k_pool.shape[:2], dtype=torch.float32, device="cuda")
        vs = torch.zeros_like(ks)
        if args.profile == "fp8":
            kc = kc.view(torch.uint8)
            vc = vc.view(torch.uint8)
            pkv.pkv_quantize_blocks_fp8(kf, vf, kc, vc, ks, vs, dev(w.used_block_ids))
            dec = pkv.pkv_paged_decode_fp8
        else:
            pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, dev(w.used_block_ids))
            dec = pkv.pkv_paged_decode_int8
        del kf, vf
        call = lambda: dec(out, q, kc, vc, ks, vs, bt, cl, w.max_context_len, w.softmax_scale,
                           ws_t)
    else:
        call = lambda: pkv.pkv_paged_decode_fp16(out, q, kf, vf, bt, cl, w.max_context_len,
                                                 w.softmax_scale, ws_t)
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    print(f"profile run: {args.profile} x{args.warmup + args.steps}", flush=True)


def run_profile_small(args):
    """Append or eviction calls alone, for ncu: the append of the benchmark
    batch's newest tokens (64 sequences, pool of 16384 blocks), or eviction
    scoring of a 65536-block pool."""
    import torch
    import paged_kv_cache_234_gb300 as pkv
    from paged_kv_cache_234_gb300 import build as pkv_build
    pkv_build.build()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if args.profile == "evict":
        st = W.eviction_state(EVICT_SIZES[-1], 7)
        ref, last = dev(st.refcnt), dev(st.last_used)
        k = pkv.evict_count(ref.numel())
        ids = torch.empty(k, dtype=torch.int32, device="cuda")
        cnt = torch.empty(1, dtype=torch.int32, device="cuda")
        sc = torch.empty(ref.numel(), dtype=torch.float32, device="cuda")
        call = lambda: pkv.pkv_evict_select(ref, last, st.current_tick, k, ids, cnt, sc)
    else:
        w = W.build(CONFIG + "_pool16k", num_heads=32, num_kv_heads=8, head_dim=128,
                    num_blocks=16384, context_lens=[2048] * 64, seed=1005)
        kn, vn, pos = W.append_tokens(w, 99)
        kf, vf = dev(w.k_pool), dev(w.v_pool)
        kc = torch.zeros(w.k_pool.shape, dtype=torch.int8, device="cuda")
        vc = torch.zeros_like(kc)
        ks = torch.zeros(w.k_pool.shape[:2], dtype=torch.float32, device="cuda")
        vs = torch.zeros_like(ks)
        a = (dev(kn), dev(vn), dev(w.block_tables), dev(pos))
        call = lambda: pkv.pkv_append_int8(kf, vf, kc, vc, ks, vs, *a)
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    print(f"profile run: {args.profile} x{args.warmup + args.steps}", flush=True)


def run_report(args):
    """Per configuration and variant: p50 / p90 us per decode call over 200
    timed calls after 20 warm-ups (--report-calls, --report-warmup), L2
    flushed before each call; KV GB/s of the logical bytes (unique bytes too
    where sequences share blocks) and sequence-steps/s.  Beside them, as
    labelled extras: the GPU time of a call with the L2 flushed before it but
    without the event pair and host overhead (flush + call pairs replayed
    from a CUDA graph, minus the flushes alone), and the mean of the same
    number of calls back to back with no flush (warm L2 for the batches that
    fit in it), issued as prepared calls (arguments marshalled once) so that
    the host keeps ahead of the GPU.  One JSON line per (configuration,
    variant), in the order the calls run."""
    import torch
    import paged_kv_cache_234_gb300 as pkv
    from paged_kv_cache_234_gb300 import build as pkv_build
    pkv_build.build()
    peak, _ = _peaks()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    fw = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    fr = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    l2_bytes = torch.cuda.get_device_properties(0).L2_cache_size

    def graph_cold_call(fn, reps=20, replays=7):
        # labelled extra: GPU time of one call with the L2 flushed before it,
        # free of event-pair and host overhead: reps x (flush, call) replayed
        # from one CUDA graph, minus the same graph without the calls
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
        torch.cuda.synchronize()
        graphs = []
        for with_call in (True, False):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(reps):
                    fw.zero_()
                    fr.view(torch.int32).max()
                    if with_call:
                        fn()
            graphs.append(g)
        med = []
        for g in graphs:
            ts = []
            for i in range(replays + 2):
                g0 = torch.cuda.Event(enable_timing=True)
                g1 = torch.cuda.Event(enable_timing=True)
                g0.record(stream)
                g.replay()
                g1.record(stream)
                g1.synchronize()
                if i >= 2:
                    ts.append(g0.elapsed_time(g1) * 1e-3)
            med.append(statistics.median(ts))
        del graphs
        return (med[0] - med[1]) / reps

    names = [c for c in args.configs.split(",") if c] or list(W.CONFIG_NAMES)
    for name in names:
        w = W.make(name)
        n, hq, d = w.query.shape
        hkv = w.num_kv_heads
        kf, vf = dev(w.k_pool), dev(w.v_pool)
        q, bt, cl = dev(w.query), dev(w.block_tables), dev(w.context_lens)
        used = dev(w.used_block_ids)
        out = torch.empty((n, hq, d), dtype=torch.float32, device="cuda")
        ws_t = pkv.decode_workspace(n, hq, hkv, d, w.max_context_len)
        pools = {}
        for kind, qfn, dt in (("int8", pkv.pkv_quantize_blocks, torch.int8),
                              ("fp8", pkv.pkv_quantize_blocks_fp8, torch.uint8)):
            kc = torch.zeros(w.k_pool.shape, dtype=dt, device="cuda")
            vc = torch.zeros_like(kc)
            ks = torch.zeros(w.k_pool.shape[:2], dtype=torch.float32, device="cuda")
            vs = torch.zeros_like(ks)
            qfn(kf, vf, kc, vc, ks, vs, used)
            pools[kind] = (kc, vc, ks, vs)
        calls = {
            "fp16": lambda: pkv.pkv_paged_decode_fp16(out, q, kf, vf, bt, cl, w.max_context_len,
                                                      w.softmax_scale, ws_t),
            "int8": lambda: pkv.pkv_paged_decode_int8(out, q, *pools["int8"], bt, cl,
                                                      w.max_context_len, w.softmax_scale, ws_t),
            "fp8": lambda: pkv.pkv_paged_decode_fp8(out, q, *pools["fp8"], bt, cl,
                                                    w.max_context_len, w.softmax_scale, ws_t),
        }
        prepared = {
            "fp16": pkv.prepare_paged_decode_fp16(out, q, kf, vf, bt, cl, w.max_context_len,
                                                  w.softmax_scale, ws_t),
            "int8": pkv.prepare_paged_decode_int8(out, q, *pools["int8"], bt, cl,
                                                  w.max_context_len, w.softmax_scale, ws_t),
            "fp8": pkv.prepare_paged_decode_fp8(out, q, *pools["fp8"], bt, cl,
                                                w.max_context_len, w.softmax_scale, ws_t),
        }
        # blocks read once per call when sequences share them (c4: shared prefix)
        uniq_ctx = np.full(w.used_block_ids.size, 16, np.int64)
        cpu = None if args.no_cpu_baseline else cpu_oracle_sample(w, W.CONFIG_NAMES.index(name))
        for variant, fn in calls.items():
            for _ in range(args.report_warmup):
                fn()
            ts = []
            for _ in range(args.report_calls):
                fw.zero_()
                fr.view(torch.int32).max()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e-3)
            eb, sc = (2, False) if variant == "fp16" else (1, True)
            b = decode_bytes(w.context_lens, hkv, d, eb, sc)
            bu = decode_bytes(uniq_ctx, hkv, d, eb, sc)
            t50, t90 = statistics.median(ts), float(np.percentile(ts, 90))
            # labelled extra: the same calls back to back, one pair of events
            # around the run, no flush (warm L2 where the batch fits in it),
            # issued as prepared calls so that the host keeps ahead
            pfn = prepared[variant]
            for _ in range(3):
                pfn()
            torch.cuda.synchronize()
            b0 = torch.cuda.Event(enable_timing=True)
            b1 = torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for _ in range(args.report_calls):
                pfn()
            b1.record(stream)
            b1.synchronize()
            tb = b0.elapsed_time(b1) * 1e-3 / args.report_calls
            tg = graph_cold_call(fn)
            rec = {"config": name, "variant": variant, "p50_us": 1e6 * t50,
                   "p90_us": 1e6 * t90, "mean_us": 1e6 * statistics.mean(ts),
                   "kv_bytes": b, "unique_kv_bytes": bu,
                   "GB/s": b / t50 / 1e9, "frac_of_peak": b / t50 / 1e9 / peak,
                   "seq_steps_per_s": n / t50,
                   "graph_cold_us": 1e6 * tg,
                   "back_to_back_us": 1e6 * tb,
                   "back_to_back_l2": "inputs larger than L2" if bu > l2_bytes
                                      else "warm L2: the batch's KV fits in L2"}
            if variant == "int8" and cpu is not None:
                rec["cpu_oracle"] = {**cpu, "us_scaled": 1e6 * b / (cpu["GB/s"] * 1e9)}
            print(json.dumps(rec), flush=True)
        del kf, vf, pools, prepared
        torch.cuda.empty_cache()


def cpu_oracle_sample(w, seed, sample=8, seconds=0.5):
    """The oracle's INT8 decode on a seeded sample of at most `sample` of the
    batch's sequences, on this host's cores: its KV GB/s (the per-configuration
    CPU baseline; the whole batch's time is its bytes at this rate)."""
    import oracle
    rng = np.random.default_rng(seed)
    k = min(sample, w.num_seqs)
    seqs = np.sort(rng.choice(w.num_seqs, size=k, replace=False))
    kp, vp, tab, lens, _ = _subpool(w, seqs)
    kc, ks = oracle.quantize(kp)
    vc, vs = oracle.quantize(vp)
    nb = decode_bytes(lens, w.num_kv_heads, w.head_dim, 1, True)
    threads = oracle.max_threads()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.decode_int8(w.query[seqs], kc, vc, ks, vs, tab, lens,
                           num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                           num_threads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return {"GB/s": nb * reps / dt / 1e9, "threads": threads,
            "sample": f"{k} of {w.num_seqs} sequences (seeded), {reps} repetitions"}


def evict_cpu_us(num_blocks, reps=20):
    """The oracle's eviction (scores + sort-based choice) on this host."""
    import oracle
    st = W.eviction_state(num_blocks, 7)
    k = (num_blocks * 15) // 100
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.evict_select(st.refcnt, st.last_used, st.current_tick, k)
        ts.append(time.perf_counter() - t0)
    return 1e6 * statistics.median(ts)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--report-configs", action="store_true",
                    help="p50/p90 of every decode variant on every configuration, one JSON "
                         "line each (no benchmark line)")
    ap.add_argument("--report-warmup", type=int, default=20)
    ap.add_argument("--report-calls", type=int, default=200)
    ap.add_argument("--configs", default="",
                    help="with --report-configs: comma-separated configuration names to "
                         "report (default: all)")
    ap.add_argument("--profile", choices=["int8", "fp8", "fp16", "quantize", "append", "evict",
                                          "int8-small", "int8-g16", "int8-long", "int8-d64"],
                    help="profiling run: the same batch over a 16384-block pool (eviction: "
                         "a 65536-block pool; int8-small: the 8 x 512 batch, whose INT8 "
                         "decode takes the one-item-per-cluster launch; int8-g16: the same "
                         "KV with 128 query heads, 16 per kv head; int8-long: one sequence "
                         "of 131072 tokens, the same KV bytes; int8-d64: 512 x 2048 in the "
                         "Qwen2-0.5B attention shape, 14 query / 2 kv heads of 64, the same "
                         "KV bytes), only warm-up + timed "
                         "calls of one kernel, no report line")
    args = ap.parse_args()
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if args.report_configs:
        run_report(args)
        return
    if args.profile in ("append", "evict"):
        run_profile_small(args)
        return
    if args.profile:
        run_profile(args)
        return

    import torch
    import paged_kv_cache_234_gb300 as pkv
    from paged_kv_cache_234_gb300 import build as pkv_build

    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    if rank == 0:
        pkv_build.build()
    if pg:
        pg.barrier()
    pkv.lib()

    w = W.make(CONFIG)
    n, hq, d = w.query.shape
    hkv = w.num_kv_heads
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kf, vf = dev(w.k_pool), dev(w.v_pool)
    q, bt, cl = dev(w.query), dev(w.block_tables), dev(w.context_lens)
    kc = torch.zeros(w.k_pool.shape, dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros(w.k_pool.shape[:2], dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    used = dev(w.used_block_ids)
    tails_np = w.tail_block_ids()
    tails = dev(tails_np)
    mcl = w.max_context_len
    ws_t = pkv.decode_workspace(n, hq, hkv, d, mcl)
    out = torch.empty((n, hq, d), dtype=torch.float32, device="cuda")
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def l2_flush():
        # write a buffer larger than L2, then read another one: no KV stays in
        # L2 and no dirty line is left for the timed kernels to write back
        flush_w.zero_()
        flush_r.view(torch.int32).max()

    # the cache contents: every used block quantized once (not timed)
    pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, used, status)
    kc8 = torch.zeros(w.k_pool.shape, dtype=torch.uint8, device="cuda")
    vc8 = torch.zeros_like(kc8)
    ks8 = torch.zeros_like(ks)
    vs8 = torch.zeros_like(ks)
    pkv.pkv_quantize_blocks_fp8(kf, vf, kc8, vc8, ks8, vs8, used, status)
    torch.cuda.synchronize()

    def step_int8():
        pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, tails, status)

    def decode_int8():
        pkv.pkv_paged_decode_int8(out, q, kc, vc, ks, vs, bt, cl, mcl, w.softmax_scale, ws_t,
                                  status)

    def decode_fp8():
        pkv.pkv_paged_decode_fp8(out, q, kc8, vc8, ks8, vs8, bt, cl, mcl, w.softmax_scale, ws_t,
                                 status)

    def decode_fp16():
        pkv.pkv_paged_decode_fp16(out, q, kf, vf, bt, cl, mcl, w.softmax_scale, ws_t, status)

    # the same calls prepared once (arguments checked and marshalled at set-up),
    # for the back-to-back runs, where the host must stay ahead of the GPU
    p_step = pkv.prepare_quantize_blocks(kf, vf, kc, vc, ks, vs, tails, status)
    p_int8 = pkv.prepare_paged_decode_int8(out, q, kc, vc, ks, vs, bt, cl, mcl,
                                           w.softmax_scale, ws_t, status)
    p_fp8 = pkv.prepare_paged_decode_fp8(out, q, kc8, vc8, ks8, vs8, bt, cl, mcl,
                                         w.softmax_scale, ws_t, status)
    p_fp16 = pkv.prepare_paged_decode_fp16(out, q, kf, vf, bt, cl, mcl, w.softmax_scale, ws_t,
                                           status)

    for _ in range(args.warmup):
        step_int8()
        decode_int8()
        decode_fp16()
        decode_fp8()
    torch.cuda.synchronize()

    # The timed region: K steps back to back, as a stream runs them, between
    # one pair of events.  No L2 flush between steps: the step reads 270 MB of
    # INT8 codes, more than the 129 MB L2, and a back-to-back call reads all
    # of its algorithmic bytes from DRAM (ncu with cache control off).
    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for _ in range(K):
        p_step()
        p_int8()
    t_end.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    if pg:
        t = torch.tensor([total_ms], device="cuda")
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        total_ms = float(t.item())

    # per-step distribution: the same steps back to back again, an event
    # after every block of ten (an event between steps costs ~3 us itself)
    blk = 10
    nblk = max(1, min(K, 500) // blk)
    evp = [torch.cuda.Event(enable_timing=True) for _ in range(nblk + 1)]
    torch.cuda.synchronize()
    evp[0].record(stream)
    for i in range(nblk):
        for _ in range(blk):
            p_step()
            p_int8()
        evp[i + 1].record(stream)
    torch.cuda.synchronize()
    step_ms = [evp[i].elapsed_time(evp[i + 1]) / blk for i in range(nblk)]

    # labelled extra: every call on its own, L2 flushed before it, one pair
    # of events around each call (an event pair alone measures ~2.2 us here,
    # and no launch overlaps the one before)
    def timed(fn, reps):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
        for i in range(reps):
            l2_flush()
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) for e in evs]

    Kd = min(K, 500)
    dec_ms = timed(decode_int8, Kd)
    f16_ms = timed(decode_fp16, Kd)
    f8_ms = timed(decode_fp8, Kd)
    q_ms = timed(step_int8, Kd)
    flushed_step_ms = timed(lambda: (step_int8(), decode_int8()), Kd)

    # each decode variant alone, back to back like the timed steps, one pair
    # of events around the run (the dominant kernel, for the roofline)
    def back_to_back(fn, reps):
        torch.cuda.synchronize()
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(reps):
            fn()
        b1.record(stream)
        b1.synchronize()
        return b0.elapsed_time(b1) / reps

    b2b = {name: back_to_back(fn, Kd) for name, fn in (("decode_int8", p_int8),
                                                        ("decode_fp8", p_fp8),
                                                        ("decode_fp16", p_fp16))}

    # labelled extra: the same step (tail quantize + INT8 decode) captured once
    # in a CUDA graph and replayed, L2 still flushed outside each replay
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step_int8()
        decode_int8()
    for _ in range(args.warmup):
        graph.replay()
    graph_ms = timed(graph.replay, Kd)

    # the write before a decode step: every sequence's newest token appended
    # (fp16 rows; INT8 with the fused re-quantize of the tail tiles)
    kn, vn, pos = W.append_tokens(w, 99)
    app_args = (dev(kn), dev(vn), bt, dev(pos))
    app16_ms = timed(lambda: pkv.pkv_append_fp16(kf, vf, *app_args, dev_status=status), Kd)
    app8_ms = timed(lambda: pkv.pkv_append_int8(kf, vf, kc, vc, ks, vs, *app_args,
                                                 dev_status=status), Kd)

    # copy-on-write copies of K and V blocks (all kv heads), fp16 pools
    copies = {}
    for n_pairs in COPY_PAIRS:
        rng_c = np.random.default_rng(n_pairs)
        perm = rng_c.permutation(w.num_blocks)
        pairs = dev(np.stack([perm[:n_pairs], perm[n_pairs:2 * n_pairs]], 1).astype(np.int32))
        fn_c = lambda: pkv.pkv_copy_blocks([kf, vf], pairs, status)
        for _ in range(args.warmup):
            fn_c()
        ms_c = timed(fn_c, Kd)
        moved = 2 * n_pairs * 2 * hkv * 16 * d * 2  # K and V, read + written
        copies[str(n_pairs)] = {"p50_us": 1e3 * statistics.median(ms_c),
                                "GB/s": moved / (statistics.mean(ms_c) * 1e-3) / 1e9,
                                "frac_of_peak": moved / (statistics.mean(ms_c) * 1e-3) / 1e9
                                / _peaks()[0],
                                "bytes": moved}
    bm_rate = {"native_blocks_per_s": block_manager_rate()}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        bm_rate["oracle_model_blocks_per_s"] = block_manager_rate(model=True)

    # eviction scoring + choice of 15 % of the blocks, at the pages' pool sizes
    evict = {}
    for nb_e in EVICT_SIZES:
        st_e = W.eviction_state(nb_e, 7)
        ref_e, last_e = dev(st_e.refcnt), dev(st_e.last_used)
        k_e = pkv.evict_count(nb_e)
        ids_e = torch.empty(k_e, dtype=torch.int32, device="cuda")
        cnt_e = torch.empty(1, dtype=torch.int32, device="cuda")
        sc_e = torch.empty(nb_e, dtype=torch.float32, device="cuda")
        fn_e = lambda: pkv.pkv_evict_select(ref_e, last_e, st_e.current_tick, k_e, ids_e,
                                            cnt_e, sc_e)
        for _ in range(args.warmup):
            fn_e()
        ms_e = timed(fn_e, Kd)
        evict[str(nb_e)] = {"p50_us": 1e3 * statistics.median(ms_e),
                            "p90_us": 1e3 * float(np.percentile(ms_e, 90)), "k": k_e,
                            "GB/s": evict_bytes(nb_e, k_e) / (statistics.mean(ms_e) * 1e-3) / 1e9,
                            "bytes": evict_bytes(nb_e, k_e)}
        if rank == 0 and ws == 1 and not args.no_cpu_baseline:
            evict[str(nb_e)]["cpu_oracle_p50_us"] = evict_cpu_us(nb_e)

    # end to end through the public API with host buffers.  The step's small
    # inputs (query, block tables, context lengths, tail ids) are staged in
    # one pinned host buffer, as a serving loop would stage them, and the
    # output goes to pinned host memory.  Headline form: the kernels read the
    # staged inputs and write the output in place over the GPU's link to the
    # host (pinned memory has one address for both; no copy operations).
    # Also timed: one copy-engine copy of the staging buffer in and one of
    # the output back around the same step.
    parts = [w.query, w.block_tables, w.context_lens, tails_np]
    offs, total_b = [], 0
    for a in parts:
        offs.append(total_b)
        total_b += (a.nbytes + 255) // 256 * 256
    host_stage = torch.empty(total_b, dtype=torch.uint8).pin_memory()
    dev_stage = torch.empty(total_b, dtype=torch.uint8, device="cuda")
    views = []
    for a, o in zip(parts, offs):
        host_stage[o:o + a.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)))
        views.append(dev_stage[o:o + a.nbytes].view(torch.from_numpy(a).dtype).view(a.shape))
    q_e, bt_e, cl_e, tl_e = views
    hviews = [host_stage[o:o + a.nbytes].view(torch.from_numpy(a).dtype).view(a.shape)
              for a, o in zip(parts, offs)]
    q_h, bt_h, cl_h, tl_h = hviews
    hout = torch.empty((n, hq, d), dtype=torch.float32).pin_memory()
    hout_ce = torch.empty((n, hq, d), dtype=torch.float32).pin_memory()
    Ke = min(K, 2000)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def e2e_in_place():
        pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, tl_h, status)
        pkv.pkv_paged_decode_int8(hout, q_h, kc, vc, ks, vs, bt_h, cl_h, mcl, w.softmax_scale,
                                  ws_t, status)

    def e2e_copies():
        dev_stage.copy_(host_stage, non_blocking=True)
        pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, tl_e, status)
        pkv.pkv_paged_decode_int8(out, q_e, kc, vc, ks, vs, bt_e, cl_e, mcl, w.softmax_scale,
                                  ws_t, status)
        hout_ce.copy_(out, non_blocking=True)

    e2e_ms, e2e_ce_ms = 0.0, 0.0
    for fn, which in ((e2e_in_place, 0), (e2e_copies, 1)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        for i in range(Ke):
            l2_flush()
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if which == 0:
                e2e_ms += e0.elapsed_time(e1)
            else:
                e2e_ce_ms += e0.elapsed_time(e1)
    assert torch.equal(hout, out.cpu()) and torch.equal(hout_ce, hout)

    # End to end, steps back to back as a serving loop runs them, the host
    # reading each step's output while the next step runs.  Labelled extra:
    # the kernels read the staged inputs and write the output in pinned host
    # memory (two output buffers, used in turn).
    hout2 = [torch.empty((n, hq, d), dtype=torch.float32).pin_memory() for _ in range(2)]
    hout2_np = [x.numpy() for x in hout2]  # host views: reading them is a plain memory read

    def pipelined_in_place(reps):
        done = [torch.cuda.Event() for _ in range(2)]
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        seen = 0.0
        torch.cuda.synchronize()
        p0.record(stream)
        for i in range(reps):
            b = i & 1
            pkv.pkv_quantize_blocks(kf, vf, kc, vc, ks, vs, tl_h, status)
            pkv.pkv_paged_decode_int8(hout2[b], q_h, kc, vc, ks, vs, bt_h, cl_h, mcl,
                                      w.softmax_scale, ws_t, status)
            done[b].record(stream)
            if i >= 1:
                done[b ^ 1].synchronize()
                seen += float(hout2_np[b ^ 1][0, 0, 0])  # the previous step's output, on the host
        p1.record(stream)
        p1.synchronize()
        seen += float(hout2_np[(reps - 1) & 1][0, 0, 0])
        return p0.elapsed_time(p1) / reps

    # Headline: a copy stream brings the next step's inputs into one of two
    # device staging buffers and the finished step's output back to one of
    # two pinned buffers while a step runs; the calls of each staging buffer
    # are prepared once.
    dev_stage2 = [dev_stage, torch.empty_like(dev_stage)]
    dviews = [[buf[o:o + a.nbytes].view(torch.from_numpy(a).dtype).view(a.shape)
               for a, o in zip(parts, offs)] for buf in dev_stage2]
    out2 = [out, torch.empty_like(out)]
    hout_ce2 = [torch.empty((n, hq, d), dtype=torch.float32).pin_memory() for _ in range(2)]
    hout_ce2_np = [x.numpy() for x in hout_ce2]
    cstream = torch.cuda.Stream()
    pq2 = [pkv.prepare_quantize_blocks(kf, vf, kc, vc, ks, vs, dviews[b][3], status)
           for b in range(2)]
    pd2 = [pkv.prepare_paged_decode_int8(out2[b], dviews[b][0], kc, vc, ks, vs, dviews[b][1],
                                         dviews[b][2], mcl, w.softmax_scale, ws_t, status)
           for b in range(2)]

    def pipelined_copies(reps):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        out_ready = [torch.cuda.Event() for _ in range(2)]
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        seen = 0.0
        torch.cuda.synchronize()
        p0.record(stream)
        cstream.wait_stream(stream)
        with torch.cuda.stream(cstream):
            dev_stage2[0].copy_(host_stage, non_blocking=True)
            in_ready[0].record(cstream)
        for i in range(reps):
            b = i & 1
            # the host, not the stream, waits for the inputs (copied a step
            # ago), so the main stream stays a chain of kernels whose launches
            # overlap under programmatic dependent launch
            in_ready[b].synchronize()
            pq2[b]()
            pd2[b]()
            done[b].record(stream)
            with torch.cuda.stream(cstream):
                if i + 1 < reps:
                    if i >= 1:
                        cstream.wait_event(done[b ^ 1])  # step i - 1 has read buffer b ^ 1
                    dev_stage2[b ^ 1].copy_(host_stage, non_blocking=True)
                    in_ready[b ^ 1].record(cstream)
                cstream.wait_event(done[b])
                hout_ce2[b].copy_(out2[b], non_blocking=True)
                out_ready[b].record(cstream)
            if i >= 1:
                out_ready[b ^ 1].synchronize()
                seen += float(hout_ce2_np[b ^ 1][0, 0, 0])  # the previous step's output, on the host
        stream.wait_stream(cstream)
        p1.record(stream)
        p1.synchronize()
        seen += float(hout_ce2_np[(reps - 1) & 1][0, 0, 0])
        return p0.elapsed_time(p1) / reps

    pipelined_in_place(200)  # warm-up: the copy paths settle over the first few hundred steps
    pipelined_copies(200)
    gc.disable()  # no collector pauses inside the host loops
    try:
        if pg:
            pg.barrier()
        e2e_pipe_ms = pipelined_in_place(Ke)
        if pg:
            pg.barrier()
        e2e_pipe_ce_ms = pipelined_copies(Ke)
    finally:
        gc.enable()
    if pg:
        # whole-job end-to-end: every rank's steps over the slowest rank's time
        t = torch.tensor([e2e_pipe_ms, e2e_pipe_ce_ms], device="cuda")
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        e2e_pipe_ms, e2e_pipe_ce_ms = float(t[0].item()), float(t[1].item())
    assert all(torch.equal(x, hout) for x in hout2 + hout_ce2)
    # bytes of the step's host inputs (read in place; a query row is read by
    # each worker holding a piece of its item) and of its output
    h2d = sum(a.nbytes for a in parts)
    d2h = n * hq * d * 4
    st_val = int(status.item())

    ntiles = len(tails_np) * hkv
    dec_b = decode_bytes(w.context_lens, hkv, d, 1, True)
    step_b = dec_b + quantize_bytes(ntiles, d)
    f16_b = decode_bytes(w.context_lens, hkv, d, 2, False)
    value = step_b * K * ws / (total_ms * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    dec_avg_ms = b2b["decode_int8"]
    achieved = dec_b / (dec_avg_ms * 1e-3) / 1e9
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9
    traffic = TRAFFIC.get("decode_int8")
    if traffic is not None and traffic[1] != _src_hash():
        traffic = None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8-kv f16-mma f32-acc",
        "data": "synthetic",
        "config": {"workload": workload_desc(w, len(tails_np)),
                   "l2": "inputs larger than L2, no flush: each step reads 270 MB of INT8 "
                         "codes against the 129 MB L2, and a back-to-back call reads all "
                         "of its algorithmic bytes from DRAM (ncu, cache control off); "
                         "steps timed back to back between one pair of events",
                   "flushed_per_call": "labelled extra: L2 flushed (256 MiB written, "
                                       "then 256 MiB read) before every call, one pair "
                                       "of events around each call",
                   "parallelism": f"weak: the batch replicated per GPU x{ws}"},
        "seq_steps_per_s": n * K * ws / (total_ms * 1e-3),
        "p50_us_per_step": 1e3 * statistics.median(step_ms),
        "p90_us_per_step": 1e3 * float(np.percentile(step_ms, 90)),
        "per_step_distribution": f"{nblk} blocks of {blk} steps back to back, an event after "
                                 "each block",
        "pct_hbm_peak": 100.0 * value / ws / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "kernel": "INT8 decode call (decode + reduce kernels), "
                               f"{dec_b} algorithmic bytes per call, {Kd} calls back "
                               "to back between one pair of events",
                     "traffic": None if traffic is None else traffic[0]},
        "flushed_per_call": {
            "step_mean_us": 1e3 * statistics.mean(flushed_step_ms),
            "step_p50_us": 1e3 * statistics.median(flushed_step_ms),
            "step_GB/s": gbs(step_b, statistics.mean(flushed_step_ms)),
            "decode_int8_mean_us": 1e3 * statistics.mean(dec_ms),
            "decode_int8_frac_of_peak": gbs(dec_b, statistics.mean(dec_ms)) / peak,
            "calls": Kd},
        "variants": {
            "decode_fp16": {"us": 1e3 * b2b["decode_fp16"],
                            "GB/s": gbs(f16_b, b2b["decode_fp16"]),
                            "frac_of_peak": gbs(f16_b, b2b["decode_fp16"]) / peak,
                            "bytes": f16_b,
                            "flushed_p50_us": 1e3 * statistics.median(f16_ms),
                            "flushed_frac_of_peak": gbs(f16_b, statistics.mean(f16_ms)) / peak},
            "decode_int8": {"us": 1e3 * b2b["decode_int8"], "GB/s": achieved,
                            "frac_of_peak": achieved / peak, "bytes": dec_b,
                            "flushed_p50_us": 1e3 * statistics.median(dec_ms),
                            "flushed_frac_of_peak": gbs(dec_b, statistics.mean(dec_ms)) / peak},
            "decode_fp8": {"us": 1e3 * b2b["decode_fp8"],
                           "GB/s": gbs(dec_b, b2b["decode_fp8"]),
                           "frac_of_peak": gbs(dec_b, b2b["decode_fp8"]) / peak,
                           "bytes": dec_b,
                           "flushed_p50_us": 1e3 * statistics.median(f8_ms),
                           "flushed_frac_of_peak": gbs(dec_b, statistics.mean(f8_ms)) / peak},
            "step_cuda_graph": {"p50_us": 1e3 * statistics.median(graph_ms),
                                "GB/s": step_b / (statistics.mean(graph_ms) * 1e-3) / 1e9,
                                "bytes": step_b},
            "quantize_tail_blocks": {"p50_us": 1e3 * statistics.median(q_ms),
                                     "tiles": 2 * ntiles,
                                     "bytes": quantize_bytes(ntiles, d)},
            "append_fp16": {"p50_us": 1e3 * statistics.median(app16_ms), "rows": 2 * ntiles,
                            "bytes": append_bytes(ntiles, d, False)},
            "append_int8_fused_requantize": {"p50_us": 1e3 * statistics.median(app8_ms),
                                             "tiles": 2 * ntiles,
                                             "bytes": append_bytes(ntiles, d, True)},
            "evict_select_15pct": evict,
            "cow_copy_blocks_fp16": copies,
            "block_manager_host": bm_rate,
        },
        "e2e": {"value": gbs(step_b * ws, e2e_pipe_ce_ms), "unit": UNIT,
                "h2d_bytes_per_step": total_b * ws, "d2h_bytes_per_step": d2h * ws, "steps": Ke,
                "form": "steps back to back through prepared calls; a copy stream copies each "
                        "step's staged inputs (query, block tables, context lengths, tail ids) "
                        "from pinned host memory into one of two device buffers while the step "
                        "before runs, and its output back into one of two pinned buffers, "
                        "which the host reads while the next step runs",
                "in_place": {"value": gbs(step_b * ws, e2e_pipe_ms),
                             "form": "labelled extra: steps back to back; the kernels read each "
                                     "step's staged inputs and write its output in place in "
                                     "pinned host memory (no copy operations)",
                             "h2d_bytes_per_step": h2d * ws, "d2h_bytes_per_step": d2h * ws},
                "per_step_sync": {
                    "ranks": "rank 0 alone",
                    "form": "labelled extra: L2 flushed, then one step with a pair of events "
                            "around it and the host waiting for its output before the next",
                    "in_place": step_b * Ke / (e2e_ms * 1e-3) / 1e9,
                    "copy_engine": step_b * Ke / (e2e_ce_ms * 1e-3) / 1e9}},
        "gpu_launches": 3 * K,
        "dev_status": st_val,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()

"""Benchmark of the Quest decode step on one GB300 (or N replicas under torchrun).

Workload: one LongChat-7B-shaped layer (32 MHA heads, d=128, page 16), 32768 prefilled
tokens, token budget 2048 (128 pages); a step is one quest_decode_step call: append one
token, score, top-K, sparse decode, through the path the library chooses (here the chain:
the estimate kernel, then the sparse-decode kernel whose work items each take their pair's
top-K; --path fused / stream / chain to force a path).  Steps cycle through the workload's
64 appended tokens (contexts 32769..32832); the cache is rewound outside the timed region.

Inputs larger than L2: 8 (or more) independent copies of the workload (4.6 GB) are taken in
rotation, so that each call's boxes and pages (67 MB) were evicted by the other copies'
calls; the calls run back to back through a DecodePlan (arguments checked once), one event
pair around the timed steps.  Also reported (detail_us): the same steps one at a time after
an L2 flush (a 512 MiB write, then a 256 MiB read) with p50 / p90 / max, quest_decode alone,
and the host time spent issuing each step.  ``e2e``: the step from pinned host buffers, one
packed host-to-device copy and one device-to-host copy of out + lse per step, on a copy
stream, double-buffered so that a step's copies overlap its neighbours' kernels.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse decode µs/step & HBM GB/s (frac of roofline), 32K ctx, 2048 budget"
PATH_NAMES = {1: "fused", 2: "chain", 3: "stream"}
FLUSH_BYTES = 512 << 20
PAGE = 16


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--copies", type=int, default=0,
                    help="workload copies taken in rotation (0: enough for the steps, 8 to 32)")
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="quest", choices=["quest", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--pages-per-split", type=int, default=0)
    ap.add_argument("--score-tile-pages", type=int, default=0)
    ap.add_argument("--trace", default="", help="write a fused-kernel timeline (npy) here")
    ap.add_argument("--path", default="auto", choices=["auto", "fused", "chain", "stream"],
                    help="quest_decode / quest_decode_step path (default: the library's choice)")
    ap.add_argument("--cluster-size", type=int, default=0,
                    help="CTAs per (sequence, kv head) cluster for --sweep / --layers (0: automatic)")
    ap.add_argument("--layers", action="store_true",
                    help="time the 32-layer 128K step in one launch against one launch per layer")
    ap.add_argument("--prefill", action="store_true",
                    help="time the chunked-prefill write (quest_prefill) at several chunk sizes")
    ap.add_argument("--sweep", action="store_true",
                    help="measure every workload (one JSON line each) instead of the step")
    ap.add_argument("--profile-decode", type=int, default=0, metavar="N",
                    help="profiling run for ncu: set up, --warmup steps, then N quest_decode "
                         "launches; no L2 flush buffer, no timing, no JSON line")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------------------------
# algorithmic bytes (what the step must move): metadata of every page of every head,
# the K and V rows of every valid token of every selected page, q in, out + lse out.
# ------------------------------------------------------------------------------------
def decode_bytes(seq_lens, counts_tokens, B, Hq, Hkv, d=128, page=PAGE):
    meta = sum(math.ceil(L / page) for L in seq_lens) * Hkv * 2 * d * 2
    kv = counts_tokens * 2 * d * 2
    qo = B * Hq * d * 2 * 2 + B * Hq * 4
    return meta + kv + qo


def append_bytes(B, Hkv, d=128):
    # read k_new, v_new; write the K and V rows; read+write the page box (min and max)
    return B * Hkv * d * 2 * (2 + 2 + 4)


def selected_tokens(idx, cnt, seq_lens, page=PAGE):
    import numpy as np
    idx = idx.cpu().numpy()
    cnt = cnt.cpu().numpy()
    total = 0
    for b in range(idx.shape[0]):
        L = int(seq_lens[b])
        for g in range(idx.shape[1]):
            for p in idx[b, g, :cnt[b, g]]:
                total += min(page, L - int(p) * page)
    return total


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]
        else:
            self.lines = []

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        busy = [s for s in sm if mx is None or s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm, and the cpu_baseline key)
# ------------------------------------------------------------------------------------
def oracle_timing(w, budget_s: float, max_steps: int, warmup: int = 0):
    import numpy as np
    import oracle
    oracle.build()
    ref = oracle.Cache.from_arrays(w.k_pool.cpu().numpy(), w.v_pool.cpu().numpy(),
                                   w.block_table.cpu().numpy(), w.seq_lens.cpu().numpy(),
                                   w.num_q_heads)
    oracle.build_meta(ref)
    qs, ks, vs = w.q.cpu().numpy(), w.k_new.cpu().numpy(), w.v_new.cpu().numpy()
    for t in range(min(warmup, w.steps)):  # untimed, then the cache is rewound
        oracle.decode_step(ref, qs[t], w.top_k, ks[t], vs[t])
    if warmup:
        ref.seq_lens[:] = w.seq_lens.cpu().numpy()
        oracle.build_meta(ref)
    times = []
    t_start = time.perf_counter()
    n = 0
    while n < max_steps:
        t = n % w.steps
        if t == 0 and n > 0:
            ref.seq_lens[:] = w.seq_lens.cpu().numpy()
            oracle.build_meta(ref)  # rewind (outside the per-step timing)
        t0 = time.perf_counter()
        oracle.decode_step(ref, qs[t], w.top_k, ks[t], vs[t])
        times.append(time.perf_counter() - t0)
        n += 1
        if time.perf_counter() - t_start > budget_s:
            break
    us = 1e6 * sum(times) / len(times)
    return us, len(times)


def oracle_timing_all_cores(w, budget_s: float):
    """The oracle's score + top-K + attend on every host core at once (one thread per core,
    each on its own query of the workload, the cache shared read-only; the C calls release
    the interpreter lock).  Returns (us per step at full occupancy, steps, threads)."""
    import concurrent.futures as cf
    import oracle
    oracle.build()
    ref = oracle.Cache.from_arrays(w.k_pool.cpu().numpy(), w.v_pool.cpu().numpy(),
                                   w.block_table.cpu().numpy(), w.seq_lens.cpu().numpy(),
                                   w.num_q_heads)
    oracle.build_meta(ref)
    qs = w.q.cpu().numpy()
    threads = max(1, os.cpu_count() or 1)

    def one(t):
        s = oracle.score(ref, qs[t % w.steps])
        i, c = oracle.topk(ref, s, w.top_k)
        oracle.attend(ref, qs[t % w.steps], i, c)

    one(0)
    steps = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:
        while True:
            list(ex.map(one, range(steps, steps + threads)))
            steps += threads
            if time.perf_counter() - t0 > budget_s:
                break
    wall = time.perf_counter() - t0
    return 1e6 * wall / steps, steps, threads


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from query_aware_kv_gb300 import workloads as wl
    w = wl.longchat_32k(seed=0, device="cpu")
    warm = max(0, args.warmup)
    us, n = oracle_timing(w, budget_s=min(240.0, 0.05 * max(1, args.steps) + 60.0),
                          max_steps=max(1, args.steps), warmup=warm)
    cpu = {"value": us, "unit": "us/step", "cores": 1, "kind": "oracle",
           "sample": f"{n} of the {args.steps} requested decode steps (append + score + "
                     f"top-K + attend), single-threaded C oracle, contexts 32769..32832"}
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us/step",
            "n_gpus": args.gpus, "steps": n, "warmup": min(warm, w.steps), "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, **w.describe()},
            "cpu_baseline": cpu,
            "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------
class _Driver:
    """Asynchronous copies and event calls through the CUDA driver (libcuda), for the
    end-to-end loop: plain cuMemcpyHtoDAsync / cuMemcpyDtoHAsync, one per copy."""

    def __init__(self):
        import ctypes
        lib = ctypes.CDLL("libcuda.so.1")
        V, SZ = ctypes.c_void_p, ctypes.c_size_t
        U64 = ctypes.c_uint64
        self._h2d = lib.cuMemcpyHtoDAsync_v2
        self._h2d.argtypes = [U64, V, SZ, V]
        self._d2h = lib.cuMemcpyDtoHAsync_v2
        self._d2h.argtypes = [V, U64, SZ, V]
        self._rec = lib.cuEventRecord
        self._rec.argtypes = [V, V]
        self._wait = lib.cuStreamWaitEvent
        self._wait.argtypes = [V, V, ctypes.c_uint]
        for f in (self._h2d, self._d2h, self._rec, self._wait):
            f.restype = ctypes.c_int

    @staticmethod
    def _ok(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed with CUresult {rc}")

    def h2d(self, dst, src, n, stream):
        self._ok(self._h2d(dst, src, n, stream), "cuMemcpyHtoDAsync")

    def d2h(self, dst, src, n, stream):
        self._ok(self._d2h(dst, src, n, stream), "cuMemcpyDtoHAsync")

    def record(self, event, stream):
        self._ok(self._rec(event, stream), "cuEventRecord")

    def wait(self, stream, event):
        self._ok(self._wait(stream, event, 0), "cuStreamWaitEvent")


def run_quest(args):
    import types

    import numpy as np
    import torch
    import torch.distributed as dist

    import query_aware_kv_gb300 as q
    from query_aware_kv_gb300 import build as cuda_build
    from query_aware_kv_gb300 import workloads as wl

    from query_aware_kv_gb300 import replicas

    ri = replicas.rank_info()
    world, rank, local = ri.world, ri.rank, ri.local
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        cuda_build.build()
    if world > 1:
        dist.barrier()
    q.load()

    # Independent copies of the workload (each rank decodes its own sequences: weak scaling,
    # no collective).  Calls rotate over the copies, so that between two calls on one copy
    # the other copies stream several times the L2's 129 MB: every call reads its boxes and
    # pages from DRAM, with the calls back to back as in a decode loop.
    n = args.steps
    ncopy = args.copies if args.copies > 0 else max(8, min(32, -(-n // 64)))
    base_seed = replicas.workload_seed(rank)
    copies = []
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    build_meta_us = 0.0
    for ci in range(ncopy):
        w = wl.longchat_32k(seed=base_seed * 1000 + ci, device=dev)
        cache = q.PagedCache.allocate_meta(w.k_pool, w.v_pool, w.block_table, w.seq_lens.clone(),
                                           w.num_q_heads)
        ws = q.workspace(cache, w.top_k)
        torch.cuda.synchronize()
        t0.record()
        q.build_meta(cache, ws)
        t1.record()
        torch.cuda.synchronize()
        if ci == 0:
            build_meta_us = 1e3 * t0.elapsed_time(t1)
        copies.append(types.SimpleNamespace(w=w, cache=cache, ws=ws, meta0=cache.meta.clone(),
                                            len0=w.seq_lens.clone()))
    w = copies[0].w
    cache, ws = copies[0].cache, copies[0].ws
    K = w.top_k
    steps_per_copy = w.steps
    seg = steps_per_copy * ncopy  # steps before the copies must be rewound
    flush_buf = None if args.profile_decode else torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sum = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        # write more than L2 holds, then read more than it holds: L2 ends clean and
        # without any of the workload's lines
        flush_buf.zero_()
        torch.sum(flush_buf[: FLUSH_BYTES // 2].view(torch.int64), dim=0, out=flush_sum)
    out = torch.empty((1, w.num_q_heads, 128), dtype=torch.float16, device=dev)
    lse = torch.empty((1, w.num_q_heads), dtype=torch.float32, device=dev)
    idx = torch.empty((1, w.num_kv_heads, K), dtype=torch.int32, device=dev)
    cnt = torch.empty((1, w.num_kv_heads), dtype=torch.int32, device=dev)
    path = {"auto": q.QUEST_PATH_AUTO, "fused": q.QUEST_PATH_FUSED,
            "chain": q.QUEST_PATH_CHAIN, "stream": q.QUEST_PATH_STREAM}[args.path]
    opts_main = q.opts(pages_per_split=args.pages_per_split,
                       score_tile_pages=args.score_tile_pages, path=path)

    def rewind_all():
        for c in copies:
            c.cache.meta.copy_(c.meta0)
            c.cache.seq_lens.copy_(c.len0)

    # one prepared call per copy (arguments checked once), and every step's inputs as their
    # own tensors, as a decode loop has them
    for c in copies:
        c.plan = q.DecodePlan(c.cache, K, c.ws, opts_main, out=out, lse=lse, idx_out=idx,
                              count_out=cnt)
        c.qs = [c.w.q[t] for t in range(steps_per_copy)]
        c.kns = [c.w.k_new[t] for t in range(steps_per_copy)]
        c.vns = [c.w.v_new[t] for t in range(steps_per_copy)]

    def step(i):
        c = copies[i % ncopy]
        t = (i // ncopy) % steps_per_copy
        c.plan.step(c.qs[t], c.kns[t], c.vns[t])

    host_issue = [0.0, 0]  # host seconds spent issuing calls, and those calls (last timed_steps)
    # Position of the next step in the rotation (0..seg-1): step i appends to copy i % ncopy.
    # The copies are rewound only when every one is full, so that a timed run follows its
    # warm-up directly instead of starting behind a rewind (whose writes leave the L2 dirty).
    cursor = [0]

    def take(m_max):
        """Room for up to m_max more steps before a rewind (rewinding first if there is
        none); returns (first position, steps)."""
        if cursor[0] >= seg:
            rewind_all()
            cursor[0] = 0
        m = min(m_max, seg - cursor[0])
        first = cursor[0]
        cursor[0] += m
        return first, m

    def timed_steps(count, fn):
        """`count` calls of fn(position) back to back, in segments that end where the copies
        must be rewound (outside the timed intervals).  Returns total ms."""
        total = 0.0
        done = 0
        host_issue[0], host_issue[1] = 0.0, 0
        while done < count:
            first, m = take(count - done)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            t0.record()
            # host time to issue the first (up to) 128 calls of the segment: later calls can
            # wait for room in the launch queue once the GPU falls behind
            h_n = min(m, 128)
            h0 = time.perf_counter()
            for i in range(first, first + h_n):
                fn(i)
            host_issue[0] += time.perf_counter() - h0
            host_issue[1] += h_n
            for i in range(first + h_n, first + m):
                fn(i)
            t1.record()
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            total += t0.elapsed_time(t1)
            done += m
        return total

    if args.profile_decode:
        rewind_all()
        for i in range(args.warmup):
            step(i)
        for i in range(args.profile_decode):
            c = copies[i % ncopy]
            q.decode(c.cache, c.w.q[i % w.steps], K, c.ws, opts_main, out=out, lse=lse,
                     idx_out=idx, count_out=cnt)
        torch.cuda.synchronize()
        rc, detail = q.read_status(ws)
        print(f"profile run: {args.warmup} steps + {args.profile_decode} quest_decode launches, "
              f"status {rc}", flush=True)
        return

    # set-up: one decode (no append, so the caches are unchanged) through every copy's
    # DecodePlan, so that no first-time host or driver cost of a copy lands in a timed step
    for c in copies:
        c.plan.decode(c.qs[0])
    torch.cuda.synchronize()
    # warm-up: the flushed per-step loop's calls, then the timed loop's own (last, so that
    # the timed steps do not start behind a flush that evicted the kernels' code from L2)
    for _ in range(max(1, args.warmup)):
        i, _m = take(1)
        flush_l2()
        t0.record()
        step(i)
        t1.record()
    torch.cuda.synchronize()
    timed_steps(max(1, args.warmup), step)
    torch.cuda.synchronize()
    for c in copies:
        rc, detail = q.read_status(c.ws)
        if rc != 0:
            raise RuntimeError(f"device status {rc} {detail}")

    # ---- timed: exactly n steps (append + score + top-K + sparse decode), back to back
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        total_ms = timed_steps(n, step)
        wall = time.perf_counter() - wall0
    mean_step = 1e3 * total_ms / n
    host_issue_us = 1e6 * host_issue[0] / max(1, host_issue[1])
    for c in copies:
        rc, detail = q.read_status(c.ws)
        if rc != 0:
            raise RuntimeError(f"device status {rc} {detail}")

    # the same steps one at a time, each after an L2 flush and between its own events (the
    # per-call latency including a launch's fixed cost; detail only)
    fn_ = min(n, 256)
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(fn_)]
    for i in range(fn_):
        pos, _m = take(1)
        flush_l2()
        fev[i][0].record()
        step(pos)
        fev[i][1].record()
    torch.cuda.synchronize()
    flushed_us = [1e3 * a.elapsed_time(b) for a, b in fev]

    # ---- kernel-only: quest_decode alone at one context per copy (after its 64 tokens)
    rewind_all()
    cursor[0] = seg  # every copy is filled below: the next step rewinds first
    for c in copies:
        for t in range(c.w.steps):
            q.append(c.cache, c.w.k_new[t], c.w.v_new[t], c.ws)
    L_fixed = [int(x) for x in cache.seq_lens.cpu().tolist()]

    def one_decode(i):
        c = copies[i % ncopy]
        c.plan.decode(c.qs[(i // ncopy) % steps_per_copy])
    kn = min(max(n, 4 * ncopy), 512)
    for i in range(ncopy):  # warm
        one_decode(i)
    torch.cuda.synchronize()
    t0.record()
    for i in range(kn):
        one_decode(i)
    t1.record()
    torch.cuda.synchronize()
    dec_us = 1e3 * t0.elapsed_time(t1) / kn
    # one call at a time after an L2 flush (detail), and back to back on one copy with the L2
    # left warm (the boxes, 32 MiB, stay in the 129 MB L2 from one call to the next: detail)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(64)]
    for i in range(64):
        flush_l2()
        kev[i][0].record()
        one_decode(i * ncopy)
        kev[i][1].record()
    torch.cuda.synchronize()
    dec_flushed_us = sum(1e3 * a.elapsed_time(b) for a, b in kev) / 64
    plan0, qs0 = copies[0].plan, copies[0].qs
    t0.record()
    for i in range(kn):
        plan0.decode(qs0[i % steps_per_copy])
    t1.record()
    torch.cuda.synchronize()
    dec_warm_us = 1e3 * t0.elapsed_time(t1) / kn
    if args.trace:
        cap = 1 << 17
        tr = torch.zeros(1 + 2 * cap, dtype=torch.int64, device=dev)
        o_tr = q.opts(pages_per_split=args.pages_per_split,
                      score_tile_pages=args.score_tile_pages, trace=tr, path=path)
        flush_l2()
        q.decode(cache, w.q[0], K, ws, o_tr, out=out, lse=lse)
        torch.cuda.synchronize()
        rec = tr[1:].view(cap, 2).cpu().numpy()
        np.save(args.trace, rec[rec[:, 0] != 0])
    q.decode(cache, w.q[0], K, ws, opts_main, out=out, lse=lse, idx_out=idx, count_out=cnt)
    tok = selected_tokens(idx, cnt, L_fixed)
    dec_bytes = decode_bytes(L_fixed, tok, 1, w.num_q_heads, w.num_kv_heads)

    # ---- the unfused chain and the dense baseline at the same context (flushed, detail)
    def timed(fn, reps=64):
        es = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a, b in es:
            flush_l2()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sum(1e3 * a.elapsed_time(b) for a, b in es) / reps

    scores = torch.empty((1, w.num_kv_heads, cache.max_pages), dtype=torch.float32, device=dev)
    qv = w.q[0]

    def chain():
        q.estimate(cache, qv, ws, scores=scores)
        i2, c2 = q.topk(cache, scores, K, ws)
        q.sparse_decode(cache, qv, i2, c2, K, ws, out=out, lse=lse)

    chain_us = timed(chain)
    dense_us = timed(lambda: q.dense_decode(cache, qv, ws, out=out, lse=lse), reps=32)
    for c in copies:
        rc, detail = q.read_status(c.ws)
        if rc != 0:
            raise RuntimeError(f"device status {rc} {detail}")

    # ---- end to end through the public API with host buffers (pinned), copies timed: each
    # step's q, k_new and v_new travel in one host->device copy of a packed staging row, and
    # out + lse come back in one device->host copy, each on a copy stream of its own,
    # double-buffered, so that step i's copies overlap steps i-1 / i+1's kernels as in a
    # serving loop; back to back over the rotating copies
    nq, nk = w.q[0].numel(), w.k_new[0].numel()
    hstage = [torch.cat([c.w.q.reshape(c.w.steps, -1), c.w.k_new.reshape(c.w.steps, -1),
                         c.w.v_new.reshape(c.w.steps, -1)], dim=1).cpu().pin_memory()
              for c in copies]
    hstage_rows = [[h[t] for t in range(steps_per_copy)] for h in hstage]
    out_bytes, lse_bytes = out.numel() * 2, lse.numel() * 4
    cs = torch.cuda.Stream(device=dev)      # inputs in
    cs_out = torch.cuda.Stream(device=dev)  # results out (a stream of its own, so that the
                                            # next step's input never queues behind a result)
    main = torch.cuda.current_stream()
    cu = _Driver()  # the copies and event calls straight through the driver: a fraction of
                    # the host time of torch's stream context and copy calls
    main_h, cs_h, out_h = main.cuda_stream, cs.cuda_stream, cs_out.cuda_stream
    slots = []
    for _ in range(2):
        dstage = torch.empty(hstage[0].shape[1], dtype=torch.float16, device=dev)
        dres = torch.empty(out_bytes + lse_bytes, dtype=torch.uint8, device=dev)
        eout = dres[:out_bytes].view(torch.float16).view_as(out)
        else_ = dres[out_bytes:].view(torch.float32).view_as(lse)
        sl = types.SimpleNamespace(
            dstage=dstage, dres=dres,
            dq=dstage[:nq].view_as(w.q[0]), dk=dstage[nq:nq + nk].view_as(w.k_new[0]),
            dv=dstage[nq + nk:].view_as(w.v_new[0]),
            hres=torch.empty(out_bytes + lse_bytes, dtype=torch.uint8).pin_memory(),
            plans=[q.DecodePlan(c.cache, K, c.ws, opts_main, out=eout, lse=else_)
                   for c in copies],
            h2d=torch.cuda.Event(), comp=torch.cuda.Event(), d2h=torch.cuda.Event())
        sl.h2d.record(main)  # creates the events; every one starts recorded
        sl.comp.record(main)
        sl.d2h.record(main)
        sl.ev = (sl.h2d.cuda_event, sl.comp.cuda_event, sl.d2h.cuda_event)
        sl.dst_in, sl.src_res = sl.dstage.data_ptr(), sl.dres.data_ptr()
        sl.hres_ptr, sl.nin, sl.nres = sl.hres.data_ptr(), sl.dstage.numel() * 2, sl.dres.numel()
        slots.append(sl)
    host_rows = [[r.data_ptr() for r in rows] for rows in hstage_rows]
    torch.cuda.synchronize()

    def e2e_step(i):
        ci = i % ncopy
        t = (i // ncopy) % steps_per_copy
        sl = slots[i & 1]
        e_h2d, e_comp, e_d2h = sl.ev
        cu.wait(cs_h, e_comp)          # step i-2 is done with this slot's input
        cu.h2d(sl.dst_in, host_rows[ci][t], sl.nin, cs_h)
        cu.record(e_h2d, cs_h)
        cu.wait(main_h, e_h2d)
        cu.wait(main_h, e_d2h)         # step i-2's result has left this slot
        sl.plans[ci].step(sl.dq, sl.dk, sl.dv)
        cu.record(e_comp, main_h)
        cu.wait(out_h, e_comp)
        cu.d2h(sl.hres_ptr, sl.src_res, sl.nres, out_h)
        cu.record(e_d2h, out_h)

    def e2e_timed(count):
        total = 0.0
        done = 0
        while done < count:
            first, m = take(count - done)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            t0.record(main)
            for i in range(first, first + m):
                e2e_step(i)
            main.wait_stream(cs_out)  # the last result is on the host
            t1.record(main)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            total += t0.elapsed_time(t1)
            done += m
        return total

    en = min(n, 512)
    e2e_timed(min(en, ncopy))  # warm
    e2e_us = 1e3 * e2e_timed(en) / en
    dstage, hres = slots[0].dstage, slots[0].hres
    h2d = dstage.numel() * 2
    d2h = hres.numel()

    # ---- max over ranks
    def rmax(x):
        return replicas.max_over_ranks(x, world, dev)

    mean_step = rmax(mean_step)
    dec_us = rmax(dec_us)
    e2e_us = rmax(e2e_us)
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return

    peak, peak_kind = peaks()
    step_bytes = dec_bytes + append_bytes(1, w.num_kv_heads)
    achieved = dec_bytes / (dec_us * 1e-6) / 1e9
    taken = PATH_NAMES[q.decode_path(cache, K, opts_main)]
    traffic = profiled_traffic(taken)
    fl = sorted(flushed_us)
    line = {
        "metric": METRIC, "value": round(mean_step, 3), "unit": "us/step", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(mean_step / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) fp16 K/V, 4 key channels x8, 8 planted needles/head)",
        "config": {**w.describe(), "storage": "fp16 K/V/q/out, fp32 arithmetic",
                   "l2": f"inputs larger than L2: {ncopy} independent copies of the workload "
                         f"({ncopy * (w.k_pool.numel() * 4 + cache.meta.numel() * 2) / 1e9:.1f} GB) "
                         "taken in rotation, so each call's boxes and pages were evicted by the "
                         "other copies' calls; calls back to back, one event pair around the "
                         "timed steps",
                   "step": "quest_decode_step: append + score + top-K + split-K decode",
                   "decode_path": taken + (" (library's choice)" if args.path == "auto" else
                                           " (forced)"),
                   "replicas": world},
        "gbs": round(replicas.job_bytes_per_second(step_bytes, world, mean_step * 1e-6) / 1e9, 1),
        "roofline": {"bound": "hbm",
                     "kernel": {"chain": "quest_decode, chain: estimate_kernel + " +
                                         ("decode_kernel (top-K in every decode work item)"
                                          if q.decode_launches(cache, K, opts_main) == 2 else
                                          "topk_kernel + decode_kernel"),
                                "fused": "quest_decode, one launch: cluster_kernel",
                                "stream": "quest_decode, one launch: stream_kernel"}[taken],
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "frac_of_nominal_8tbs": round(achieved / 8000.0, 4),
                     "algorithmic_bytes": dec_bytes, "launch_us": round(dec_us, 3),
                     "traffic": traffic},
        "e2e": {"value": round(e2e_us, 3), "unit": "us/step", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": n * q.decode_launches(cache, K, opts_main),
        "clocks": clk.summary(),
        "detail_us": {"step_mean": round(mean_step, 3),
                      "step_l2_flushed_mean": round(sum(fl) / len(fl), 3),
                      "step_l2_flushed_p50": round(statistics.median(fl), 3),
                      "step_l2_flushed_p90": round(fl[int(0.9 * (len(fl) - 1))], 3),
                      "step_l2_flushed_max": round(fl[-1], 3),
                      "quest_decode": round(dec_us, 3),
                      "quest_decode_l2_flushed": round(dec_flushed_us, 3),
                      "quest_decode_l2_warm_one_copy": round(dec_warm_us, 3),
                      "unfused_chain_l2_flushed": round(chain_us, 3),
                      "dense_decode_l2_flushed": round(dense_us, 3),
                      "host_issue_per_step": round(host_issue_us, 3),
                      "build_meta": round(build_meta_us, 3),
                      "timed_wall_s": round(wall, 3)},
    }
    if not args.no_cpu_baseline:
        us, k = oracle_timing(w, budget_s=args.cpu_seconds, max_steps=w.steps)
        line["cpu_baseline"] = {
            "value": round(us, 1), "unit": "us/step", "cores": 1, "kind": "oracle",
            "sample": f"{k} decode steps (append + score + top-K + attend) of the same "
                      f"workload, single-threaded C oracle"}
        us_all, k_all, threads = oracle_timing_all_cores(w, budget_s=min(10.0, args.cpu_seconds))
        line["cpu_baseline_all_cores"] = {
            "value": round(us_all, 1), "unit": "us/step", "cores": threads, "kind": "oracle",
            "sample": f"{k_all} score + top-K + attend steps at the prefill context, one "
                      f"thread per host core, time per step at full occupancy"}
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """quest_decode (fused, kernel only), the unfused estimate + top-K + sparse-decode chain,
    quest_append and quest_dense_decode on every workload, L2 flushed before each timed
    launch; one JSON line per workload (not the benchmark's contract line)."""
    import torch

    import query_aware_kv_gb300 as q
    from query_aware_kv_gb300 import build as cuda_build
    from query_aware_kv_gb300 import workloads as wl

    cuda_build.build()
    q.load()
    dev = torch.device("cuda")
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sum = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        flush_buf.zero_()
        torch.sum(flush_buf[: FLUSH_BYTES // 2].view(torch.int64), dim=0, out=flush_sum)

    def timed(fn, reps):
        es = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for _ in range(3):
            fn()
        for a, b in es:
            flush_l2()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sum(1e3 * a.elapsed_time(b) for a, b in es) / reps

    peak, _ = peaks()
    cases = [("tiny", lambda: wl.tiny(seed=0, device=dev))]
    cases.append(("longchat_32k", lambda: wl.longchat_32k(seed=0, device=dev, steps=4)))
    for budget in (256, 512, 1024, 2048, 4096):
        cases.append((f"batched_ragged_budget{budget}",
                      lambda budget=budget: wl.batched_ragged(seed=0, device=dev, budget=budget,
                                                              steps=1)))
    for budget in (1024, 2048):
        cases.append((f"yarn_128k_layer0_budget{budget}",
                      lambda budget=budget: wl.yarn_128k_layer(0, seed=0, device=dev,
                                                               budget=budget)))
    for page in (16, 32):
        cases.append((f"gqa_llama31_p{page}",
                      lambda page=page: wl.gqa_llama31(seed=0, device=dev, page_size=page)))
    for name, make in cases:
        w = make()
        cache = q.PagedCache.allocate_meta(w.k_pool, w.v_pool, w.block_table, w.seq_lens.clone(),
                                           w.num_q_heads)
        K = w.top_k
        ws = q.workspace(cache, K)
        q.build_meta(cache, ws)
        B, Hq, Hkv, P = w.batch, w.num_q_heads, w.num_kv_heads, w.page_size
        out = torch.empty((B, Hq, 128), dtype=torch.float16, device=dev)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        idx = torch.empty((B, Hkv, K), dtype=torch.int32, device=dev)
        cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
        qv = w.q[0]
        reps = 64 if name != "tiny" else 256
        o = q.opts(cluster_size=args.cluster_size, path=q.QUEST_PATH_FUSED)
        fused = timed(lambda: q.decode(cache, qv, K, ws, o, out=out, lse=lse, idx_out=idx,
                                       count_out=cnt), reps)
        # the library's own choice between the one-launch kernel and the chain
        auto_us = timed(lambda: q.decode(cache, qv, K, ws, None, out=out, lse=lse, idx_out=idx,
                                         count_out=cnt), reps)
        # the chain forced, and the stream kernel where its shape fits
        oc = q.opts(path=q.QUEST_PATH_CHAIN)
        chain_path_us = timed(lambda: q.decode(cache, qv, K, ws, oc, out=out, lse=lse), reps)
        os_ = q.opts(path=q.QUEST_PATH_STREAM)
        try:
            q.decode_path(cache, K, os_)
            stream_us = round(timed(lambda: q.decode(cache, qv, K, ws, os_, out=out, lse=lse),
                                    reps), 2)
        except q.QuestError:
            stream_us = None
        L = [int(x) for x in cache.seq_lens.cpu().tolist()]
        tok = selected_tokens(idx, cnt, L, P)
        nbytes = decode_bytes(L, tok, B, Hq, Hkv, page=P)
        scores = torch.empty((B, Hkv, cache.max_pages), dtype=torch.float32, device=dev)

        def chain():
            q.estimate(cache, qv, ws, scores=scores)
            i2, c2 = q.topk(cache, scores, K, ws)
            q.sparse_decode(cache, qv, i2, c2, K, ws, out=out, lse=lse)

        chain_us = timed(chain, reps)
        union = {}
        G = Hq // Hkv
        if G > 1:
            # the union form of the group-level selection: per-head bounds, each head's top-K,
            # their union (rows of G*K), sparse decode over it
            cap = min(G * K, cache.max_pages)
            ws_u = q.workspace(cache, cap)
            sh = torch.empty((B, Hq, cache.max_pages), dtype=torch.float32, device=dev)
            ou = q.opts(gqa_union=True)
            iu, cu = q.topk(cache, q.estimate_heads(cache, qv, ws_u, scores=sh), K, ws_u, ou)

            def union_chain():
                q.estimate_heads(cache, qv, ws_u, scores=sh)
                i3, c3 = q.topk(cache, sh, K, ws_u, ou)
                q.sparse_decode(cache, qv, i3, c3, cap, ws_u, out=out, lse=lse)

            u_us = timed(union_chain, reps)
            u_tok = selected_tokens(iu, cu, L, P)
            u_bytes = decode_bytes(L, u_tok, B, Hq, Hkv, page=P)
            union = {"union_chain_us": round(u_us, 2), "union_pages_mean":
                     round(float(cu.float().mean()), 1), "union_algorithmic_bytes": u_bytes,
                     "union_gbs": round(u_bytes / (u_us * 1e-6) / 1e9, 1)}
        dense_us = timed(lambda: q.dense_decode(cache, qv, ws, out=out, lse=lse), max(8, reps // 4))
        snap_meta, snap_len = cache.meta.clone(), cache.seq_lens.clone()

        def append_once():
            q.append(cache, w.k_new[0], w.v_new[0], ws)
            cache.seq_lens.copy_(snap_len)

        append_us = timed(append_once, reps)
        cache.meta.copy_(snap_meta)
        rc, detail = q.read_status(ws)
        gbs = nbytes / (fused * 1e-6) / 1e9
        print(json.dumps({
            "workload": name, "cluster_size": args.cluster_size, "batch": B, "num_q_heads": Hq,
            "num_kv_heads": Hkv,
            "page_size": P, "top_k_pages": K, "seq_lens_mean": round(sum(L) / len(L), 1),
            "quest_decode_us": round(fused, 2), "quest_decode_auto_us": round(auto_us, 2),
            "quest_decode_chain_us": round(chain_path_us, 2), "quest_decode_stream_us": stream_us,
            "algorithmic_bytes": nbytes,
            "gbs": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
            "frac_of_nominal_8tbs": round(gbs / 8000.0, 4),
            "unfused_chain_us": round(chain_us, 2), "append_plus_len_reset_us": round(append_us, 2),
            "dense_decode_us": round(dense_us, 2), "status": rc, **union}), flush=True)
        del w, cache, ws, scores
        torch.cuda.empty_cache()


def prefill_bytes(batch, n, num_kv_heads, page, first_lens):
    """Algorithmic bytes of one quest_prefill: the chunk's K and V read once and written once,
    and the box of every page the chunk touches written (read too when it was partial)."""
    rows = 2 * batch * n * num_kv_heads * 256
    boxes = 0
    for L in first_lens:
        touched = (L + n - 1) // page - L // page + 1
        boxes += touched * num_kv_heads * 512 + (num_kv_heads * 512 if L % page else 0)
    return 2 * rows + boxes


def run_prefill(args):
    """quest_prefill on the 32K-context MHA geometry (1 x 32 heads, page 16) and the GQA
    geometry (4 x 8 kv heads, page 16): chunks of 512, 4096 and 32768 tokens from an empty
    cache, and a 32K prompt written with a torch scatter + quest_build_meta for comparison;
    L2 flushed before each timed launch; one JSON line per case."""
    import torch

    import query_aware_kv_gb300 as q
    from query_aware_kv_gb300 import build as cuda_build

    cuda_build.build()
    q.load()
    dev = torch.device("cuda")
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sum = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        flush_buf.zero_()
        torch.sum(flush_buf[: FLUSH_BYTES // 2].view(torch.int64), dim=0, out=flush_sum)

    def timed(reset, fn, reps):
        es = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for _ in range(3):
            reset()
            fn()
        for a, b in es:
            reset()
            flush_l2()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sum(1e3 * a.elapsed_time(b) for a, b in es) / reps

    peak, _ = peaks()
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    for name, B, Hq, Hkv in (("longchat_32k_mha", 1, 32, 32), ("llama31_gqa", 4, 32, 8)):
        P, total = 16, 32768
        pages = total // P
        num_phys = B * pages
        k_pool = torch.empty((num_phys, Hkv, P, 128), dtype=torch.float16, device=dev)
        v_pool = torch.empty_like(k_pool)
        bt = torch.randperm(num_phys, generator=gen, device=dev).to(torch.int32).view(B, pages)
        lens = torch.zeros(B, dtype=torch.int32, device=dev)
        cache = q.PagedCache.allocate_meta(k_pool, v_pool, bt, lens, Hq)
        ws = q.workspace(cache, 64)
        for n in (512, 4096, 32768):
            kc = torch.randn((B, n, Hkv, 128), generator=gen, device=dev).to(torch.float16)
            vc = torch.randn((B, n, Hkv, 128), generator=gen, device=dev).to(torch.float16)
            us = timed(lambda: lens.zero_(),
                       lambda: q.prefill(cache, kc, vc, ws), 32 if n < 32768 else 8)
            nbytes = prefill_bytes(B, n, Hkv, P, [0] * B)
            rec = {"workload": name, "batch": B, "num_kv_heads": Hkv, "page_size": P,
                   "chunk_tokens": n, "quest_prefill_us": round(us, 2), "algorithmic_bytes": nbytes,
                   "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                   "frac_of_measured": round(nbytes / (us * 1e-6) / 1e9 / peak, 4)}
            if n == total:
                fused_meta = cache.meta.clone()
                # the same prompt written without the fused boxes: scatter into the pages,
                # then a box pass that reads every key again
                flat = bt.view(-1).long()

                def scatter():
                    k_pool[flat] = kc.view(B, pages, P, Hkv, 128).permute(0, 1, 3, 2, 4) \
                        .reshape(-1, Hkv, P, 128)
                    v_pool[flat] = vc.view(B, pages, P, Hkv, 128).permute(0, 1, 3, 2, 4) \
                        .reshape(-1, Hkv, P, 128)

                def unfused():
                    scatter()
                    lens.fill_(total)
                    q.build_meta(cache, ws)

                rec["scatter_plus_build_meta_us"] = round(timed(lambda: None, unfused, 8), 2)
                rec["boxes_equal_build_meta"] = bool(torch.equal(
                    fused_meta.view(torch.int16), cache.meta.view(torch.int16)))
            rc, _ = q.read_status(ws)
            rec["status"] = rc
            print(json.dumps(rec), flush=True)
        del cache, k_pool, v_pool, kc, vc
        torch.cuda.empty_cache()


def run_layers(args):
    """All 32 layers of the 128K-context model in one quest_decode_layers launch against 32
    quest_decode calls (automatic path, and forced to the one-launch kernel), L2 flushed
    before each timed step; one JSON line."""
    import torch

    import query_aware_kv_gb300 as q
    from query_aware_kv_gb300 import build as cuda_build
    from query_aware_kv_gb300 import workloads as wl

    cuda_build.build()
    q.load()
    dev = torch.device("cuda")
    n_layers = 32
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sum = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        flush_buf.zero_()
        torch.sum(flush_buf[: FLUSH_BYTES // 2].view(torch.int64), dim=0, out=flush_sum)

    ws_ = [wl.yarn_128k_layer(i, seed=0, device=dev, budget=2048) for i in range(n_layers)]
    w0 = ws_[0]
    K = w0.top_k
    base = q.PagedCache.allocate_meta(w0.k_pool, w0.v_pool, w0.block_table, w0.seq_lens.clone(),
                                      w0.num_q_heads)
    layers = [base] + [q.PagedCache.allocate_meta(w.k_pool, w.v_pool, base.block_table,
                                                   base.seq_lens, w.num_q_heads) for w in ws_[1:]]
    ws = q.workspace(base, K)
    for lay in layers:
        q.build_meta(lay, ws)
    qs = [w.q[0] for w in ws_]
    outs = [torch.empty((1, 32, 128), dtype=torch.float16, device=dev) for _ in range(n_layers)]
    lses = [torch.empty((1, 32), dtype=torch.float32, device=dev) for _ in range(n_layers)]

    o = q.opts(cluster_size=args.cluster_size)
    o_fused = q.opts(cluster_size=args.cluster_size, path=q.QUEST_PATH_FUSED)

    def one_launch():
        q.decode_layers(base, layers, qs, K, ws, o, out=outs, lse=lses)

    def one_launch_kernel():
        q.decode_layers(base, layers, qs, K, ws, o_fused, out=outs, lse=lses)

    def per_layer():
        for i, lay in enumerate(layers):
            q.decode(lay, qs[i], K, ws, o, out=outs[i], lse=lses[i])

    def per_layer_fused():
        for i, lay in enumerate(layers):
            q.decode(lay, qs[i], K, ws, o_fused, out=outs[i], lse=lses[i])

    def timed(fn, reps=16):
        es = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for _ in range(3):
            fn()
        for a, b in es:
            flush_l2()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sum(1e3 * a.elapsed_time(b) for a, b in es) / reps

    fused_us = timed(one_launch)
    per_us = timed(per_layer)
    per_fused_us = timed(per_layer_fused)
    one_kernel_us = timed(one_launch_kernel)
    rc, _ = q.read_status(ws)
    L = int(base.seq_lens[0])
    nbytes = n_layers * decode_bytes([L], 32 * K * PAGE, 1, 32, 32)
    peak, _ = peaks()
    gbs = nbytes / (fused_us * 1e-6) / 1e9
    print(json.dumps({"workload": "yarn_128k_32_layers_budget2048", "layers": n_layers,
                      "cluster_size": args.cluster_size,
                      "decode_layers_us": round(fused_us, 1),
                      "decode_layers_one_launch_kernel_us": round(one_kernel_us, 1),
                      "decode_per_layer_launches_us": round(per_us, 1),
                      "decode_per_layer_one_launch_kernel_us": round(per_fused_us, 1),
                      "algorithmic_bytes": nbytes, "gbs": round(gbs, 1),
                      "frac_of_measured": round(gbs / peak, 4), "status": rc}), flush=True)


def profiled_traffic(path: str):
    """DRAM bytes per quest_decode call on the bench workload, for the path it took, from
    the committed ncu summaries, if they were taken on the current kernel sources (else
    null)."""
    try:
        import hashlib
        with open(os.path.join(ROOT, "profiles", "quest_decode_traffic.json")) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        csrc = os.path.join(ROOT, "query_aware_kv_gb300", "csrc")
        for name in sorted(os.listdir(csrc)):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
        if rec.get("csrc_sha256") != h.hexdigest():
            return None
        return rec[path]["dram_bytes_per_launch_full_workload"]
    except Exception:
        return None


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    elif args.layers:
        run_layers(args)
    elif args.prefill:
        run_prefill(args)
    else:
        run_quest(args)


if __name__ == "__main__":
    main()

"""Benchmark of the tree speculative-decoding verify step on GB300.

One step = tv_build_ancestors -> tv_tree_attention -> tv_argmax -> tv_tree_walk
-> tv_commit_kv over one batch of the throughput-stress workload (64 sequences
x 16384 context tokens, N=32 random trees of depth <= 8, 32 query / 8 KV heads,
head dim 128, bf16, 16-token blocks behind shuffled block tables, bf16 logits
over a 151936-token vocabulary).  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (fp64, OpenMP over the host cores) on a
bounded sample of sequences of the same workload, scaled to whole steps.
Multi-GPU runs (torchrun) are independent replicas: every rank verifies its
own batch, no collective touches the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("tree-verify steps/s and attention KV GB/s (% of GB300 HBM peak), "
          "bit-exact walk")
HBM_FALLBACK_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "tv_tree_attention_stress_traffic.txt")
ATTN_SOURCES = [os.path.join(ROOT, "tree_speculative_decoding_build_gb300", "csrc", f)
                for f in ("attention.cu", "attention_tc.cu", "attention.cuh")]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stress")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="only the workload's own measurements (no overlapped, draft or graph lines)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (smaller cases for profiling)")
    ap.add_argument("--path", choices=["verify", "draft", "graph", "gdn"], default="verify",
                    help="verify: the verify step (default); draft: draft-tree construction; "
                         "graph: the multi-layer step, eager launches vs one CUDA-graph replay; "
                         "gdn: tree verification through a Gated DeltaNet layer + state commit")
    ap.add_argument("--layers", type=int, default=8, help="attention layers for --path graph")
    ap.add_argument("--draft-workload", default="tree_build")
    ap.add_argument("--window-left", type=int, default=None,
                    help="override the workload's sliding window (-1: global attention)")
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(name, rank):
    """Each rank verifies its own batch: the workload's seed offset by the rank."""
    import workloads
    return workloads.get(name).seed + rank


E2E_PASSES = 3  # timed passes of the end-to-end loop; the median is reported


def pipelined_e2e(step, host, bufs, results, E, stream, dev, copy_streams=4, passes=1):
    """Milliseconds per step, end to end: every step uploads its inputs from pinned
    host memory, runs, and reads its results back, inside the timed region.  The
    device inputs are double-buffered, so step s+1's upload (on copy streams, big
    tensors cut into one chunk per stream to use several copy engines) overlaps
    step s; an upload waits until the step that last used its buffer is done.
    The timed region (E steps) runs ``passes`` times and the median is returned,
    so that one transient on a shared host does not decide the figure."""
    import torch
    css = [torch.cuda.Stream(device=dev) for _ in range(copy_streams)]
    up = [[torch.cuda.Event() for _ in css] for _ in bufs]
    used = [torch.cuda.Event() for _ in bufs]

    def upload(b, after):
        for cs in css:
            cs.wait_event(after)
        j = 0
        for k, src in host.items():
            dst = bufs[b][k]
            nbytes = src.numel() * src.element_size()
            if nbytes >= (64 << 20):
                flat_s, flat_d = src.view(-1), dst.view(-1)
                n = flat_s.numel()
                for c, cs in enumerate(css):
                    lo, hi = n * c // len(css), n * (c + 1) // len(css)
                    with torch.cuda.stream(cs):
                        flat_d[lo:hi].copy_(flat_s[lo:hi], non_blocking=True)
            else:
                with torch.cuda.stream(css[j % len(css)]):
                    dst.copy_(src, non_blocking=True)
                j += 1
        for cs, ev in zip(css, up[b]):
            ev.record(cs)

    def compute(b):
        for ev in up[b]:
            stream.wait_event(ev)
        step(bufs[b])
        for dst, src in results:
            dst.copy_(src, non_blocking=True)
        used[b].record(stream)

    def run(steps, e_start):
        upload(0, e_start)
        for s in range(steps):
            nb = (s + 1) % len(bufs)
            if s + 1 < steps:
                upload(nb, used[nb] if s + 1 >= len(bufs) else e_start)
            compute(s % len(bufs))

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(2, e0)  # warm-up
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(max(1, passes)):
        e0.record(stream)
        run(E, e0)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1) / E)
    return sorted(times)[len(times) // 2]


def max_over_ranks(x, world, device):
    """The largest of every rank's ``x`` (a time), on every rank."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, steps, ms):
    """Whole-job steps/s: every rank ran ``steps`` steps, the slowest took ``ms``."""
    return world * steps / (ms * 1e-3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def source_digest():
    h = hashlib.sha256()
    for p in ATTN_SOURCES:
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload="stress", batch=None, window_left=None):
    """dram read+write bytes per launch from the committed ncu summary, or None
    when it is missing, was taken on a different attention source, or the run
    is not the stress workload it describes (64 sequences, global window)."""
    if workload != "stress" or batch not in (None, 64) or window_left not in (None, -1):
        return None
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha") != source_digest():
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every ``period_ms`` from a
    background thread.  Every sample carries the host time it arrived, so any
    window of the run (the whole measurement, the timed loop, the sustained
    loop) can be summarised afterwards."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index, period_ms=100):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.samples = []   # (host time, sm MHz, max MHz, power W, set of active reasons)
        self.proc = None

    def start(self, timeout=5.0):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < timeout:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                pw = float(parts[3])
            except ValueError:
                pw = None
            active = {n for n, v in zip(self.REASONS, parts[5:9]) if v.lower() == "active"}
            self.samples.append((time.time(), sm, mx, pw, active))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summary(self, t0, t1, window):
        """Median SM clock, the maximum, the samples and every throttle reason
        seen between host times t0 and t1 (widened by one sampling period on
        each side when no sample fell inside)."""
        sel = [s for s in list(self.samples) if t0 <= s[0] <= t1]
        if not sel:
            pad = self.period_ms / 1000.0
            sel = [s for s in list(self.samples) if t0 - pad <= s[0] <= t1 + pad]
        if not sel:
            return None
        sm = sorted(s[1] for s in sel)
        pw = [s[3] for s in sel if s[3] is not None]
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(s[2] for s in sel),
                "samples": len(sel), "reasons": sorted(set().union(*(s[4] for s in sel))),
                "power_w_max": max(pw) if pw else None, "window": window,
                "window_s": round(t1 - t0, 3)}


def l2_bytes(dev):
    import torch
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        return 126 << 20


class L2Flush:
    """A read of twice the L2 size: nothing a timed launch reads stays cached.
    A read rather than a write, so that no dirty lines are left for the timed
    launch to write back."""

    def __init__(self, dev):
        import torch
        self.buf = torch.ones(2 * l2_bytes(dev) // 4, dtype=torch.int32, device=dev)
        self.out = torch.empty((), dtype=torch.int32, device=dev)

    def __call__(self):
        import torch
        torch.amax(self.buf, dim=0, out=self.out)


def capture(fn, reps, dev):
    """A CUDA graph holding ``reps`` calls of fn() (the library's calls enqueue on
    the current stream, which is the capture stream here)."""
    import torch
    fn()  # first call outside capture: one-time host set-up (function attributes)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        for _ in range(reps):
            fn()
    torch.cuda.synchronize(dev)
    return g


def graph_device_ms(fn, dev, iters, flush=None, reps=1):
    """Device milliseconds per fn() call, from CUDA-graph replays timed with
    CUDA events on the replay stream.  With ``flush`` every replay (one call)
    is preceded by an L2 flush outside its event pair, and the events are
    enqueued while the flush runs, so the GPU never waits on the host inside
    a pair; without, ``reps`` calls are captured into one graph and replayed
    back to back."""
    import torch
    stream = torch.cuda.current_stream(dev)
    g = capture(fn, 1 if flush else reps, dev)
    for _ in range(3):
        if flush:
            flush()
        g.replay()
    torch.cuda.synchronize(dev)
    if flush:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        for e0, e1 in evs:
            flush()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / iters
    else:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / (iters * reps)
    del g
    return ms


def h2d_link(nbytes, dev, streams=4, reps=5):
    """Host-to-device copy rate from pinned memory for an upload of ``nbytes``:
    one cudaMemcpyAsync, and the same bytes cut into one chunk per copy stream."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    css = [torch.cuda.Stream(device=dev) for _ in range(streams)]

    def one():
        dst.copy_(src, non_blocking=True)

    def chunked():
        done = []
        for c, cs in enumerate(css):
            cs.wait_stream(stream)
            lo, hi = nbytes * c // streams, nbytes * (c + 1) // streams
            with torch.cuda.stream(cs):
                dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(cs)
            done.append(ev)
        for ev in done:
            stream.wait_event(ev)

    out = {}
    for name, fn in (("single_copy_gbs", one), (f"{streams}_streams_gbs", chunked)):
        fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        out[name] = nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    return out


def workload_config(name, B=None, window_left=None, l2=None):
    """The workload, described from its specification (both arms use this);
    ``l2`` is the line's statement of how L2 was handled between timed steps."""
    import workloads
    w = workloads.get(name)
    B = w.B if B is None else B
    if window_left is not None:
        w = dataclasses.replace(w, window_left=window_left)
    ctx = f"{w.ctx[0]}..{w.ctx[1]}" if isinstance(w.ctx, tuple) else str(w.ctx)
    return {
        "workload": (f"{name}: B={B} ctx={ctx} N={w.N} Hq/Hkv/D={w.Hq}/{w.Hkv}/{w.D} bf16 KV, "
                     f"block 16{', shuffled block tables' if w.shuffle_blocks else ''}, "
                     f"V={w.V} {w.logits_dtype} logits"),
        "batch": B, "tree_nodes": w.N, "ctx_len": ctx, "window_left": w.window_left,
        "l2": l2,
    }


def attention_algorithmic_bytes(inp):
    import workloads
    B, N, Hq, Hkv, D = inp["B"], inp["N"], inp["Hq"], inp["Hkv"], inp["D"]
    kv = workloads.kv_bytes(inp)
    q = B * N * Hq * D * 2
    tree_kv = 2 * B * N * Hkv * D * 2
    out = B * N * Hq * D * 2
    ctx = inp["ctx_len"].cpu().numpy()
    table = int(sum((int(c) + 15) // 16 for c in ctx)) * 4
    return kv + q + tree_kv + out + table


def step_working_set(inp, alg):
    """Bytes one verify step reads from memory: the attention's algorithmic
    bytes plus the logits (the rest is a few MB at most)."""
    return alg + inp["logits"].numel() * inp["logits"].element_size()


def bench_ours(args, rank, world, local):
    import math
    import torch
    import torch.distributed as dist
    import workloads
    import tree_speculative_decoding_build_gb300 as tv

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    if rank == 0:
        sampler.start()
    t_run0 = time.time()
    inp = workloads.make(args.workload, dev, seed=rank_seed(args.workload, rank), B=args.batch,
                         window_left=args.window_left)
    step = tv.VerifyStep(inp["B"], inp["N"], inp["Hq"], inp["Hkv"], inp["D"], inp["V"],
                         inp["max_blocks"], window_left=inp["window_left"],
                         logits_dtype=inp["logits_dtype"], device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        step(inp)
    torch.cuda.synchronize(dev)
    eager_ms = None
    if rank == 0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            step(inp)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        eager_ms = e0.elapsed_time(e1) / 5

    # kernels launched per step: fixed by the launch plan
    ws_attn = tv.tv_tree_attention_workspace_size(inp["B"], inp["N"], inp["Hq"], inp["Hkv"],
                                                  inp["D"], inp["max_blocks"], inp["window_left"])
    dt = tv.TV_F32 if inp["logits_dtype"] == "f32" else tv.TV_BF16
    ws_arg = tv.tv_argmax_workspace_size(inp["B"] * inp["N"], inp["V"], dt)
    launches_per_step = 5 + (1 if ws_attn else 0) + (1 if ws_arg else 0)
    alg = attention_algorithmic_bytes(inp)
    l2 = l2_bytes(dev)
    ws_bytes = step_working_set(inp, alg)
    flush = L2Flush(dev)
    per_step_flush = ws_bytes <= 2 * l2

    # the timed region: K replays of a CUDA graph holding one whole verify step
    # (the same five calls through the binding); back to back when a step reads
    # more than twice the L2, else each replay after an L2 flush
    K = args.steps
    g_step = capture(lambda: step(inp), 1, dev)
    for _ in range(3):
        g_step.replay()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_loop0 = time.time()
    if per_step_flush:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for e0, e1 in evs:
            flush()
            e0.record(stream)
            g_step.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    else:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(K):
            g_step.replay()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        ms = t0.elapsed_time(t1)
    t_loop1 = time.time()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ms, world, dev)
    status_ok = bool((step.out.status == 0).all().item())

    # sustained: the same replays for at least a second, with their own clock record
    n_sus = max(1, int(math.ceil(1250.0 / max(ms / K, 1e-3))))
    t_sus0 = time.time()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(n_sus):
        if per_step_flush:
            flush()
        g_step.replay()
    s1.record(stream)
    torch.cuda.synchronize(dev)
    t_sus1 = time.time()
    sus_ms = s0.elapsed_time(s1) / n_sus
    del g_step

    # tv_tree_attention alone (its two launches), L2 flushed before every launch
    o = step.out

    def attn():
        tv.tv_tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"],
                             inp["v_cache"], inp["block_table"], inp["ctx_len"], o.pos, o.anc,
                             o.attn, o.status, window_left=inp["window_left"],
                             workspace=step.ws_attn)
    attn_iters = max(20, min(K, 300))
    attn_ms = graph_device_ms(attn, dev, attn_iters, flush=flush)
    attn_warm_ms = graph_device_ms(attn, dev, max(5, attn_iters // 10), reps=10)

    # end to end through the public API: pinned host inputs in, tokens out
    host_keys = ["tokens", "parent", "depth", "ctx_len", "root_pred", "block_table", "q",
                 "k_tree", "v_tree", "logits"]
    host = {k: inp[k].cpu().pin_memory() for k in host_keys}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    res_keys = ["out_tokens", "n_emit", "n_acc", "ctx_len_out"]
    res_host = {k: torch.empty_like(getattr(o, k), device="cpu").pin_memory() for k in res_keys}
    d2h = sum(v.numel() * v.element_size() for v in res_host.values())
    bufs = [dict(inp)] + [dict(inp, **{k: torch.empty_like(inp[k]) for k in host_keys})]
    results = [(res_host[k], getattr(o, k)) for k in res_keys]
    e2e_ms = pipelined_e2e(lambda d: step(d), host, bufs, results, max(1, args.e2e_steps),
                           stream, dev, passes=E2E_PASSES)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    link = h2d_link(h2d, dev) if rank == 0 else None
    t_run1 = time.time()

    if rank != 0:
        return None
    sampler.stop()
    peak, peak_kind = peaks()
    achieved = alg / (attn_ms * 1e-3) / 1e9
    l2_note = (f"{'every replay after an L2 flush: ' if per_step_flush else ''}"
               f"a step reads {ws_bytes / 1e6:.0f} MB (attention {alg / 1e6:.0f} MB + logits), "
               f"L2 {l2 / 1e6:.0f} MB; the attention roofline launches each follow an L2 flush")
    e2e_value = job_throughput(world, 1, e2e_ms)
    link_peak = max(link.values()) if link else None
    line = {
        "metric": METRIC,
        "value": job_throughput(world, K, ms),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "impl": "ours",
        "config": workload_config(args.workload, args.batch, args.window_left, l2=l2_note),
        "timing": ("device: CUDA events around CUDA-graph replays of one whole verify step "
                   "(tv_build_ancestors, tv_tree_attention, tv_argmax, tv_tree_walk, "
                   "tv_commit_kv through the binding)"),
        "eager_ms_per_step": eager_ms,
        "attention": {"ms": attn_ms, "warm_ms": attn_warm_ms, "kv_gbs": achieved,
                      "algorithmic_bytes": alg, "frac_of_8tbs_nominal": achieved / 8000.0,
                      "frac_of_peak": achieved / peak, "peak_kind": peak_kind,
                      "timing": (f"CUDA events around {attn_iters} graph replays of one "
                                 "tv_tree_attention call (its counter-clearing and attention "
                                 "kernels), each after an L2 flush; warm_ms: 10 calls per "
                                 "replay, back to back")},
        "roofline": {"kernel": "tv_tree_attention", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic(args.workload, args.batch, args.window_left),
                     "peak_source": peak_kind},
        "e2e": {"value": e2e_value, "unit": "steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "h2d_gbs": h2d * e2e_value / 1e9,
                "h2d_link": link,
                "frac_of_link": (h2d * e2e_value / 1e9) / link_peak if link_peak else None,
                "timing": (f"median of {E2E_PASSES} passes, each CUDA events around "
                           f"{max(1, args.e2e_steps)} pipelined steps through VerifyStep")},
        "gpu_launches": launches_per_step * K,
        "status_ok": status_ok,
        "clocks": sampler.summary(t_run0, t_run1, "whole measurement: warm-up, timed loop, "
                                  "sustained loop, attention and end-to-end timing"),
        "clocks_timed_loop": sampler.summary(t_loop0, t_loop1, "timed loop"),
        "sustained": {"ms_per_step": sus_ms, "steps_per_s": 1000.0 / sus_ms, "steps": n_sus,
                      "seconds": round(t_sus1 - t_sus0, 3),
                      "clocks": sampler.summary(t_sus0, t_sus1, "sustained loop")},
    }
    if world == 1 and not args.quick:
        # the same step with tv_argmax on 16 SMs beside the attention (two streams)
        line["overlapped_step"] = measure_overlap(args.workload, inp, min(K, 300), dev)
        # the draft-tree path (the step before verify), timed on its own
        d = measure_draft("tree_build", 50, 3, dev)
        d.pop("_inputs")
        d["top_w"] = measure_top_w(dev)
        line["draft_path"] = d
        # the multi-layer step as one CUDA-graph replay, on the small best-first batch
        line["graph_path"] = measure_graph("best_first", 8, 50, 3, dev)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=12.0,
                                            window_left=args.window_left)
    return line


def measure_overlap(name, inp, steps, dev, argmax_sms=16):
    """The verify step with tv_argmax_sm on `argmax_sms` SMs of a second stream
    beside tv_tree_attention on the others (VerifyStep(argmax_sms=...)):
    CUDA events on the main stream around `steps` steps."""
    import torch
    import tree_speculative_decoding_build_gb300 as tv
    step = tv.VerifyStep(inp["B"], inp["N"], inp["Hq"], inp["Hkv"], inp["D"], inp["V"],
                         inp["max_blocks"], window_left=inp["window_left"],
                         logits_dtype=inp["logits_dtype"], device=dev, argmax_sms=argmax_sms)
    stream = torch.cuda.current_stream(dev)
    for _ in range(5):
        step(inp)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step(inp)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    return {"argmax_sms": argmax_sms, "ms_per_step": ms, "steps_per_s": 1000.0 / ms,
            "status_ok": bool((step.out.status == 0).all().item())}


def cpu_baseline(name, budget_s=12.0, seqs_max=None, window_left=None):
    """The oracle, as it stands, on a bounded sample: whole verify steps for a
    few sequences at a time (all heads, all nodes), until the time budget is
    spent; scaled to whole-batch steps/s."""
    import numpy as np
    import torch
    import oracle
    import workloads
    w = workloads.get(name)
    oracle.build()
    done, spent = 0, 0.0
    B = w.B
    seqs_max = B if seqs_max is None else seqs_max
    b = 0
    while done < seqs_max and spent < budget_s:
        inp = workloads.make(name, "cpu", seed=w.seed + 7919 * (b + 1), B=1, window_left=window_left)
        npi = workloads.to_numpy(inp)
        t = time.perf_counter()
        oracle.verify_step(npi)
        spent += time.perf_counter() - t
        done += 1
        b += 1
    per_step = spent / done * B
    return {"value": 1.0 / per_step, "unit": "steps/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{done} of {B} sequences of the {name} workload, full verify step each "
                      f"(fp64 attention over all heads/nodes, argmax, walk, commit); "
                      f"{spent:.1f} s of oracle time scaled by {B}/{done}"}


DRAFT_METRIC = "draft-tree construction steps/s (tv_topk + tv_build_tree) and top-k GB/s"


def measure_draft(name, steps, warmup, dev, seed_offset=0, batch=None):
    """Time the draft path on one GPU: tv_topk over the per-position log-probs,
    then tv_build_tree; CUDA events on the launching stream around each."""
    import torch
    import workloads
    import tree_speculative_decoding_build_gb300 as tv
    w = workloads.DRAFT_WORKLOADS[name]
    B = w.B if batch is None else batch
    lp = workloads.make_draft(name, dev, seed=w.seed + seed_offset, B=B)
    dt = tv.DraftTree(B, w.L, w.V, w.K, w.budget, w.w, device=dev)
    o = dt.out
    stream = torch.cuda.current_stream(dev)
    x = lp.view(B * w.L, w.V)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        tv.tv_topk(x, w.K, o.cand_lp.view(B * w.L, w.K), o.cand_idx.view(B * w.L, w.K), dt.ws)
        if ev is not None:
            ev[1].record(stream)
        tv.tv_build_tree(o.cand_lp, o.cand_idx, w.budget, w.w, o.tokens, o.parent, o.depth,
                         o.score, o.n_nodes)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize(dev)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / steps
    topk_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    tree_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / steps
    topk_bytes = B * w.L * w.V * lp.element_size() + B * w.L * w.K * 8
    peak, peak_kind = peaks()
    gbs = topk_bytes / (topk_ms * 1e-3) / 1e9
    return {
        "workload": (f"{name}: B={B} L={w.L} V={w.V} fp32 log-probs, top_k={w.K}, "
                     f"budget={w.budget}, w={w.w}"),
        "ms_per_step": ms, "steps_per_s": 1000.0 / ms,
        "tv_topk": {"ms": topk_ms, "bytes": topk_bytes, "gbs": gbs, "frac_of_peak": gbs / peak,
                    "peak": peak, "peak_source": peak_kind},
        "tv_build_tree": {"us": tree_ms * 1000.0, "trees": B},
        "launches_per_step": 3 if tv.tv_topk_workspace_size(B * w.L, w.V, w.K, tv.TV_F32) else 2,
        "_inputs": (lp, o),
    }


def measure_top_w(dev, iters=200):
    """The leaf-sibling proposer's top-W emission on its own shape (4 spine
    positions x 262144-token vocabulary, W = 4, fp32 log-probabilities):
    tv_topk alone, timed by CUDA-graph replays, each after an L2 flush (cold)
    and back to back (its 4 MB stay in L2)."""
    import torch
    import workloads
    import tree_speculative_decoding_build_gb300 as tv
    w = workloads.DRAFT_WORKLOADS["top_w"]
    lp = workloads.make_draft("top_w", dev, B=w.B).view(w.B * w.L, w.V)
    vals = torch.empty(w.B * w.L, w.K, dtype=torch.float32, device=dev)
    idx = torch.empty(w.B * w.L, w.K, dtype=torch.int32, device=dev)
    need = tv.tv_topk_workspace_size(w.B * w.L, w.V, w.K, tv.TV_F32)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    fn = lambda: tv.tv_topk(lp, w.K, vals, idx, ws)
    cold = graph_device_ms(fn, dev, iters, flush=L2Flush(dev))
    warm = graph_device_ms(fn, dev, max(5, iters // 10), reps=10)
    nbytes = lp.numel() * lp.element_size() + vals.numel() * 8
    peak, peak_kind = peaks()
    return {"workload": f"top_w: {w.B * w.L} rows x V={w.V} fp32 log-probs, W={w.K}",
            "us": cold * 1000.0, "warm_us": warm * 1000.0, "bytes": nbytes,
            "gbs": nbytes / (cold * 1e-3) / 1e9, "frac_of_peak": nbytes / (cold * 1e-3) / 1e9 / peak,
            "peak_source": peak_kind,
            "timing": "CUDA-graph replays of one tv_topk call, each after an L2 flush; warm_us: "
                      "10 calls per replay, back to back"}


def draft_cpu_baseline(name, budget_s=10.0):
    """The oracle on a bounded sample of the draft workload: whole sequences
    (top-k of every position, then the construction) until the budget is spent."""
    import oracle
    import workloads
    from oracle import tree_build as tb
    w = workloads.DRAFT_WORKLOADS[name]
    done, spent = 0, 0.0
    while done < w.B and spent < budget_s:
        lp = workloads.make_draft(name, "cpu", seed=w.seed + 7919 * (done + 1), B=1).numpy()
        t = time.perf_counter()
        vals, idx = tb.topk(lp.reshape(w.L, w.V), w.K, "f32")
        tb.build_tree(vals.reshape(1, w.L, w.K), idx.reshape(1, w.L, w.K), w.budget, w.w)
        spent += time.perf_counter() - t
        done += 1
    return {"value": 1.0 / (spent / done * w.B), "unit": "steps/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {w.B} sequences of the {name} workload (numpy top-k + "
                      f"heap construction, one thread), scaled by {w.B}/{done}"}


def bench_draft(args, rank, world, local):
    """--path draft: one JSON line for the draft-tree construction path."""
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    r = measure_draft(args.draft_workload, args.steps, args.warmup, dev, seed_offset=rank,
                      batch=args.batch)
    ms = max_over_ranks(r["ms_per_step"], world, dev)
    lp, o = r.pop("_inputs")
    # end to end: pinned host log-probs in, trees out
    lp_host = lp.cpu().pin_memory()
    outs = [o.tokens, o.parent, o.depth, o.n_nodes]
    res_host = [torch.empty_like(t, device="cpu").pin_memory() for t in outs]
    import tree_speculative_decoding_build_gb300 as tv
    import workloads
    w = workloads.DRAFT_WORKLOADS[args.draft_workload]
    B = lp.shape[0]
    dt = tv.DraftTree(B, w.L, w.V, w.K, w.budget, w.w, device=dev)
    stream = torch.cuda.current_stream(dev)
    oo = dt(lp)  # the outputs live in fixed buffers
    results = list(zip(res_host, [oo.tokens, oo.parent, oo.depth, oo.n_nodes]))
    bufs = [{"lp": lp}, {"lp": torch.empty_like(lp)}]
    e2e_ms = pipelined_e2e(lambda d: dt(d["lp"]), {"lp": lp_host}, bufs, results,
                           max(1, args.e2e_steps), stream, dev, passes=E2E_PASSES)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    if rank != 0:
        return None
    line = {
        "metric": DRAFT_METRIC, "value": job_throughput(world, 1, ms), "unit": "steps/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "impl": "ours", "path": "draft",
        "config": {"workload": r["workload"], "batch": B,
                   "l2": (f"inputs larger than L2 ({r['tv_topk']['bytes'] / 1e6:.0f} MB of "
                          "log-probs per step)" if r["tv_topk"]["bytes"] > 129e6 else
                          f"inputs L2-resident ({r['tv_topk']['bytes'] / 1e6:.0f} MB of "
                          "log-probs per step, reused)")},
        "roofline": {"kernel": "tv_topk", "bound": "hbm", "achieved": r["tv_topk"]["gbs"],
                     "peak": r["tv_topk"]["peak"], "unit": "GB/s",
                     "frac": r["tv_topk"]["frac_of_peak"], "traffic": None,
                     "peak_source": r["tv_topk"]["peak_source"]},
        "tv_build_tree_us": r["tv_build_tree"]["us"],
        "top_w": measure_top_w(dev) if world == 1 else None,
        "e2e": {"value": job_throughput(world, 1, e2e_ms), "unit": "steps/s",
                "h2d_bytes_per_step": lp_host.numel() * lp_host.element_size(),
                "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h in res_host),
                "timing": (f"median of {E2E_PASSES} passes, each CUDA events around "
                           f"{max(1, args.e2e_steps)} pipelined steps through DraftTree")},
        "gpu_launches": r["launches_per_step"] * args.steps,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = draft_cpu_baseline(args.draft_workload)
    return line


GRAPH_METRIC = "multi-layer verify steps/s: one CUDA-graph replay vs eager launches"


def measure_graph(name, layers, steps, warmup, dev, batch=None, seed_offset=0):
    """The L-layer step (ModelStep) on one GPU: eager launches and graph
    replays, each timed with CUDA events over `steps` steps."""
    import torch
    import workloads
    import tree_speculative_decoding_build_gb300 as tv
    w = workloads.get(name)
    inp = workloads.make(name, dev, seed=w.seed + seed_offset, B=batch, plant="path")
    lys = workloads.make_layers(inp, layers, seed=w.seed + seed_offset)
    ms = tv.ModelStep(inp, lys, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(max(3, warmup)):
            fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps

    eager_ms = timed(lambda: ms.run())
    ms.capture()
    graph_ms = timed(lambda: ms.replay())
    launches = ms.launches
    ok = int(ms.out.status.abs().sum()) == 0
    ms.close()
    per_layer = attention_algorithmic_bytes(inp)
    return {
        "workload": (f"{name}: B={inp['B']} N={inp['N']} Hq/Hkv/D={inp['Hq']}/{inp['Hkv']}/"
                     f"{inp['D']}, {layers} layers (own q/k/v/caches each), V={inp['V']}"),
        "layers": layers, "eager_ms_per_step": eager_ms, "graph_ms_per_step": graph_ms,
        "graph_speedup": eager_ms / graph_ms, "launches_per_step": launches,
        "attention_bytes_per_step": per_layer * layers, "status_ok": ok,
    }


def bench_graph(args, rank, world, local):
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.workload
    r = measure_graph(name, args.layers, args.steps, args.warmup, dev, batch=args.batch,
                      seed_offset=rank)
    ms = max_over_ranks(r["graph_ms_per_step"], world, dev)
    if rank != 0:
        return None
    peak, peak_kind = peaks()
    gbs = r["attention_bytes_per_step"] / (ms * 1e-3) / 1e9
    return {
        "metric": GRAPH_METRIC, "value": job_throughput(world, 1, ms), "unit": "steps/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "impl": "ours", "path": "graph",
        "config": {"workload": r["workload"], "l2": "inputs larger than L2"},
        "eager": {"ms_per_step": r["eager_ms_per_step"], "value": 1000.0 / r["eager_ms_per_step"]},
        "graph_speedup": r["graph_speedup"],
        "roofline": {"kernel": "whole step (all layers)", "bound": "hbm", "achieved": gbs,
                     "peak": peak, "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                     "peak_source": peak_kind},
        "gpu_launches": r["launches_per_step"] * args.steps, "status_ok": r["status_ok"],
    }


GDN_METRIC = "GDN tree-verify steps/s (tv_gdn_tree_verify + tv_gdn_commit)"
FP32_FMA_LANES_PER_SM = 128   # fp32 FMA lanes per SM (4 partitions x 32)


def gdn_flops(x):
    """Algorithmic flops of one verification: K S_0 and Q S_0 (2 x N x dk x dv
    multiply-adds per value head), the ancestor-pair dot products, the solve and
    the output sums (2 x pairs x dv each)."""
    B, N, Hv, dk, dv = x["B"], x["N"], x["Hv"], x["dk"], x["dv"]
    pairs = int(x["depth"].sum().item())  # over all sequences: sum of |ancestors-or-self|
    return B * Hv * 2 * (2 * N * dk * dv) + Hv * (2 * (2 * pairs * dk) + 2 * (2 * pairs * dv))


def gdn_bytes(x):
    B, N, Hk, Hv, dk, dv = x["B"], x["N"], x["Hk"], x["Hv"], x["dk"], x["dv"]
    return (B * Hv * dv * dk * 4 + 2 * B * N * Hk * dk * 2 + B * N * Hv * dv * 2 + 2 * B * N * Hv * 4
            + 2 * B * N * Hv * dv * 4 + B * N * Hv * 4 + B * N * 8)


def measure_gdn(name, steps, warmup, dev, batch=None, seed_offset=0):
    import torch
    import workloads
    import tree_speculative_decoding_build_gb300 as tv
    w = workloads.GDN_WORKLOADS[name]
    x = workloads.make_gdn(name, dev, seed=w.seed + seed_offset, B=batch)
    B, N, Hv, dv = x["B"], x["N"], x["Hv"], x["dv"]
    anc = torch.empty(B, N, dtype=torch.int64, device=dev)
    pos = torch.empty(B, N, dtype=torch.int32, device=dev)
    st = torch.empty(B, dtype=torch.int32, device=dev)
    ctx = torch.full((B,), 1000, dtype=torch.int32, device=dev)
    tv.tv_build_ancestors(x["parent"], x["depth"], ctx, anc, pos, st)
    out = torch.empty(B, N, Hv, dv, device=dev)
    u = torch.empty_like(out)
    g = torch.empty(B, N, Hv, device=dev)
    new = torch.empty_like(x["state"])
    # accepted path per sequence: root to the first node at depth min(4, deepest), a
    # typical accepted length (the path's nodes are its ancestors-or-self, root first)
    par, dep = x["parent"].cpu(), x["depth"].cpu()
    acc_h = torch.zeros(B, N, dtype=torch.int32)
    n_acc_h = torch.zeros(B, dtype=torch.int32)
    for b in range(B):
        want = min(4, int(dep[b].max()))
        t = int((dep[b] == want).nonzero()[0, 0])
        path = []
        while t >= 0:
            path.append(t)
            t = int(par[b, t])
        path.reverse()
        acc_h[b, :len(path)] = torch.tensor(path, dtype=torch.int32)
        n_acc_h[b] = len(path)
    acc, n_acc = acc_h.to(dev), n_acc_h.to(dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        tv.tv_gdn_tree_verify(x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], anc, out,
                              u, g, st)
        if ev is not None:
            ev[1].record(stream)
        tv.tv_gdn_commit(x["state"], x["k"], u, x["alpha"], acc, n_acc, new, st)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize(dev)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / steps
    v_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    c_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / steps
    flops = gdn_flops(x)
    sm_mhz = 2070.0
    try:
        sm_mhz = float(torch.cuda.get_device_properties(dev).clock_rate) / 1000.0 or sm_mhz
    except Exception:
        pass
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak = sms * FP32_FMA_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    commit_bytes = 2 * B * Hv * dv * x["dk"] * 4
    return {
        "workload": (f"{name}: B={B} N={N} Hk/Hv={x['Hk']}/{x['Hv']} dk/dv={x['dk']}/{dv}, "
                     f"fp32 state, bf16 q/k/v"),
        "ms_per_step": ms, "verify_ms": v_ms, "commit_ms": c_ms,
        "verify_tflops": flops / (v_ms * 1e-3) / 1e12, "verify_flops": flops,
        "verify_bytes": gdn_bytes(x), "fp32_peak_tflops": alu_peak, "sm_mhz_for_peak": sm_mhz,
        "commit_gbs": commit_bytes / (c_ms * 1e-3) / 1e9, "status_ok": int(st.abs().sum()) == 0,
    }


def gdn_cpu_baseline(name, budget_s=10.0):
    """The oracle (fp64 per-path recurrence) on a bounded sample of the GDN
    workload: whole (sequence, value head) problems until the budget is spent,
    scaled to the full step."""
    import numpy as np
    import workloads
    from oracle import gdn as ogdn
    import oracle
    w = workloads.GDN_WORKLOADS[name]
    oracle.build()
    done, spent = 0, 0.0
    while spent < budget_s and done < w.B * w.Hv:
        x = workloads.make_gdn(name, "cpu", seed=w.seed + 7919 * (done + 1), B=1, Hk=1, Hv=1)
        mask, _, _ = oracle.ancestors(x["parent"].numpy(), x["depth"].numpy(),
                                      np.full(1, 10, np.int32))
        anc = (mask.astype(np.uint64) << np.arange(mask.shape[2], dtype=np.uint64)).sum(-1)
        f = lambda t: t.double().numpy()
        st = np.swapaxes(f(x["state"]), -1, -2)
        t0 = time.perf_counter()
        ogdn.tree_verify(st, f(x["q"]), f(x["k"]), f(x["v"]), f(x["alpha"]), f(x["beta"]), anc)
        spent += time.perf_counter() - t0
        done += 1
    per_step = spent / done * w.B * w.Hv
    return {"value": 1.0 / per_step, "unit": "steps/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {w.B * w.Hv} (sequence, value head) problems of {name} "
                      f"(numpy fp64 per-path recurrence), scaled by {w.B * w.Hv}/{done}"}


def bench_gdn(args, rank, world, local):
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    r = measure_gdn("gdn_stress", args.steps, args.warmup, dev, batch=args.batch,
                    seed_offset=rank)
    ms = max_over_ranks(r["ms_per_step"], world, dev)
    if rank != 0:
        return None
    return {
        "metric": GDN_METRIC, "value": job_throughput(world, 1, ms), "unit": "steps/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "impl": "ours", "path": "gdn",
        "config": {"workload": r["workload"], "l2": "state 134 MB read per step"},
        # the product runs on the tensor cores, so the kernel's bound is HBM:
        # the state, q / k / v and the outputs it must move once per step
        "roofline": {"kernel": "tv_gdn_tree_verify", "bound": "hbm",
                     "achieved": r["verify_bytes"] / (r["verify_ms"] * 1e-3) / 1e9,
                     "peak": peaks()[0], "unit": "GB/s",
                     "frac": r["verify_bytes"] / (r["verify_ms"] * 1e-3) / 1e9 / peaks()[0],
                     "traffic": None, "peak_source": peaks()[1]},
        "verify_fp32_tflops": r["verify_tflops"],
        "verify_ms": r["verify_ms"], "commit_ms": r["commit_ms"], "commit_gbs": r["commit_gbs"],
        "gpu_launches": 2 * args.steps, "status_ok": r["status_ok"],
        **({"cpu_baseline": gdn_cpu_baseline("gdn_stress")}
           if not args.no_cpu_baseline and world == 1 else {}),
    }


def oracle_step_sample(npi, heads):
    """One verify step of the oracle on a one-sequence input, attention limited
    to the first ``heads`` query heads.  Returns (attention seconds, rest seconds)."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    mask, pos, status = oracle.ancestors(npi["parent"], npi["depth"], npi["ctx_len"])
    t1 = time.perf_counter()
    Hq = npi["q"].shape[2]
    sel = np.zeros((1, Hq), bool)
    sel[:, :heads] = True
    oracle.attention(npi["q"], npi["k_tree"], npi["v_tree"], npi["k_cache"], npi["v_cache"],
                     npi["block_table"], npi["ctx_len"], mask, pos,
                     window_left=npi["window_left"], row_sel=sel)
    t2 = time.perf_counter()
    N = npi["tokens"].shape[1]
    am = oracle.argmax(npi["logits"].reshape(N, -1), npi["logits_dtype"]).reshape(1, N)
    _, _, acc_nodes, n_acc = oracle.walk(npi["tokens"], npi["parent"], am, npi["root_pred"],
                                         status)
    oracle.commit(npi["k_tree"], npi["v_tree"], acc_nodes, n_acc, npi["ctx_len"],
                  npi["block_table"], npi["k_cache"], npi["v_cache"])
    t3 = time.perf_counter()
    return t2 - t1, (t1 - t0) + (t3 - t2)


def reference_plan(est_attn_s, est_rest_s, Hq, steps, warmup, budget_s=150.0):
    """Query heads of attention per sampled step so that (steps + warmup) steps of
    one sequence fit in ``budget_s``: all heads when they fit, else fewer."""
    per_head = est_attn_s / Hq
    room = budget_s / max(1, steps + warmup) - est_rest_s
    heads = int(room // per_head) if per_head > 0 else Hq
    return max(1, min(Hq, heads))


def bench_reference(args, rank, world):
    """The oracle on the host cores: exactly K timed steps after W warm-up steps,
    each on a bounded sample (one sequence of the workload; all query heads when
    the run fits in a few minutes, else the first h of them), scaled to a whole
    batch.  Only rank 0 runs under torchrun."""
    if rank != 0:
        return None
    import workloads
    import oracle
    K, W = max(1, args.steps), max(0, args.warmup)
    w = workloads.get(args.workload)
    oracle.build()
    npi = workloads.to_numpy(workloads.make(args.workload, "cpu", seed=w.seed + 7919, B=1))
    Hq = npi["q"].shape[2]
    ea, er = oracle_step_sample(npi, Hq)
    heads = reference_plan(ea, er, Hq, K, W)
    for _ in range(W):
        oracle_step_sample(npi, heads)
    t = time.perf_counter()
    attn_s = rest_s = 0.0
    for _ in range(K):
        a, r = oracle_step_sample(npi, heads)
        attn_s += a
        rest_s += r
    elapsed = time.perf_counter() - t
    # one whole-batch step: B sequences, attention over all Hq heads
    Bj = w.B if args.batch is None else args.batch
    per_step = Bj * (attn_s / K * Hq / heads + rest_s / K)
    value = 1.0 / per_step
    cb = {"value": value, "unit": "steps/s", "cores": oracle.num_threads(), "kind": "oracle",
          "sample": (f"each of {K} steps: 1 of {Bj} sequences of the {args.workload} workload, "
                     f"full verify step with attention over {heads} of {Hq} query heads; "
                     f"attention time scaled by {Hq}/{heads}, the step by {Bj}")}
    return {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": 1000.0 / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": workload_config(args.workload, args.batch,
                                  l2="not applicable: the oracle runs on the host cores"),
        "cpu_baseline": cb,
        # what ran: one sequence per step (and `heads` of the query heads); the
        # line's value and ms_per_step are that time scaled to the whole batch
        "scaled_from": {"sequences_timed_per_step": 1, "batch": Bj, "query_heads_timed": heads,
                        "query_heads": Hq, "steps_timed": K, "wall_s_timed": elapsed,
                        "factor": Bj * Hq / heads if heads else None},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": elapsed,
    }


def main():
    args = parse()
    rank, world, local = dist_info()
    if args.impl == "reference":
        line = bench_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if args.path == "draft":
        line = bench_draft(args, rank, world, local)
    elif args.path == "graph":
        line = bench_graph(args, rank, world, local)
    elif args.path == "gdn":
        line = bench_gdn(args, rank, world, local)
    else:
        line = bench_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

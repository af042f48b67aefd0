"""Benchmark: MoE routing layout + bf16 dispatch + weighted combine on one GB300.

Workload (prefill shape): T=8192 tokens, H=7168, E=256 experts, top-8,
R=8 logical rank slabs; x bf16 ~N(0,1), K distinct uniform experts per token,
fp32 weights U(0,1) normalised, expert outputs y bf16 ~N(0,1) [N, H].
One step = ep_layout + ep_dispatch(bf16) + ep_combine through the C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line on rank 0. Under torchrun every rank runs its own
replica of the workload on its own GPU (no data exchange); the step time is
the max over ranks and `value` counts the bytes of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gen import inputs as gi  # noqa: E402

METRIC = "dispatch & combine HBM GB/s + tokens/s, T=8192 H=7168 E=256 top-8 bf16"
WORKLOAD = "prefill"
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------- bytes

def bytes_layout(T, K, E, R):
    # topk_idx read, counts/offsets/masks written, slot -> row map written
    return 8 * T * K + 4 * E + 4 * R + T * R + 4 * (E + 1) + 4 * T * K


def bytes_dispatch_bf16(T, K, H, N):
    return 2 * T * H + 2 * N * H + 4 * T * K


def bytes_dispatch_fp8(T, K, H, N):
    return 2 * T * H + N * H + 4 * N * (H // 128) + 4 * T * K


def bytes_combine(T, K, H, N):
    return 2 * N * H + 4 * T * K + 4 * T * K + 2 * T * H


# ---------------------------------------------------------------- environment

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.samples = []   # (t, sm, max, reasons set)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={self.period}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            reasons = {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}
            self.samples.append((time.perf_counter(), sm, mx, reasons))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "timed region"
        if not win and self.samples:
            # the timed region was shorter than one sampling period: use the
            # samples closest to it (warm-up and timed work run back to back)
            win = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            note = "nearest samples (timed region shorter than the sampling period)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        reasons = sorted(set().union(*[s[3] for s in win]))
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": max(s[2] for s in win),
                "reasons": reasons, "samples": len(win), "note": note}


def smi_id(local: int) -> str:
    """nvidia-smi's id of CUDA device `local` (honours CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


def read_traffic(kernel: str, T: int, case: str = "prefill"):
    """Per-launch DRAM bytes of `kernel` on workload `case` from the committed
    ncu summary profiles/dram_traffic_<case>_T<T>.md, if the capture was of
    this token count and the kernel source has not changed since (else None)."""
    import hashlib
    import re

    path = os.path.join(ROOT, "profiles", f"dram_traffic_{case}_T{T}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(rf"<!-- traffic kernel={kernel}(?: case={case})? T=(\d+) bytes=(\d+) src_sha256=([0-9a-f]+) -->",
                  txt)
    if not m or int(m.group(1)) != T:
        return None
    src = {"dispatch_bf16": "ep_dispatch.cu", "combine": "ep_combine.cu"}.get(kernel)
    if src is None:
        return None
    h = hashlib.sha256(open(os.path.join(ROOT, "combine_get_dispatch_layout_gb300", "csrc", src), "rb").read())
    return int(m.group(2)) if h.hexdigest()[:16] == m.group(3) else None


def aggregate_over_ranks(local_ms: float, local_bytes: int, device=None):
    """Whole-job numbers for replicas on several ranks: the step time is the
    slowest rank's, the bytes are every rank's. Returns (max_ms, total_bytes).
    One scalar all-reduce each; nothing on the data path is exchanged."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local_ms, local_bytes
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor([local_bytes], dtype=torch.float64, device=device)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


# ---------------------------------------------------------------- device timing

class L2Flush:
    """Empties L2 of the workload: writes one buffer twice the L2 size, then
    reads another of that size, so L2 is left holding clean lines of the
    second (no dirty line is left for the next kernel to write back). Call it
    with `stream` current; it is never inside a timed interval."""

    def __init__(self, torch, dev, stream):
        l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or L2_BYTES
        with torch.cuda.stream(stream):
            self.w = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
            self.r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
            self.acc = torch.empty((), dtype=torch.float32, device=dev)
        self.torch = torch
        self.mib = 2 * l2 >> 20

    def __call__(self):
        self.w.fill_(1.0)
        self.torch.sum(self.r, dim=0, out=self.acc)


def graph_us(torch, stream, body, n=20, replays=10):
    """Device time (us) of one body() from a CUDA graph of n copies of it,
    replayed between two events: no host launch cost, and the library's
    kernels keep their programmatic edges inside the graph (so one copy's
    first kernel may start while the previous copy's last one drains)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        body()
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                body()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    del g
    return e0.elapsed_time(e1) / (n * replays) * 1e3


def graph_prefix_us(torch, stream, bodies, n=20, rounds=30):
    """Device time (us) per copy of each body in `bodies`, each captured n
    times into its own CUDA graph. The graphs are replayed round-robin
    `rounds` times with events around every replay, and the median replay
    time is taken, so slow drift of the clock or the memory system affects
    all bodies alike. Bodies that extend one another (flush; flush + layout;
    flush + layout + dispatch; ...) give each kernel's marginal cost inside
    the step as the difference of neighbours."""
    graphs = []
    with torch.cuda.stream(stream):
        for body in bodies:
            body()
        stream.synchronize()
        for body in bodies:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(n):
                    body()
            g.replay()
            graphs.append(g)
        stream.synchronize()
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in graphs]
              for _ in range(rounds)]
        for r in range(rounds):
            for j, g in enumerate(graphs):
                ev[r][j][0].record(stream)
                g.replay()
                ev[r][j][1].record(stream)
    stream.synchronize()
    out = [float(np.median([ev[r][j][0].elapsed_time(ev[r][j][1]) for r in range(rounds)])) * 1e3 / n
           for j in range(len(graphs))]
    del graphs
    return out


# ---------------------------------------------------------------- GPU arm

def gpu_arm(args, rank, world, local):
    import torch

    import combine_get_dispatch_layout_gb300 as ep

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    ep.lib()   # raises if the library is missing: there is no other path

    inp = gi.make(WORKLOAD, seed=args.seed + rank, T=args.tokens)
    w = inp.w
    T, H, E, K, R, N = w.T, w.H, w.E, w.K, w.R, inp.num_valid

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        idx = torch.from_numpy(inp.topk_idx).to(dev)
        x = torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16)
        wt = torch.from_numpy(inp.topk_weights).to(dev)
        y = torch.from_numpy(inp.y.view(np.int16)).to(dev).view(torch.bfloat16)
        cnt = torch.empty(E, dtype=torch.int32, device=dev)
        ntr = torch.empty(R, dtype=torch.int32, device=dev)
        itr = torch.empty(T, R, dtype=torch.uint8, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        recv = torch.empty(N, H, dtype=torch.bfloat16, device=dev)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    stream.synchronize()
    handle = ep.ep_layout(idx, E, R, cnt, ntr, itr, off, stream=stream)   # creates the handle once

    def step(ev=None):
        # timed step: the dispatch is the layout's programmatic dependent, so
        # it loads x on the SMs the layout leaves idle
        ep.ep_layout(idx, E, R, cnt, ntr, itr, off, handle=handle, stream=stream)
        ep.ep_dispatch_ex(handle, x, recv, N, out_dtype=ep.EP_DTYPE_BF16, overlap_layout=True, stream=stream)
        ep.ep_combine(handle, y, out, topk_weights=wt, stream=stream)

    def step_split(ev):
        # the same work with an event after every call (no overlap), for the
        # per-kernel breakdown
        ev[0].record(stream)
        ep.ep_layout(idx, E, R, cnt, ntr, itr, off, handle=handle, stream=stream)
        ev[1].record(stream)
        ep.ep_dispatch(handle, x, ep.EP_DTYPE_BF16, recv, N, stream=stream)
        ev[2].record(stream)
        ep.ep_combine(handle, y, out, topk_weights=wt, stream=stream)
        ev[3].record(stream)

    sampler = ClockSampler(smi_id(local))
    sampler.start()
    time.sleep(0.3)
    t_host0 = time.perf_counter()
    for _ in range(args.warmup):
        step()
    host_s_per_step = (time.perf_counter() - t_host0) / args.warmup   # enqueue time (bounded by the GPU)
    stream.synchronize()
    events = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    # The stream is empty here: without a lead, the GPU would idle between the
    # first event and the first kernel while the host enqueues it. A sleep
    # kernel ahead of the first event (outside the timed interval) holds the
    # stream while the host queues the first steps, so the events time the
    # device alone.
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(min(1e8, 2.1e9 * host_s_per_step * min(args.steps, 8) + 2e5)))
    events[0].record(stream)
    for i in range(args.steps):
        step()
    events[args.steps].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.perf_counter()
    layout_kernels = ep.ep_handle_layout_kernels(handle)
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.15)
    sampler.stop()
    total_ms = float(events[0].elapsed_time(events[args.steps]))

    reps_split = max(3, min(args.steps, 200))
    split = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps_split)]
    for i in range(reps_split):
        step_split(split[i])
    stream.synchronize()
    per = np.array([[split[i][j].elapsed_time(split[i][j + 1]) for j in range(3)] for i in range(reps_split)])
    ms_layout, ms_dispatch, ms_combine = (float(per[:, j].mean()) for j in range(3))

    # layout + dispatch end to end (the dispatch as the layout's programmatic
    # dependent), events only at the pair boundaries
    ev_ld = [torch.cuda.Event(enable_timing=True) for _ in range(reps_split + 1)]
    for i in range(-3, reps_split):
        if i >= 0:
            ev_ld[i].record(stream)
        ep.ep_layout(idx, E, R, cnt, ntr, itr, off, handle=handle, stream=stream)
        ep.ep_dispatch_ex(handle, x, recv, N, out_dtype=ep.EP_DTYPE_BF16, overlap_layout=True, stream=stream)
    ev_ld[reps_split].record(stream)
    stream.synchronize()
    ms_lay_dis = float(np.mean([ev_ld[i].elapsed_time(ev_ld[i + 1]) for i in range(reps_split)]))
    b_lay = bytes_layout(T, K, E, R)
    b_dis = bytes_dispatch_bf16(T, K, H, N)
    b_com = bytes_combine(T, K, H, N)
    b_step = b_lay + b_dis + b_com
    total_ms, job_bytes = aggregate_over_ranks(total_ms, b_step, device=dev)
    ms_step = total_ms / args.steps
    peak, peak_src = load_peaks()

    # fp8 quantise-permute on the fp8 workload (same shapes and routing recipe)
    fp8 = gi.make("fp8", seed=args.seed + rank, with_y=False, T=args.tokens)
    with torch.cuda.stream(stream):
        x8 = torch.from_numpy(fp8.x.view(np.int16)).to(dev).view(torch.bfloat16)
        idx8 = torch.from_numpy(fp8.topk_idx).to(dev)
        q = torch.empty(fp8.num_valid, H, dtype=torch.uint8, device=dev)
        sc = torch.empty(fp8.num_valid, H // 128, dtype=torch.float32, device=dev)
    h8 = ep.ep_layout(idx8, E, R, cnt, ntr, itr, off, stream=stream)
    reps8 = max(3, min(args.steps, 200))
    ev8 = [torch.cuda.Event(enable_timing=True) for _ in range(reps8 + 1)]
    for _ in range(3):
        ep.ep_dispatch(h8, x8, ep.EP_DTYPE_FP8_E4M3, q, fp8.num_valid, recv_scales=sc, stream=stream)
    for i in range(reps8):
        ev8[i].record(stream)
        ep.ep_dispatch(h8, x8, ep.EP_DTYPE_FP8_E4M3, q, fp8.num_valid, recv_scales=sc, stream=stream)
    ev8[reps8].record(stream)
    stream.synchronize()
    ms_fp8 = float(np.mean([ev8[i].elapsed_time(ev8[i + 1]) for i in range(reps8)]))
    b_fp8 = bytes_dispatch_fp8(T, K, H, fp8.num_valid)
    # the same dispatch back to back (20 launches in a CUDA graph, each the
    # programmatic dependent of the one before): the per-call ramp and tail
    # overlap the neighbouring launches, as they do inside a chained step
    us_fp8_chained = graph_us(torch, stream, lambda: ep.ep_dispatch(h8, x8, ep.EP_DTYPE_FP8_E4M3, q, fp8.num_valid,
                                                                    recv_scales=sc, stream=stream), n=20, replays=5)

    # fp8 variants on the same routing: power-of-two scales; UE8M0 byte scales
    # in column-major layout; fp8 input pass-through (codes and scales moved)
    n8, nb = fp8.num_valid, H // 128
    with torch.cuda.stream(stream):
        sc_u = torch.empty(nb * n8, dtype=torch.uint8, device=dev)
        codes_in = torch.randint(0, 256, (T, H), dtype=torch.uint8, device=dev)
        scales_in = torch.rand(T, nb, dtype=torch.float32, device=dev)

    def time_variant(fn):
        for _ in range(3):
            fn()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps8 + 1)]
        for i in range(reps8):
            evs[i].record(stream)
            fn()
        evs[reps8].record(stream)
        stream.synchronize()
        return float(np.mean([evs[i].elapsed_time(evs[i + 1]) for i in range(reps8)]))

    ms_pow2 = time_variant(lambda: ep.ep_dispatch_ex(h8, x8, q, n8, scale_mode=ep.EP_SCALE_POW2, recv_scales=sc,
                                                     stream=stream))
    ms_ue8 = time_variant(lambda: ep.ep_dispatch_ex(h8, x8, q, n8, scale_mode=ep.EP_SCALE_UE8M0, recv_scales=sc_u,
                                                    scales_col_major=True, scales_ld=n8, stream=stream))
    ms_pass = time_variant(lambda: ep.ep_dispatch_ex(h8, codes_in, q, n8, in_dtype=ep.EP_DTYPE_FP8_E4M3,
                                                     x_scales=scales_in, recv_scales=sc, H=H, stream=stream))
    ms_e5m2 = time_variant(lambda: ep.ep_dispatch_ex(h8, x8, q, n8, out_dtype=ep.EP_DTYPE_FP8_E5M2,
                                                     recv_scales=sc, stream=stream))
    b_ue8 = 2 * T * H + n8 * H + n8 * nb + 4 * T * K
    b_pass = T * H + 4 * T * nb + n8 * H + 4 * n8 * nb + 4 * T * K
    del codes_in, scales_in, sc_u

    # the fp8 workload's step: layout, fp8 dispatch as its programmatic
    # dependent (x prefetched during the layout), combine of bf16 expert
    # outputs (y of the prefill workload stands in: same row count)
    with torch.cuda.stream(stream):
        wt8 = torch.from_numpy(fp8.topk_weights).to(dev)
    n_y = min(N, n8)

    def step8():
        ep.ep_layout(idx8, E, R, cnt, ntr, itr, off, handle=h8, stream=stream)
        ep.ep_dispatch_ex(h8, x8, q, n8, recv_scales=sc, overlap_layout=True, stream=stream)
        ep.ep_combine(h8, y, out, topk_weights=wt8, y_rows=n_y, stream=stream)

    for _ in range(3):
        step8()
    ev_s8 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev_s8[0].record(stream)
    for _ in range(reps8):
        step8()
    ev_s8[1].record(stream)
    stream.synchronize()
    ms_step8 = ev_s8[0].elapsed_time(ev_s8[1]) / reps8
    b_step8 = b_lay + b_fp8 + bytes_combine(T, K, H, n8)

    # backward passes on the same routing: combine backward (x stands in for
    # grad_out, y for the forward expert outputs, recv receives grad_y) and
    # dispatch backward (y stands in for grad_recv, out receives grad_x)
    with torch.cuda.stream(stream):
        gw = torch.empty(T, K, dtype=torch.float32, device=dev)
        grw = torch.randn(N, dtype=torch.float32, device=dev)
        gtw = torch.empty(T, K, dtype=torch.float32, device=dev)
    reps_b = max(3, min(args.steps, 100))
    ev_b = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps_b)]
    for i in range(-3, reps_b):
        if i >= 0:
            ev_b[i][0].record(stream)
        ep.ep_combine_backward(handle, x, y=y, topk_weights=wt, grad_y=recv, grad_topk_weights=gw, stream=stream)
        if i >= 0:
            ev_b[i][1].record(stream)
        ep.ep_dispatch_backward(handle, y, out, grad_recv_weights=grw, grad_topk_weights=gtw, stream=stream)
        if i >= 0:
            ev_b[i][2].record(stream)
    stream.synchronize()
    ms_cbw = float(np.mean([e[0].elapsed_time(e[1]) for e in ev_b]))
    ms_dbw = float(np.mean([e[1].elapsed_time(e[2]) for e in ev_b]))
    b_cbw = 2 * T * H + 4 * N * H + 4 * T * K * 3
    b_dbw = bytes_combine(T, K, H, N) + 4 * T * K + 4 * N + 4 * T * K

    # dense routing map <-> sparse top-k conversions on the prefill routing
    with torch.cuda.stream(stream):
        rmap = torch.empty(T, E, dtype=torch.uint8, device=dev)
        probs = torch.empty(T, E, dtype=torch.float32, device=dev)
        idx_back = torch.empty(T, K, dtype=torch.int64, device=dev)
        w_back = torch.empty(T, K, dtype=torch.float32, device=dev)
    # each conversion captured 20 times into a CUDA graph and replayed, so the
    # GPU time is not hidden behind the host cost of launching a ~5 us kernel
    ms_t2m = graph_us(torch, stream, lambda: ep.ep_topk_to_routing_map(idx, E, rmap, topk_weights=wt, probs=probs,
                                                                       stream=stream)) / 1e3
    ms_m2t = graph_us(torch, stream, lambda: ep.ep_routing_map_to_topk(rmap, K, idx_back, probs=probs,
                                                                       topk_weights=w_back, stream=stream)) / 1e3
    b_t2m = 12 * T * K + 5 * T * E
    b_m2t = 5 * T * E + 12 * T * K
    del rmap, probs, idx_back, w_back

    # aligned layout (expert rows start on multiples of 128) + bf16 dispatch
    # including the pad rows' zero fill, on the prefill routing
    A = 128
    with torch.cuda.stream(stream):
        off_a = torch.empty(E + 1, dtype=torch.int32, device=dev)
        recv_a = torch.empty(N + E * (A - 1), H, dtype=torch.bfloat16, device=dev)
    h_a = ep.ep_layout_aligned(idx, E, R, A, cnt, ntr, itr, off_a, stream=stream)
    n_pad, _ = ep.ep_handle_query(h_a)
    reps_a = max(3, min(args.steps, 100))
    ev_a = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps_a)]
    for i in range(-3, reps_a):
        if i >= 0:
            ev_a[i][0].record(stream)
        ep.ep_layout_aligned(idx, E, R, A, cnt, ntr, itr, off_a, handle=h_a, stream=stream)
        if i >= 0:
            ev_a[i][1].record(stream)
        ep.ep_dispatch(h_a, x, ep.EP_DTYPE_BF16, recv_a, recv_a.shape[0], stream=stream)
        if i >= 0:
            ev_a[i][2].record(stream)
    stream.synchronize()
    ms_lay_a = float(np.mean([e[0].elapsed_time(e[1]) for e in ev_a]))
    ms_dis_a = float(np.mean([e[1].elapsed_time(e[2]) for e in ev_a]))
    b_dis_a = 2 * T * H + 2 * n_pad * H + 4 * T * K
    h_a.destroy()
    del recv_a

    # non-expand layout (one row per (token, rank)) + bf16 dispatch, prefill routing
    with torch.cuda.stream(stream):
        off_r = torch.empty(R + 1, dtype=torch.int32, device=dev)
        recv_ne = torch.empty(T * R, H, dtype=torch.bfloat16, device=dev)
    h_ne = ep.ep_layout_nonexpand(idx, E, R, cnt, ntr, itr, off_r, stream=stream)
    n_ne, _ = ep.ep_handle_query(h_ne)
    ev_ne = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps_b)]
    for i in range(-3, reps_b):
        if i >= 0:
            ev_ne[i][0].record(stream)
        ep.ep_layout_nonexpand(idx, E, R, cnt, ntr, itr, off_r, handle=h_ne, stream=stream)
        if i >= 0:
            ev_ne[i][1].record(stream)
        ep.ep_dispatch(h_ne, x, ep.EP_DTYPE_BF16, recv_ne, T * R, stream=stream)
        if i >= 0:
            ev_ne[i][2].record(stream)
    stream.synchronize()
    ms_ne = [float(np.mean([e[j].elapsed_time(e[j + 1]) for e in ev_ne])) for j in range(2)]
    b_ne = 2 * T * H + 2 * n_ne * H + 4 * T * K
    h_ne.destroy()
    del recv_ne

    others = other_configs(torch, ep, dev, stream, args, rank, peak, reps_b)

    # end to end through the public API with pinned host buffers
    e2e = e2e_measure(torch, ep, dev, inp, args, stream)
    e2e["ms_per_step"], _ = aggregate_over_ranks(e2e["ms_per_step"], 0, device=dev)
    handle.destroy()
    h8.destroy()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    dominant = "dispatch_bf16" if ms_dispatch >= ms_combine else "combine"
    dom_ms = ms_dispatch if dominant == "dispatch_bf16" else ms_combine
    dom_bytes = b_dis if dominant == "dispatch_bf16" else b_com
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    clocks = sampler.summary(t_wall0 - 0.3, t_wall1)
    line = {
        "metric": METRIC,
        "value": round(job_bytes / (ms_step * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64; recipe in gen/inputs.py)",
        "config": {"workload": f"prefill dispatch+combine: T={T} H=7168 E=256 K=8 R=8, bf16 rows, "
                               "uniform distinct routing, fp32 weights U(0,1) normalised",
                   "T": T, "H": H, "E": E, "K": K, "R": R, "N": N,
                   "step": "ep_layout + ep_dispatch(bf16) + ep_combine",
                   "l2": "no flush: every step moves >1 GB (> 129 MB L2) through each of dispatch and combine",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(world * T / (ms_step * 1e-3), 1),
        "step_note": "step = layout, then bf16 dispatch launched as the layout's programmatic dependent "
                     "(overlap_layout), then combine; the kernels' separate times below come from the same "
                     "calls with an event between each (no overlap); a sleep kernel ahead of the first timed "
                     "event keeps the host's first launches out of the device-timed interval",
        "overlap_saved_us": round((ms_layout + ms_dispatch + ms_combine - ms_step) * 1e3, 2),
        "kernels": {
            "layout": {"us": round(ms_layout * 1e3, 2), "bytes": b_lay,
                       "note": "CUDA events around the one call, after the previous step's combine, not chained: "
                               "includes the launch of a 16-CTA cluster and ~2 us of event overhead; inside the "
                               "timed step the layout runs beside the dispatch's prefetch of x"},
            "dispatch_bf16": {"us": round(ms_dispatch * 1e3, 2), "bytes": b_dis,
                              "tokens_per_s": round(T / (ms_dispatch * 1e-3), 1),
                              "rows_per_s": round(N / (ms_dispatch * 1e-3), 1),
                              "gbs": round(b_dis / (ms_dispatch * 1e-3) / 1e9, 1),
                              "frac_of_measured": round(b_dis / (ms_dispatch * 1e-3) / 1e9 / peak, 4),
                              "frac_of_8tbs": round(b_dis / (ms_dispatch * 1e-3) / 8e12, 4)},
            "combine": {"us": round(ms_combine * 1e3, 2), "bytes": b_com,
                        "tokens_per_s": round(T / (ms_combine * 1e-3), 1),
                        "rows_per_s": round(N / (ms_combine * 1e-3), 1),
                        "gbs": round(b_com / (ms_combine * 1e-3) / 1e9, 1),
                        "frac_of_measured": round(b_com / (ms_combine * 1e-3) / 1e9 / peak, 4),
                        "frac_of_8tbs": round(b_com / (ms_combine * 1e-3) / 8e12, 4)},
            "layout_plus_dispatch_bf16": {"us": round(ms_lay_dis * 1e3, 2), "bytes": b_lay + b_dis,
                                          "gbs": round((b_lay + b_dis) / (ms_lay_dis * 1e-3) / 1e9, 1),
                                          "note": "dispatch launched as the layout's programmatic dependent"},
            "dispatch_bf16_aligned128": {"rows_padded": n_pad, "layout_us": round(ms_lay_a * 1e3, 2),
                                         "us": round(ms_dis_a * 1e3, 2), "bytes": b_dis_a,
                                         "gbs": round(b_dis_a / (ms_dis_a * 1e-3) / 1e9, 1),
                                         "frac_of_measured": round(b_dis_a / (ms_dis_a * 1e-3) / 1e9 / peak, 4),
                                         "frac_of_8tbs": round(b_dis_a / (ms_dis_a * 1e-3) / 8e12, 4)},
            "dispatch_fp8_pow2": {"us": round(ms_pow2 * 1e3, 2), "bytes": b_fp8,
                                  "gbs": round(b_fp8 / (ms_pow2 * 1e-3) / 1e9, 1),
                                  "frac_of_measured": round(b_fp8 / (ms_pow2 * 1e-3) / 1e9 / peak, 4)},
            "dispatch_fp8_ue8m0_colmajor": {"us": round(ms_ue8 * 1e3, 2), "bytes": b_ue8,
                                            "gbs": round(b_ue8 / (ms_ue8 * 1e-3) / 1e9, 1),
                                            "frac_of_measured": round(b_ue8 / (ms_ue8 * 1e-3) / 1e9 / peak, 4)},
            "dispatch_fp8_e5m2": {"us": round(ms_e5m2 * 1e3, 2), "bytes": b_fp8,
                                  "gbs": round(b_fp8 / (ms_e5m2 * 1e-3) / 1e9, 1),
                                  "frac_of_measured": round(b_fp8 / (ms_e5m2 * 1e-3) / 1e9 / peak, 4)},
            "dispatch_fp8_passthrough": {"us": round(ms_pass * 1e3, 2), "bytes": b_pass,
                                         "gbs": round(b_pass / (ms_pass * 1e-3) / 1e9, 1),
                                         "frac_of_measured": round(b_pass / (ms_pass * 1e-3) / 1e9 / peak, 4)},
            "topk_to_routing_map": {"us": round(ms_t2m * 1e3, 2), "bytes": b_t2m,
                                    "gbs": round(b_t2m / (ms_t2m * 1e-3) / 1e9, 1), "timing": "CUDA graph"},
            "routing_map_to_topk": {"us": round(ms_m2t * 1e3, 2), "bytes": b_m2t,
                                    "gbs": round(b_m2t / (ms_m2t * 1e-3) / 1e9, 1), "timing": "CUDA graph"},
            "dispatch_bf16_nonexpand": {"rows": n_ne, "layout_us": round(ms_ne[0] * 1e3, 2),
                                        "us": round(ms_ne[1] * 1e3, 2), "bytes": b_ne,
                                        "gbs": round(b_ne / (ms_ne[1] * 1e-3) / 1e9, 1),
                                        "frac_of_measured": round(b_ne / (ms_ne[1] * 1e-3) / 1e9 / peak, 4)},
            **others,
            "combine_backward": {"us": round(ms_cbw * 1e3, 2), "bytes": b_cbw,
                                 "gbs": round(b_cbw / (ms_cbw * 1e-3) / 1e9, 1),
                                 "frac_of_measured": round(b_cbw / (ms_cbw * 1e-3) / 1e9 / peak, 4)},
            "dispatch_backward": {"us": round(ms_dbw * 1e3, 2), "bytes": b_dbw,
                                  "gbs": round(b_dbw / (ms_dbw * 1e-3) / 1e9, 1),
                                  "frac_of_measured": round(b_dbw / (ms_dbw * 1e-3) / 1e9 / peak, 4)},
            "fp8_step": {"workload": "fp8 routing: layout + e4m3 dispatch (overlapped) + bf16 combine",
                         "us": round(ms_step8 * 1e3, 2), "bytes": b_step8,
                         "gbs": round(b_step8 / (ms_step8 * 1e-3) / 1e9, 1),
                         "frac_of_measured": round(b_step8 / (ms_step8 * 1e-3) / 1e9 / peak, 4)},
            "dispatch_fp8": {"workload": "fp8: x ~N(0,2^2) + 7 outlier channels x50, same shapes",
                             "us": round(ms_fp8 * 1e3, 2), "bytes": b_fp8,
                             "gbs": round(b_fp8 / (ms_fp8 * 1e-3) / 1e9, 1),
                             "frac_of_measured": round(b_fp8 / (ms_fp8 * 1e-3) / 1e9 / peak, 4),
                             "frac_of_8tbs": round(b_fp8 / (ms_fp8 * 1e-3) / 8e12, 4),
                             "timing": "us: CUDA events around each call (includes the launch ramp and tail); "
                                       "us_chained: 20 launches back to back in a CUDA graph",
                             "us_chained": round(us_fp8_chained, 2),
                             "gbs_chained": round(b_fp8 / us_fp8_chained / 1e3, 1),
                             "frac_of_measured_chained": round(b_fp8 / us_fp8_chained / 1e3 / peak, 4)},
        },
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": read_traffic(dominant, T),
                     "note": "timed inside the step; the combine also writes back the dispatch's last ~61 MB "
                             "of dirty L2 lines, which are not in its algorithmic bytes"
                             if dominant == "combine" else "timed inside the step"},
        "e2e": {"value": round(job_bytes / (e2e["ms_per_step"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e["ms_per_step"], 4), "steps": e2e["steps"], "how": e2e["how"]},
        "gpu_launches": (layout_kernels + 2) * args.steps,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def other_configs(torch, ep, dev, stream, args, rank, peak, reps):
    """The skewed workload's step (T=16384, H=4096, E=64, top-6 with drops),
    and the decode (T=256, H=7168, E=256, top-8) and tiny (T=128, H=256, E=8,
    top-2) steps with device times L2-cold and warm."""
    out = {}

    def split_loop(calls):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(reps)]
        for i in range(-3, reps):
            for j, call in enumerate(calls):
                if i >= 0:
                    ev[i][j].record(stream)
                call()
            if i >= 0:
                ev[i][len(calls)].record(stream)
        stream.synchronize()
        return [float(np.mean([e[j].elapsed_time(e[j + 1]) for e in ev])) for j in range(len(calls))]

    def tensors(inp, rows):
        w = inp.w
        with torch.cuda.stream(stream):
            t = {"idx": torch.from_numpy(inp.topk_idx).to(dev),
                 "x": torch.from_numpy(inp.x.view(np.int16)).to(dev),
                 "w": torch.from_numpy(inp.topk_weights).to(dev),
                 "recv": torch.empty(rows, w.H, dtype=torch.int16, device=dev),
                 "out": torch.empty(w.T, w.H, dtype=torch.int16, device=dev),
                 "cnt": torch.empty(w.E, dtype=torch.int32, device=dev),
                 "ntr": torch.empty(w.R, dtype=torch.int32, device=dev),
                 "itr": torch.empty(w.T, w.R, dtype=torch.uint8, device=dev),
                 "off": torch.empty(w.E + 1, dtype=torch.int32, device=dev)}
        return t

    # skewed: Zipf expert popularity, 5% dropped slots; y stands in for the
    # expert outputs. The receive and expert-output buffers hold T*K rows, the
    # most the routing can need, so no call waits for the layout's row count
    sk = gi.make("skewed", seed=args.seed + rank)
    ws, Ns = sk.w, sk.num_valid
    cap = ws.T * ws.K
    t = tensors(sk, cap)
    with torch.cuda.stream(stream):
        y = torch.zeros(cap, ws.H, dtype=torch.int16, device=dev)
        y[:Ns] = torch.from_numpy(sk.y.view(np.int16)).to(dev)
    h = ep.ep_layout(t["idx"], ws.E, ws.R, t["cnt"], t["ntr"], t["itr"], t["off"], stream=stream)
    ms = split_loop([
        lambda: ep.ep_layout(t["idx"], ws.E, ws.R, t["cnt"], t["ntr"], t["itr"], t["off"], handle=h, stream=stream),
        lambda: ep.ep_dispatch(h, t["x"], ep.EP_DTYPE_BF16, t["recv"], cap, stream=stream),
        lambda: ep.ep_combine(h, y, t["out"], topk_weights=t["w"], stream=stream)])

    def sk_step():
        ep.ep_layout(t["idx"], ws.E, ws.R, t["cnt"], t["ntr"], t["itr"], t["off"], handle=h, stream=stream)
        ep.ep_dispatch_ex(h, t["x"], t["recv"], cap, out_dtype=ep.EP_DTYPE_BF16, overlap_layout=True, stream=stream)
        ep.ep_combine(h, y, t["out"], topk_weights=t["w"], stream=stream)

    for _ in range(3):
        sk_step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        sk_step()
    e1.record(stream)
    stream.synchronize()
    ms_sk_step = e0.elapsed_time(e1) / reps
    h.destroy()
    bd, bc = bytes_dispatch_bf16(ws.T, ws.K, ws.H, Ns), bytes_combine(ws.T, ws.K, ws.H, Ns)
    out["skewed_step"] = {
        "workload": f"skewed: T={ws.T} H={ws.H} E={ws.E} K={ws.K} R={ws.R}, Zipf(1.2) experts, "
                    f"5% dropped slots, N={Ns}",
        "layout_us": round(ms[0] * 1e3, 2),
        "dispatch_us": round(ms[1] * 1e3, 2), "dispatch_gbs": round(bd / (ms[1] * 1e-3) / 1e9, 1),
        "dispatch_frac_of_measured": round(bd / (ms[1] * 1e-3) / 1e9 / peak, 4),
        "combine_us": round(ms[2] * 1e3, 2), "combine_gbs": round(bc / (ms[2] * 1e-3) / 1e9, 1),
        "combine_frac_of_measured": round(bc / (ms[2] * 1e-3) / 1e9 / peak, 4),
        "tokens_per_s": round(ws.T / (sum(ms) * 1e-3), 1),
        "step_us_chained": round(ms_sk_step * 1e3, 2),
        "step_gbs_chained": round((bytes_layout(ws.T, ws.K, ws.E, ws.R) + bd + bc) / (ms_sk_step * 1e-3) / 1e9, 1),
        "step_frac_of_measured_chained": round((bytes_layout(ws.T, ws.K, ws.E, ws.R) + bd + bc) / (ms_sk_step * 1e-3)
                                               / 1e9 / peak, 4),
        "tokens_per_s_chained": round(ws.T / (ms_sk_step * 1e-3), 1),
        "combine_traffic": read_traffic("combine", ws.T, "skewed"),
        "traffic_note": "the combine's per-launch DRAM read + write bytes from one ncu pass "
                        "(profiles/dram_traffic_skewed_T16384.md), null if its source changed since"}
    del t, y

    flush = L2Flush(torch, dev, stream)

    # decode as configured (T=256, H=7168, E=256, top-8): expand layout,
    # dispatch, combine of y [T*K, H] in dispatch order
    dec = gi.make("decode", seed=args.seed + rank)
    wd, Nd = dec.w, dec.num_valid
    t = tensors(dec, Nd)
    with torch.cuda.stream(stream):
        y = torch.from_numpy(dec.y.view(np.int16)).to(dev)
    h = ep.ep_layout(t["idx"], wd.E, wd.R, t["cnt"], t["ntr"], t["itr"], t["off"], stream=stream)
    out["decode_step"] = small_step_report(
        torch, stream, flush, peak, wd, Nd,
        f"decode T={wd.T} H={wd.H} E={wd.E} K={wd.K} R={wd.R}: ep_layout (expand) + ep_dispatch(bf16) + "
        f"ep_combine, y [T*K, H] in dispatch order, N={Nd}",
        lambda: ep.ep_layout(t["idx"], wd.E, wd.R, t["cnt"], t["ntr"], t["itr"], t["off"], handle=h, stream=stream),
        lambda: ep.ep_dispatch(h, t["x"], ep.EP_DTYPE_BF16, t["recv"], Nd, stream=stream),
        lambda: ep.ep_dispatch_ex(h, t["x"], t["recv"], Nd, out_dtype=ep.EP_DTYPE_BF16, overlap_layout=True,
                                  stream=stream),
        lambda: ep.ep_combine(h, y, t["out"], topk_weights=t["w"], stream=stream))
    h.destroy()
    del t, y

    # the same decode routing through the padded 3-D low-latency layout
    # [E, cap, H], cap = T (every token could pick one expert)
    cap = wd.T
    t = tensors(dec, wd.E * cap)
    with torch.cuda.stream(stream):
        y = torch.randn(wd.E * cap, wd.H, device=dev).to(torch.bfloat16).view(torch.int16)
    h = ep.ep_layout_strided(t["idx"], wd.E, wd.R, cap, t["cnt"], t["ntr"], t["itr"], t["off"], stream=stream)
    out["decode_ll_step"] = small_step_report(
        torch, stream, flush, peak, wd, Nd,
        f"decode T={wd.T} H={wd.H} E={wd.E} K={wd.K} R={wd.R}: ep_layout_strided (cap={cap}) + ep_dispatch(bf16) "
        "+ ep_combine",
        lambda: ep.ep_layout_strided(t["idx"], wd.E, wd.R, cap, t["cnt"], t["ntr"], t["itr"], t["off"], handle=h,
                                     stream=stream),
        lambda: ep.ep_dispatch(h, t["x"], ep.EP_DTYPE_BF16, t["recv"], wd.E * cap, stream=stream),
        lambda: ep.ep_dispatch_ex(h, t["x"], t["recv"], wd.E * cap, out_dtype=ep.EP_DTYPE_BF16, overlap_layout=True,
                                  stream=stream),
        lambda: ep.ep_combine(h, y, t["out"], topk_weights=t["w"], stream=stream))
    h.destroy()
    del t, y

    # the tiny workload (T=128, H=256, E=8, top-2): the identity expert, so the
    # combine reads the dispatched rows
    tn = gi.make("tiny", seed=args.seed + rank)
    wt_, Nt = tn.w, tn.num_valid
    t = tensors(tn, Nt)
    h = ep.ep_layout(t["idx"], wt_.E, wt_.R, t["cnt"], t["ntr"], t["itr"], t["off"], stream=stream)
    out["tiny_step"] = small_step_report(
        torch, stream, flush, peak, wt_, Nt,
        f"tiny T={wt_.T} H={wt_.H} E={wt_.E} K={wt_.K} R={wt_.R}: ep_layout + ep_dispatch(bf16) + ep_combine of the "
        "dispatched rows (identity expert)",
        lambda: ep.ep_layout(t["idx"], wt_.E, wt_.R, t["cnt"], t["ntr"], t["itr"], t["off"], handle=h,
                             stream=stream),
        lambda: ep.ep_dispatch(h, t["x"], ep.EP_DTYPE_BF16, t["recv"], Nt, stream=stream),
        lambda: ep.ep_dispatch_ex(h, t["x"], t["recv"], Nt, out_dtype=ep.EP_DTYPE_BF16, overlap_layout=True,
                                  stream=stream),
        lambda: ep.ep_combine(h, t["recv"], t["out"], topk_weights=t["w"], stream=stream))
    h.destroy()
    del t, flush
    return out


def small_step_report(torch, stream, flush, peak, w, N, workload, lay, dis, dis_overlap, com):
    """Device times of a small step (layout, dispatch as the layout's
    programmatic dependent, combine) and of its kernels, from CUDA graphs of
    20 copies replayed round-robin (graph_prefix_us):
      cold: L2 emptied before every step (x, y and the routing come from
            HBM); each kernel's time is its marginal cost inside the step,
            the difference between the graphs of [flush, layout, ...] up to
            and without it; the step's is [flush, step] minus [flush];
      warm: the same without the flush (every byte already in L2), steps
            chained back to back;
      alone: 20 launches of that kernel alone, chained, warm.
    GB/s counts the algorithmic bytes; the HBM fraction is of the measured
    copy rate (a warm figure above 1 means L2 served the bytes)."""
    T, K, H, E, R = w.T, w.K, w.H, w.E, w.R
    nbytes = {"layout": bytes_layout(T, K, E, R), "dispatch": bytes_dispatch_bf16(T, K, H, N),
              "combine": bytes_combine(T, K, H, N)}
    nbytes["step"] = sum(nbytes.values())
    f_, fl, fld, flc = graph_prefix_us(torch, stream, [
        flush, lambda: (flush(), lay()), lambda: (flush(), lay(), dis_overlap()),
        lambda: (flush(), lay(), dis_overlap(), com())])
    wl, wld, wlc = graph_prefix_us(torch, stream, [lay, lambda: (lay(), dis_overlap()),
                                                   lambda: (lay(), dis_overlap(), com())])
    al, ad, ac = graph_prefix_us(torch, stream, [lay, dis, com])
    cold = {"layout": fl - f_, "dispatch": fld - fl, "combine": flc - fld, "step": flc - f_}
    warm = {"layout": wl, "dispatch": wld - wl, "combine": wlc - wld, "step": wlc}
    alone = {"layout": al, "dispatch": ad, "combine": ac}
    rep = {"workload": workload, "N": N,
           "timing": "CUDA graphs of 20 copies, replayed round-robin 30 times, median; cold = L2 emptied "
                     f"({flush.mib} MiB written, then {flush.mib} MiB read) before every step, kernel times are "
                     "marginal costs inside the step; warm = no flush, steps chained; alone = 20 chained launches "
                     "of one kernel, warm",
           "flush_us": round(f_, 2)}
    for name in ("layout", "dispatch", "combine", "step"):
        b = nbytes[name]
        r = {"bytes": b}
        kinds = [("cold", cold[name]), ("warm", warm[name])] + ([("alone_warm", alone[name])] if name in alone else [])
        for kind, us in kinds:
            r[f"us_{kind}"] = round(us, 2)
            if name != "layout":
                r[f"gbs_{kind}"] = round(b / us / 1e3, 1)
                r[f"frac_of_measured_hbm_{kind}"] = round(b / us / 1e3 / peak, 4)
        if name == "step":
            r["tokens_per_s_cold"] = round(T / (cold[name] * 1e-6), 1)
            r["tokens_per_s_warm"] = round(T / (warm[name] * 1e-6), 1)
        rep[name] = r
    return rep


def e2e_measure(torch, ep, dev, inp, args, stream):
    """The same step through the public C ABI with HOST buffers: topk_idx,
    weights, x and y live in pinned host memory and out is written to pinned
    host memory. The kernels read and write those buffers directly over
    NVLink-C2C (unified addressing), so every step's host-to-device input
    traffic and device-to-host result traffic happen inside the timed region,
    without separate copies. Only the receive buffer lives in HBM."""
    w = inp.w
    T, H, E, K, R, N = w.T, w.H, w.E, w.K, w.R, inp.num_valid
    h_idx = torch.from_numpy(inp.topk_idx).pin_memory()
    h_w = torch.from_numpy(inp.topk_weights).pin_memory()
    h_x = torch.from_numpy(inp.x.view(np.int16)).pin_memory()
    h_y = torch.from_numpy(inp.y.view(np.int16)).pin_memory()
    h_out = torch.empty((T, H), dtype=torch.int16).pin_memory()
    with torch.cuda.stream(stream):
        cnt = torch.empty(E, dtype=torch.int32, device=dev)
        ntr = torch.empty(R, dtype=torch.int32, device=dev)
        itr = torch.empty(T, R, dtype=torch.uint8, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        recv = torch.empty(N, H, dtype=torch.int16, device=dev)
    stream.synchronize()
    handle = ep.ep_layout(h_idx, E, R, cnt, ntr, itr, off, stream=stream)

    def one():
        ep.ep_layout(h_idx, E, R, cnt, ntr, itr, off, handle=handle, stream=stream)
        ep.ep_dispatch(handle, h_x, ep.EP_DTYPE_BF16, recv, N, stream=stream)
        ep.ep_combine(handle, h_y, h_out, topk_weights=h_w, stream=stream)

    for _ in range(3):
        one()
    stream.synchronize()
    steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    stream.synchronize()
    handle.destroy()
    h2d = h_idx.numel() * 8 + h_w.numel() * 4 + h_x.numel() * 2 + h_y.numel() * 2
    return {"ms_per_step": e0.elapsed_time(e1) / steps, "h2d": h2d, "d2h": h_out.numel() * 2, "steps": steps,
            "how": "pinned host buffers passed to the C ABI; kernels access them over NVLink-C2C"}


# ---------------------------------------------------------------- CPU oracle

def _oracle_step(oracle, inp):
    w = inp.w
    L = oracle.layout(inp.topk_idx, w.E, w.R)
    N = int(L["expert_offsets"][-1])
    oracle.dispatch_bf16(inp.x, L["row_of_slot"], N)
    oracle.combine(inp.y, L["row_of_slot"], inp.topk_weights)
    w = inp.w
    return (bytes_layout(w.T, w.K, w.E, w.R) + bytes_dispatch_bf16(w.T, w.K, w.H, N)
            + bytes_combine(w.T, w.K, w.H, N))


def cpu_baseline(budget_s: float = 15.0):
    """The oracle as it stands (single-threaded C) on the prefill workload:
    whole steps (or a token sample if one step exceeds the budget), repeated
    to fill about `budget_s` seconds; GB/s of the same algorithmic bytes."""
    import oracle

    oracle.build()
    probe = gi.make(WORKLOAD, seed=0, T=256)
    t0 = time.perf_counter()
    _oracle_step(oracle, probe)
    dt = max(time.perf_counter() - t0, 1e-3)
    full_T = gi.WORKLOADS[WORKLOAD].T
    T_s = int(min(full_T, max(256, 256 * budget_s / dt)))
    T_s -= T_s % 64
    sample = gi.make(WORKLOAD, seed=0, T=T_s)
    nbytes, reps = 0, 0
    t0 = time.perf_counter()
    while True:
        nbytes += _oracle_step(oracle, sample)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or reps >= 50:
            break
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "host_cores": host_cores(),
            "sample": f"prefill recipe (seed 0), T={T_s} of {full_T} tokens, layout + bf16 dispatch + combine, "
                      f"{reps} repetition(s) in {dt:.1f} s, single-threaded"}


def reference_arm(args, rank, world):
    """The oracle timed on the host cores, one bounded token sample per step."""
    if rank != 0:
        return
    import oracle

    oracle.build()
    per_step_budget = max(0.05, args.ref_budget / max(1, args.steps + args.warmup))
    probe = gi.make(WORKLOAD, seed=0, T=128)
    t0 = time.perf_counter()
    _oracle_step(oracle, probe)
    dt = max(time.perf_counter() - t0, 1e-3)
    T_s = int(min(gi.WORKLOADS[WORKLOAD].T, max(16, 128 * per_step_budget / dt)))
    sample = gi.make(WORKLOAD, seed=0, T=T_s)
    for _ in range(args.warmup):
        _oracle_step(oracle, sample)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += _oracle_step(oracle, sample)
    dt = time.perf_counter() - t0
    val = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64; recipe in gen/inputs.py)",
        "config": {"workload": "prefill dispatch+combine: T=8192 H=7168 E=256 K=8 R=8 (token sample per step)",
                   "T_sample": T_s},
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "host_cores": host_cores(),
                         "sample": f"T={T_s} tokens of the prefill recipe per step, single-threaded C oracle"},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def case_arm(args):
    """One workload's step only (layout; dispatch as its programmatic
    dependent reading x during the layout, as the timed step does -- fp8 e4m3
    for the fp8 recipe, bf16 otherwise; combine), W + K times with a
    synchronize around the K: a small, single-workload program for profiler
    captures. It prints the mean step time; it is not the benchmark line."""
    import torch

    import combine_get_dispatch_layout_gb300 as ep

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ep.lib()
    inp = gi.make(args.case, seed=args.seed, T=args.tokens)
    w, N = inp.w, inp.num_valid
    fp8 = args.case == "fp8"
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        idx = torch.from_numpy(inp.topk_idx).to(dev)
        x = torch.from_numpy(inp.x.view(np.int16)).to(dev)
        wt = torch.from_numpy(inp.topk_weights).to(dev)
        y = torch.from_numpy(inp.y.view(np.int16)).to(dev) if w.y != "identity" else None
        o = [torch.empty(w.E, dtype=torch.int32, device=dev), torch.empty(w.R, dtype=torch.int32, device=dev),
             torch.empty(w.T, w.R, dtype=torch.uint8, device=dev), torch.empty(w.E + 1, dtype=torch.int32, device=dev)]
        recv = torch.empty(N, w.H, dtype=torch.uint8 if fp8 else torch.int16, device=dev)
        sc = torch.empty(N, w.H // 128, dtype=torch.float32, device=dev) if fp8 else None
        out = torch.empty(w.T, w.H, dtype=torch.int16, device=dev)
    s.synchronize()
    h = ep.ep_layout(idx, w.E, w.R, *o, stream=s)

    def step():
        ep.ep_layout(idx, w.E, w.R, *o, handle=h, stream=s)
        ep.ep_dispatch_ex(h, x, recv, N, out_dtype=ep.EP_DTYPE_FP8_E4M3 if fp8 else ep.EP_DTYPE_BF16,
                          recv_scales=sc, overlap_layout=True, stream=s)
        ep.ep_combine(h, recv if y is None else y, out, topk_weights=wt, y_rows=N, stream=s)

    for _ in range(args.warmup):
        step()
    s.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.steps):
        step()
    e1.record(s)
    s.synchronize()
    h.destroy()
    print(json.dumps({"case": args.case, "T": w.T, "H": w.H, "E": w.E, "K": w.K, "R": w.R, "N": N,
                      "steps": args.steps, "us_per_step": round(e0.elapsed_time(e1) / args.steps * 1e3, 2),
                      "note": "profiling driver: one workload's step, events around all steps"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=None,
                    help="token count of the recipe (default: the recipe's own; smaller only for profiling captures)")
    ap.add_argument("--case", choices=sorted(gi.WORKLOADS),
                    help="profiling driver: run only this workload's plain step (with --tokens, a smaller T)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.case:
        case_arm(args)
    elif args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        gpu_arm(args, rank, world, local)


if __name__ == "__main__":
    main()

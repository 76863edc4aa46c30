"""Benchmark of the fused MoE decode layer on GB300: microseconds per layer step and the HBM
bandwidth it sustains, on synthetic seeded inputs.

Headline workload: one full-size layer at 48 rows (8 requests x 6 rows, causal window 128,
contexts uniform in [1024, 65536], 128 experts top-6), the configuration the 60%-of-HBM
target is set on.  The same JSON line carries the 1-row and 6-row (draft, top-3,
non-causal 192-wide rows) shapes under "rows_sweep", together with the FFN launch alone at 6
and 48 rows ("ffn_launch_r6", "ffn_launch_r48": the residual from an attention output, then
the FFN seam and the MoE) and the stacked decode step (30 full-size 48-row layers with
distinct weights and KV caches, each layer's output the next one's input, one CUDA graph:
"stacked_30x48").

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

* value: device time per layer step, K steps replayed from CUDA graphs with every input
  resident in HBM; the layer's weights rotate over several distinct copies so that no step
  finds its weights in L2.
* e2e: the same step through the public C ABI from pinned host buffers (inputs copied in,
  output copied out, every step; the copies run on a second stream, overlapping the
  neighbouring steps' compute).
* roofline: the dominant kernel's algorithmic bytes per launch over its CUDA-event time.
* cpu_baseline: the CPU oracle on the host cores (a reported baseline only).
* --impl reference: the oracle, timed as it stands, is the reference arm.
Under torchrun each rank runs an independent replica (no collective in the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402

METRIC = "us per fused decode-layer step (achieved HBM GB/s vs ~8 TB/s at rows 1/6/48)"
UNIT = "us/step"
HEADLINE = "full_r48"
NOMINAL_HBM_GBS = 8000.0
KV_BYTES_READ = 516  # per cached token read: 512 e4m3 codes + f32 scale (pad not counted)


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------------------- bytes
def step_bytes(spec: dict, step: dict, topk_idx: np.ndarray) -> dict:
    """Algorithmic bytes of one step: every weight, scale and KV record it must touch, once.

    attention + shared + router + norm weights, the hit experts (D_hit x one expert's
    MXFP4 gate_up + down incl. scales), the union of each request's windows of KV records,
    the KV records written, and the hidden rows read and written."""
    wb = gen.weight_bytes(spec)
    valid = np.asarray(step["positions"].cpu()) >= 0
    d_hit = len(np.unique(topk_idx[valid]))
    pos = np.asarray(step["positions"].cpu())
    req = np.asarray(step["row_req"].cpu())
    kv_tokens = 0
    for q in np.unique(req[valid]):
        ps = pos[(req == q) & valid]
        keys = set()
        for p in ps:
            hi = p if spec["causal"] else ps.max()
            width = spec["window"] if spec["causal"] else spec["swa_width"]
            keys.update(range(max(0, hi - width + 1), hi + 1))
        kv_tokens += len(keys)
    rows = int(valid.sum())
    H = spec["hidden"]
    kv_rec = spec["kv_dim"] + 4
    b = dict(attn=wb["attn"], shared=wb["shared"], router=wb["router"], norms=wb["norms"],
             experts=d_hit * wb["expert"], kv_read=kv_tokens * kv_rec, kv_write=rows * kv_rec,
             hidden=2 * rows * H * 2)
    b["total"] = sum(b.values())
    b["d_hit"] = d_hit
    return b


def expert_gate_up_bytes(spec, d_hit, n_slots, rows):
    """Per-launch algorithmic bytes of the routed gate_up GEMM: the hit experts' MXFP4
    gate_up weights and scales, the normed rows it reads, the SwiGLU rows it writes."""
    H, I = spec["hidden"], spec["moe_inter"]
    w = 2 * I * H // 2 + 2 * I * (H // 32)
    return d_hit * w + rows * H * 2 + n_slots * I * 2


def expert_down_bytes(spec, d_hit, n_slots):
    H, I = spec["hidden"], spec["moe_inter"]
    w = H * I // 2 + H * (I // 32)
    return d_hit * w + n_slots * I * 2 + n_slots * H * 4


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) while the GPU works."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.p:
            time.sleep(0.1)
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()

    def summary(self):
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                clk, mxc = float(r[1]), float(r[2])
            except (ValueError, IndexError):
                continue
            mx = mxc
            sm.append(clk)
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        load = [c for c in sm if c > 0.5 * (mx or max(sm))] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------ ranks
def max_over_ranks(value: float, device) -> float:
    """The largest value over the ranks of the initialised process group (a job's time is
    its slowest replica's); the value itself when there is no process group."""
    if not torch.distributed.is_initialized():
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------ our arm
def _layer_copies(name, n_copies, dev, seed0=None):
    import moe_decode_layer_mxfp8_gb300 as m
    wl = gen.WORKLOADS[name]
    spec = gen.spec_of(name)
    step = gen.make_step(spec, wl, device=dev)
    spec["max_rows"] = step["rows"]
    layers = []
    base = wl["seed"] if seed0 is None else seed0
    for c in range(n_copies):
        w = gen.make_weights(spec, base + 1000 * c, device=dev)
        layers.append((m.Layer(spec, w), w))
    return spec, step, layers


def _capture(layers, step, outs, stream, n_steps):
    """A graph of n_steps layer steps rotating over the copies."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n_steps):
            lay, _ = layers[i % len(layers)]
            lay.step(step["x"], outs[i % len(layers)], step["positions"], step["row_req"],
                     step["block_table"], step["kv_cache"], stream=stream)
    return g


def measure_device(name, steps, warmup, dev, n_copies, sampler=None):
    spec, step, layers = _layer_copies(name, n_copies, dev)
    C = len(layers)
    outs = [torch.empty_like(step["x"]) for _ in range(C)]
    stream = torch.cuda.Stream(dev)
    idx = torch.empty((step["rows"], spec["topk"]), dtype=torch.int32, device=dev)
    # routing of every copy (for the bytes it touches), eager
    byte_list = []
    with torch.cuda.stream(stream):
        for c, (lay, _) in enumerate(layers):
            lay.step(step["x"], outs[c], step["positions"], step["row_req"], step["block_table"],
                     step["kv_cache"], stream=stream, topk_idx_out=idx)
            stream.synchronize()
            byte_list.append(step_bytes(spec, step, idx.cpu().numpy()))
        for lay, _ in layers:
            assert lay.status() == 0
        # one graph per layer copy holding one step, replayed once per step (a graph of 64
        # consecutive steps measured ~4 us a step slower at 48 rows)
        ones = [_capture([layers[c]], step, [outs[c]], stream, 1) for c in range(C)]
    torch.cuda.synchronize(dev)

    def run(k):
        for i in range(k):
            ones[i % C].replay()

    with torch.cuda.stream(stream):
        run(max(warmup, 3))
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        t0.record(stream)
        run(steps)
        t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(t0.elapsed_time(t1), dev)
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    us = ms * 1000.0 / steps
    # the distribution of single steps: an event before and after each of >= 100 replays
    n_rep = max(100, min(steps, 500))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(n_rep):
            ones[i % C].replay()
            evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    per = np.array([evs[i].elapsed_time(evs[i + 1]) * 1000.0 for i in range(n_rep)])
    dist = dict(replays=n_rep, median=round(float(np.median(per)), 2),
                p10=round(float(np.percentile(per, 10)), 2),
                p90=round(float(np.percentile(per, 90)), 2),
                mean=round(float(per.mean()), 2))
    # bytes per step averaged over the rotation actually run
    seq = [byte_list[i % C]["total"] for i in range(steps)]
    avg_bytes = float(np.mean(seq))
    res = dict(spec=spec, step=step, layers=layers, outs=outs, stream=stream, us=us, ms=ms,
               dist=dist,
               bytes=avg_bytes, bytes_detail=byte_list[0], d_hit=[b["d_hit"] for b in byte_list],
               launches=steps * layers[0][0].kernels_last_step(), copies=C)
    return res


STACKED_LAYERS = 30


def measure_stacked(n_layers, steps, warmup, dev):
    """The stacked decode step: n_layers full-size 48-row layers with distinct weights and
    KV caches, each layer's output the next one's input, captured as one CUDA graph.
    Returns us per stacked step and the algorithmic bytes it touches."""
    import moe_decode_layer_mxfp8_gb300 as m
    name = "full_r48"
    wl = gen.WORKLOADS[name]
    spec = gen.spec_of(name)
    step = gen.make_step(spec, wl, device=dev)
    spec["max_rows"] = step["rows"]
    caches = [step["kv_cache"]] + [step["kv_cache"].clone() for _ in range(n_layers - 1)]
    layers = [m.Layer(spec, gen.make_weights(spec, wl["seed"] + 1000 * (c + 7), device=dev))
              for c in range(n_layers)]
    xs = [step["x"].clone(), torch.empty_like(step["x"])]
    stream = torch.cuda.Stream(dev)
    idx = torch.empty((step["rows"], spec["topk"]), dtype=torch.int32, device=dev)
    total = 0.0
    d_hit = []
    with torch.cuda.stream(stream):
        for i, lay in enumerate(layers):  # eager once: routing of every layer, for its bytes
            lay.step(xs[i % 2], xs[(i + 1) % 2], step["positions"], step["row_req"],
                     step["block_table"], caches[i], stream=stream, topk_idx_out=idx)
            stream.synchronize()
            b = step_bytes(spec, step, idx.cpu().numpy())
            total += b["total"]
            d_hit.append(b["d_hit"])
        for lay in layers:
            assert lay.status() == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i, lay in enumerate(layers):
                lay.step(xs[i % 2], xs[(i + 1) % 2], step["positions"], step["row_req"],
                         step["block_table"], caches[i], stream=stream)
        for _ in range(max(3, warmup)):
            g.replay()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(steps):
            g.replay()
        t1.record(stream)
    torch.cuda.synchronize(dev)
    us = t0.elapsed_time(t1) * 1000.0 / steps
    for lay in layers:
        lay.close()
    del layers, caches, g
    torch.cuda.empty_cache()
    return dict(layers=n_layers, rows=step["rows"], us_per_step=round(us, 1),
                us_per_layer=round(us / n_layers, 2), bytes_per_step=int(total),
                hbm_gbs=round(total / us / 1e3, 1),
                frac_of_measured_copy=None, d_hit_min=int(min(d_hit)), d_hit_max=int(max(d_hit)))


def ffn_bytes(spec: dict, rows: int, d_hit: int) -> int:
    """Algorithmic bytes of one FFN launch: the FFN-seam gamma, the router, the shared
    expert, the hit experts, and the hidden rows (x and the attention output read, h
    written, the output written)."""
    wb = gen.weight_bytes(spec)
    return (2 * spec["hidden"] + wb["router"] + wb["shared"] + d_hit * wb["expert"]
            + 4 * rows * spec["hidden"] * 2)


def measure_ffn(rows, steps, warmup, dev, n_copies):
    """The FFN launch (residual from an attention output, then the FFN seam and the MoE) on
    the first `rows` rows of the 48-row step (6 rows = one request of 6 tokens), on FFN-only
    handles rotating over n_copies distinct weight sets, each launch replayed from its copy's
    one-launch CUDA graph."""
    import moe_decode_layer_mxfp8_gb300 as m
    name = "full_r48"
    wl = gen.WORKLOADS[name]
    spec = gen.spec_of(name)
    step = gen.make_step(spec, wl, device=dev)
    spec["max_rows"] = rows
    x = step["x"][:rows].contiguous()
    pos = step["positions"][:rows].contiguous()
    a = gen.make_attn_out(spec, step, seed=wl["seed"], device=dev)[:rows].contiguous()
    layers = []
    for c in range(n_copies):
        w = gen.make_weights(spec, wl["seed"] + 1000 * c, device=dev)
        w = {k: v for k, v in w.items() if k not in m.ATTN_WEIGHT_FIELDS}
        layers.append(m.Layer(spec, w))
    outs = [torch.empty_like(x) for _ in layers]
    stream = torch.cuda.Stream(dev)
    idx = torch.empty((rows, spec["topk"]), dtype=torch.int32, device=dev)
    d_hit = []
    with torch.cuda.stream(stream):
        for c, lay in enumerate(layers):
            lay.ffn_step(x, a, outs[c], pos, stream=stream, topk_idx_out=idx)
            stream.synchronize()
            d_hit.append(len(np.unique(idx.cpu().numpy())))
            assert lay.status() == 0
        # one graph per weight copy holding one launch, replayed once per launch
        gs = []
        for c, lay in enumerate(layers):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                lay.ffn_step(x, a, outs[c], pos, stream=stream)
            gs.append(g)
        for i in range(max(3, warmup)):
            gs[i % len(gs)].replay()
    torch.cuda.synchronize(dev)
    n = max(len(gs), steps)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(n):
            gs[i % len(gs)].replay()
        t1.record(stream)
    torch.cuda.synchronize(dev)
    us = t0.elapsed_time(t1) * 1000.0 / n
    byts = float(np.mean([ffn_bytes(spec, rows, d) for d in d_hit]))
    for lay in layers:
        lay.close()
    del layers, gs
    torch.cuda.empty_cache()
    return dict(rows=rows, us_per_launch=round(us, 2), hbm_gbs=round(byts / us / 1e3, 1),
                bytes_per_launch=int(byts), d_hit=d_hit, copies=n_copies)


def kernel_profile(res, dev, reps=20):
    """Per-launch CUDA-event times (eager steps, programmatic overlap off while profiling)."""
    spec, step, layers, stream = res["spec"], res["step"], res["layers"], res["stream"]
    lay0 = layers[0][0]
    n = lay0.launches_per_step()
    names = lay0.launch_names()
    per = {k: [] for k in names}
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    with torch.cuda.stream(stream):
        for e in evs:
            e.record(stream)
        for lay, _ in layers:
            lay.set_profile_events(evs)
        for i in range(reps + 3):
            lay, _ = layers[i % len(layers)]
            torch.cuda._sleep(2_000_000)  # the GPU waits here while the step is enqueued
            lay.step(step["x"], res["outs"][i % len(layers)], step["positions"], step["row_req"],
                     step["block_table"], step["kv_cache"], stream=stream)
            stream.synchronize()
            if i >= 3:
                for j, k in enumerate(names):
                    per[k].append(evs[j].elapsed_time(evs[j + 1]) * 1000.0)
        for lay, _ in layers:
            lay.set_profile_events(None)
    torch.cuda.synchronize(dev)
    return {k: float(np.mean(v)) for k, v in per.items()}


def measure_e2e(res, steps, warmup, dev):
    """Public API with host buffers: every step's inputs are copied in from pinned host memory
    and its output copied back out, all inside the timed region.  The copies run on a copy
    stream with two sets of device buffers, so that step i + 1's inputs arrive and step
    i - 1's output leaves while step i computes (each step's copies still bracket its own
    compute).  The step itself is the public call captured once per (layer copy, buffer
    set) into a CUDA graph and replayed, as a serving loop would run it."""
    spec, step, layers = res["spec"], res["step"], res["layers"]
    stream = res["stream"]
    copy = torch.cuda.Stream(dev)
    rows, H = step["rows"], spec["hidden"]
    h_in = {k: step[k].cpu().pin_memory() for k in ("x", "positions", "row_req", "block_table")}
    h_out = [torch.empty((rows, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    d_in = [{k: torch.empty_like(step[k]) for k in h_in} for _ in range(2)]
    d_out = [torch.empty_like(step["x"]) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def h2d(i):
        b = i % 2
        with torch.cuda.stream(copy):
            if used[b]:  # step i - 2 has finished reading these inputs
                copy.wait_event(ev_done[b])
            for k, t in h_in.items():
                d_in[b][k].copy_(t, non_blocking=True)
            ev_in[b].record(copy)

    graphs = {}

    def step_graph(li, b):
        if (li, b) not in graphs:
            lay, _ = layers[li]
            d = d_in[b]
            with torch.cuda.stream(stream):  # one eager call first, then the capture
                lay.step(d["x"], d_out[b], d["positions"], d["row_req"], d["block_table"],
                         step["kv_cache"], stream=stream)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                lay.step(d["x"], d_out[b], d["positions"], d["row_req"], d["block_table"],
                         step["kv_cache"], stream=stream)
            graphs[(li, b)] = g
        return graphs[(li, b)]

    for i in range(2 * len(layers)):  # every (layer copy, buffer set) the loop uses
        step_graph(i % len(layers), i % 2)
    torch.cuda.synchronize(dev)

    def compute(i):
        b = i % 2
        g = step_graph(i % len(layers), b)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[b])
            if used[b]:  # step i - 2's output has left this buffer
                stream.wait_event(ev_out[b])
            g.replay()
            ev_done[b].record(stream)
        used[b] = True

    def d2h(i):
        b = i % 2
        with torch.cuda.stream(copy):
            copy.wait_event(ev_done[b])
            h_out[b].copy_(d_out[b], non_blocking=True)
            ev_out[b].record(copy)

    def run(n):
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d(i + 1)
            compute(i)
            d2h(i)

    run(max(3, warmup))
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(copy)
    run(steps)
    t1.record(copy)
    torch.cuda.synchronize(dev)
    us = t0.elapsed_time(t1) * 1000.0 / steps
    h2d_b = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h_b = h_out[0].numel() * h_out[0].element_size()
    return dict(value=us, unit=UNIT, h2d_bytes_per_step=int(h2d_b), d2h_bytes_per_step=int(d2h_b))


def _cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


CPU_WORKLOADS = ("full_r1", "draft_r6", "full_r48")


def cpu_baseline(dev):
    """The oracle, as it stands, on the host cores (a reported baseline, not a target): one
    full layer step of each single-layer configuration (1 row, 6 draft rows, 48 rows), once
    single-threaded and once with OpenMP over every core, and the stacked 30-layer step
    extrapolated from two distinct 48-row layers on every core (x 15).  The value is the
    headline 48-row step on every core.  About 25 s of host time."""
    import oracle
    from tests.helpers import np_inputs
    oracle.build()
    cores = os.cpu_count() or 1
    per = {}
    keep = None
    for name in CPU_WORKLOADS:
        spec, wl = gen.spec_of(name), gen.WORKLOADS[name]
        w = gen.make_weights(spec, wl["seed"], device=dev)
        wn, sn = np_inputs(w, gen.make_step(spec, wl))
        del w
        d = {}
        for threads in (1, cores):
            oracle.set_threads(threads)
            t = time.perf_counter()
            out = oracle.layer(spec, wn, sn)["out"]
            d["us_1_thread" if threads == 1 else "us_all_cores"] = round(
                (time.perf_counter() - t) * 1e6, 1)
        per[name] = d
        if name == HEADLINE:
            keep = (spec, wn, sn, out)
    # the stacked step: a second 48-row layer with its own weights on the first one's output
    spec, wn, sn, out = keep
    w2 = gen.make_weights(spec, gen.WORKLOADS[HEADLINE]["seed"] + 1000, device=dev)
    wn2, _ = np_inputs(w2, {})
    del w2
    oracle.set_threads(cores)
    t = time.perf_counter()
    out1 = oracle.layer(spec, wn, sn)["out"]
    oracle.layer(spec, wn2, dict(sn, x=out1))
    two = time.perf_counter() - t
    v = per[HEADLINE]["us_all_cores"]
    return dict(value=v, unit=UNIT, cores=cores, kind="oracle", cpu_model=_cpu_model(),
                nproc=cores,
                sample=f"one full {sn['x'].shape[0]}-row layer step of the headline workload, "
                       f"OpenMP over {cores} host threads; per_workload: one step of each "
                       f"configuration single-threaded and on every core",
                per_workload=per,
                stacked_30x48_extrapolated=dict(
                    us=round(two * 15 * 1e6, 1),
                    note="two distinct 48-row layers timed on every core (the second on the "
                         "first's output), times 15: an extrapolation, not a measurement"))


# ------------------------------------------------------------------------ reference arm
REFERENCE_BUDGET_S = 120.0  # host seconds the reference arm may spend on timed steps


def run_reference(args, rank):
    """The oracle as the reference arm: timed steps of the headline workload on the host
    cores, each a full layer step (rank 0 only).  The run is bounded: one warm-up step at
    most, then up to K timed steps while the time budget lasts (at least one); the line
    reports the mean over the steps timed and says how many that was."""
    if rank != 0:
        return
    import oracle
    from tests.helpers import np_inputs
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    spec = gen.spec_of(HEADLINE)
    wl = gen.WORKLOADS[HEADLINE]
    w = gen.make_weights(spec, wl["seed"], device=dev)
    st = gen.make_step(spec, wl)
    wn, sn = np_inputs(w, st)
    cores = os.cpu_count() or 1
    oracle.build()
    oracle.set_threads(cores)
    if args.warmup > 0:
        oracle.layer(spec, wn, sn)
    timed, spent = 0, 0.0
    while timed < max(1, args.steps) and (timed == 0 or spent < REFERENCE_BUDGET_S):
        t = time.perf_counter()
        oracle.layer(spec, wn, sn)
        spent += time.perf_counter() - t
        timed += 1
    dt = spent / timed
    v = dt * 1e6
    sample = (f"{timed} of the {args.steps} requested steps timed ({REFERENCE_BUDGET_S:.0f} s "
              f"budget), each one full {st['rows']}-row layer step, OpenMP over {cores} host "
              f"threads; {min(args.warmup, 1)} warm-up step")
    line = dict(impl="reference", metric=METRIC, value=v, unit=UNIT, n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=dt * 1e3,
                higher_is_better=False, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic",
                config=dict(workload=_workload_desc(HEADLINE, spec, st["rows"]),
                            l2="n/a (host)"),
                cpu_baseline=dict(value=v, unit=UNIT, cores=cores, kind="oracle",
                                  sample=sample),
                e2e=dict(value=v, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0),
                gpu_launches=0)
    print(json.dumps(line), flush=True)


def _workload_desc(name, spec, rows):
    d = {"full_r48": "MoE decode layer, full size, 48 rows (8 requests x 6), causal window 128, "
                     "contexts U[1024,65536], 128 experts top-6",
         "full_r1": "MoE decode layer, full size, 1 row, causal window 128, context 8192, top-6",
         "draft_r6": "MoE decode layer, full size, 6 draft rows, non-causal 192-wide, "
                     "context 65536, top-3"}[name]
    return (f"{d}; hidden {spec['hidden']}, {spec['n_q_heads']}x{spec['head_dim']} q heads, "
            f"kv latent {spec['kv_dim']}, MXFP8 attention/shared, MXFP4 experts "
            f"(moe {spec['moe_inter']}, shared {spec['shared_inter']})")


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the dominant
# kernel, from an ncu capture of one launch, keyed by the md5 of the kernel's sources it was
# taken on: reported only while those are unchanged.
NCU_TRAFFIC = {
    ("full_r48", "expert_gate_up"): (503_944_448, "2472908a64ea93377cde950225ba4334"
                                                  "06e4e11ed408713cfcd80ad3695d0c0c"
                                                  "be64dae3d39c85a34e55a21d81c7b9b0"),
}


def _gemm_source_hash():
    import hashlib
    d = os.path.join(os.path.dirname(os.path.abspath(__file__)), "moe_decode_layer_mxfp8_gb300", "csrc")
    return "".join(hashlib.md5(open(os.path.join(d, f), "rb").read()).hexdigest()
                   for f in ("k_expert_tc.cu", "tc_common.cuh", "common.cuh"))


def schedule_probe():
    """The cost of one stage boundary of a layer step, both ways (csrc/probe_schedule.cu): a
    graph of n programmatically serialised launches of a kernel that only triggers and waits,
    against n grid-wide barriers inside one cooperative launch of one CTA per SM."""
    import ctypes as C
    from moe_decode_layer_mxfp8_gb300 import build
    lib = C.CDLL(build.build_probe())
    torch.cuda.init()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = dict(sms=sms, pdl_boundary_us={}, grid_barrier_us={})
    v = C.c_float(0.0)
    for ctas in (1, 48, sms, 2 * sms):  # the step's launch widths: 1 (top-k) .. 2 x SMs
        rc = lib.mono_probe_pdl_chain(64, ctas, 50, C.byref(v))
        out["pdl_boundary_us"][str(ctas)] = round(v.value, 3) if rc == 0 else f"error {rc}"
    for ctas in (sms // 2, sms):
        rc = lib.mono_probe_grid_barrier(2000, ctas, C.byref(v))
        out["grid_barrier_us"][str(ctas)] = round(v.value, 3) if rc == 0 else f"error {rc}"
    print(json.dumps(out))


def run_eager(name, n):
    """N eager layer steps (launch order: per step the slots of mono_layer_launch_name)."""
    from moe_decode_layer_mxfp8_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    spec, step, layers = _layer_copies(name, 1, dev)
    out = torch.empty_like(step["x"])
    stream = torch.cuda.Stream(dev)
    lay = layers[0][0]
    with torch.cuda.stream(stream):
        for _ in range(n):
            lay.step(step["x"], out, step["positions"], step["row_req"], step["block_table"],
                     step["kv_cache"], stream=stream)
    torch.cuda.synchronize(dev)
    if lay.status() != 0:
        raise SystemExit(f"layer status {lay.status()}")
    print(json.dumps({"eager_steps": n, "workload": name, "rows": step["rows"]}))


# ------------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--workload", default=HEADLINE, choices=["full_r48", "full_r1", "draft_r6"])
    ap.add_argument("--eager", type=int, default=0, metavar="N",
                    help="only run N eager steps of the workload (one layer copy) and exit: a "
                         "short command for ncu captures of single launches")
    ap.add_argument("--schedule-probe", action="store_true",
                    help="only measure a stage boundary as a programmatically serialised launch "
                         "and as a grid-wide barrier of one persistent launch, and exit")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.eager:
        run_eager(args.workload, args.eager)
        return
    if args.schedule_probe:
        schedule_probe()
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    from moe_decode_layer_mxfp8_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, peak_kind = _peaks()

    def copies_for(name):
        """Distinct layer copies so that the weights one rotation touches exceed 3x L2."""
        spec, wl = gen.spec_of(name), gen.WORKLOADS[name]
        wb = gen.weight_bytes(spec)
        rpr = wl["rows_per_req"]
        n_req = int(str(wl["contexts"]).split(":")[-1]) if isinstance(wl["contexts"], str) else len(wl["contexts"])
        rows = rpr * n_req if isinstance(rpr, int) else sum(rpr)
        d_hit = min(spec["n_experts"], (1 if wl.get("repeat_input") else rows) * spec["topk"])
        touched = wb["attn"] + wb["shared"] + wb["router"] + d_hit * wb["expert"]
        return max(2, int(np.ceil(3 * l2 / touched)))

    with ClockSampler(local) as clk:
        res = measure_device(args.workload, args.steps, args.warmup, dev, copies_for(args.workload))
        sweep = {}
        if not args.no_sweep:
            for name in ("full_r1", "draft_r6"):
                if name == args.workload:
                    continue
                r = measure_device(name, min(args.steps, 2000), args.warmup, dev, copies_for(name))
                sweep[name] = dict(rows=r["step"]["rows"], us_per_step=round(r["us"], 2),
                                   us_per_step_dist=r["dist"],
                                   hbm_gbs=round(r["bytes"] / r["us"] / 1e3, 1),
                                   frac_of_8tbs=round(r["bytes"] / r["us"] / 1e3 / NOMINAL_HBM_GBS, 4),
                                   bytes_per_step=int(r["bytes"]), d_hit=r["d_hit"])
                del r
                torch.cuda.empty_cache()
            # the FFN launch alone at one request x 6 tokens and at 8 requests x 6 tokens
            for r_ffn in (6, 48):
                f = measure_ffn(r_ffn, 1000, args.warmup, dev, 2 if r_ffn == 48 else 3)
                f["frac_of_measured_copy"] = round(f["hbm_gbs"] / peak, 4)
                sweep[f"ffn_launch_r{r_ffn}"] = f
            # the stacked decode step: 30 full-size 48-row layers, one graph, residual carried
            stacked = measure_stacked(STACKED_LAYERS, 20, args.warmup, dev)
            stacked["frac_of_measured_copy"] = round(stacked["hbm_gbs"] / peak, 4)
            sweep["stacked_30x48"] = stacked
    clocks = clk.summary()

    prof = kernel_profile(res, dev)
    e2e = measure_e2e(res, args.steps if args.steps <= 500 else 500, args.warmup, dev)
    spec, step = res["spec"], res["step"]
    rows = step["rows"]
    # dominant kernel and its roofline
    top = max(prof, key=prof.get)
    d_hit = res["bytes_detail"]["d_hit"]
    n_slots = rows * spec["topk"]
    if top == "expert_gate_up":
        alg = expert_gate_up_bytes(spec, d_hit, n_slots, rows)
    elif top == "expert_down":
        alg = expert_down_bytes(spec, d_hit, n_slots)
    else:
        alg = None
    roof = None
    if alg is not None:
        ach = alg / (prof[top] * 1e-6) / 1e9
        roof = dict(kernel=top, bound="hbm", achieved=round(ach, 1), peak=peak,
                    peak_kind=peak_kind, unit="GB/s", frac=round(ach / peak, 4),
                    traffic=None, bytes_per_launch=int(alg), us_per_launch=round(prof[top], 2))
        t = NCU_TRAFFIC.get((args.workload, top))
        if t is not None and t[1] == _gemm_source_hash():
            roof["traffic"] = t[0]
            roof["traffic_source"] = "ncu capture of one launch"
    total_prof = sum(prof.values())
    gbs = res["bytes"] / res["us"] / 1e3
    line = dict(
        metric=METRIC, value=round(res["us"], 3), unit=UNIT, n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=round(res["us"] / 1e3, 6), higher_is_better=False,
        scaling="weak", vs_baseline=None,
        dtype="f16 x f16 -> f32 tensor-core products of exactly decoded MXFP8/MXFP4 weights and bf16 activations",
        data="synthetic",
        config=dict(workload=_workload_desc(args.workload, spec, rows), rows=rows,
                    layer_copies=res["copies"],
                    l2=f"inputs larger than L2: weights rotate over {res['copies']} distinct layer "
                       f"copies ({res['bytes'] / 1e6:.0f} MB touched per step, L2 {l2 / 1e6:.0f} MB)",
                    graph="each step replayed from a one-step CUDA graph of programmatically "
                          "serialised launches"),
        us_per_step_dist=res["dist"],
        hbm_gbs=round(gbs, 1), frac_of_8tbs=round(gbs / NOMINAL_HBM_GBS, 4),
        frac_of_measured_copy=round(gbs / peak, 4), bytes_per_step=int(res["bytes"]),
        d_hit=res["d_hit"],
        roofline=roof,
        per_kernel_us={k: round(v, 2) for k, v in prof.items()},
        per_kernel_share={k: round(v / total_prof, 4) for k, v in prof.items()},
        rows_sweep=sweep,
        e2e={k: (round(v, 3) if isinstance(v, float) else v) for k, v in e2e.items()},
        clocks=clocks,
        gpu_launches=res["launches"],
    )
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

"""Benchmark of the block-hybrid attention step on one B300 (or N replicas).

Default workload: the continuous-batching step of one linearized layer —
64 requests with 16 heads (d=128, f=64, L=32) and prefixes of 32*U{8..128}
tokens held as fixed-size states; one hb_block_attend for all 64 requests
plus an hb_commit_block for the 16 requests that finish their block. A step
cycles through 6 independent layer instances (own W, gate, states and
activations), as the 6 linearized layers of the model would, so that a
layer's 80+ MB working set has left the 126 MB L2 by the time it comes back.

Metric: active-block tokens/s (B*L per step) and the attend kernel's HBM
GB/s against the measured peak. ``--impl reference`` times the fp64 CPU
oracle on a bounded sample of the same step instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs its own 64 requests (weak scaling); rank 0
prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "hybrid-attn active-block tokens/s and HBM GB/s vs ~8 TB/s, 1 B300"
UNIT = "tokens/s"
N_LAYERS = 6
B, H, D, FH, L, N_COMMIT = 64, 16, 128, 64, 32, 16
F = 2 * FH

# Algorithmic bytes of one hb_block_attend launch at this shape: per request
# the state S (F*d fp32) and Z (F fp32), q/k/v (3*L*H*d bf16) and o (L*H*d
# bf16); W (H*d*f bf16) once per launch.
ATTEND_BYTES_PER_REQUEST = H * (F * D * 4 + F * 4) + 4 * L * H * D * 2
ATTEND_BYTES_W = H * D * FH * 2
# hb_commit_block: read and write S and Z, read k/v; W once.
COMMIT_BYTES_PER_REQUEST = H * 2 * (F * D * 4 + F * 4) + 2 * L * H * D * 2
# hb_block_attend_commit: the attend bytes, plus the write of S and Z for each
# committing request (its state and block were already read by the attend).
STEP_BYTES = B * ATTEND_BYTES_PER_REQUEST + ATTEND_BYTES_W + N_COMMIT * H * (F * D * 4 + F * 4)
# hb_block_attend_commit_s16: a request that does not commit reads its bf16
# copy of S (F*d bf16) instead of the fp32 master; a committing one reads the
# master and writes the new master, Z and the new copy.
ATTEND_S16_BYTES_PER_REQUEST = H * (F * D * 2 + F * 4) + 4 * L * H * D * 2
DUAL_STEP_BYTES = ((B - N_COMMIT) * ATTEND_S16_BYTES_PER_REQUEST + ATTEND_BYTES_W
                   + N_COMMIT * (ATTEND_BYTES_PER_REQUEST + H * (F * D * 4 + F * 4) + H * F * D * 2))


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_ms: float, local_units: float, world: int):
    """Max of the per-rank step times and sum of the units over ranks."""
    if world == 1:
        return local_ms, local_units
    import torch.distributed as dist

    t = torch.tensor([local_ms], dtype=torch.float64)
    u = torch.tensor([local_units], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t, u = t.cuda(), u.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def _barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running; every
    sample keeps its host time, so a summary can cover one window."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []  # (host time, csv line)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 5.0:  # sampler is up
                time.sleep(0.02)
        except (OSError, ValueError):
            self.proc = None
        return self

    def mark(self):
        """Start of the window of interest: earlier samples are dropped."""
        self.samples = []

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float = None, t1: float = None):
        """Median SM clock, max clock and the throttle reasons seen, over the
        samples taken between host times t0 and t1 (all samples if None)."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in list(self.samples):
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, "fallback"


def _traffic(kernel: str):
    """Per-launch DRAM bytes of ``kernel`` from the committed ncu summary, if
    the summary was taken on the kernel source as it is now."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    from linear_attention_diffusion_feature_b300 import build

    if rec.get("source_sha") != build.source_digest(rec.get("sources")):
        return None
    return rec.get("bytes_per_launch")


def make_layers(device, rank=0):
    """6 independent layer instances of the continuous-batching workload, with
    states built by hb_prefill_state from each layer's own prefixes. Each rank
    draws its own requests (rank 0 keeps the single-GPU seeds)."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    layers = []
    cfg = hb.Config(H, D, FH, L, dtype=hb.DTYPE_BF16, merge=hb.MERGE_SHARED_NORM)
    for layer in range(N_LAYERS):
        w = inputs.continuous_batching(seed=2 + 100 * layer + 100000 * rank, device=device, B=B,
                                       n_commit=N_COMMIT)
        t = w.tensors
        S = torch.empty((B, H, F, D), dtype=torch.float32, device=device)
        Z = torch.empty((B, H, F), dtype=torch.float32, device=device)
        sl = torch.arange(B, dtype=torch.int32, device=device)
        hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                            w.meta["max_prefix"], t["W"], S, Z)
        ci = t["commit_idx"]
        mask = torch.zeros(B, dtype=torch.int32, device=device)
        mask[ci] = 1
        layers.append(dict(mask=mask,
            W=t["W"], gate=t["gate"], q=t["q"], k=t["k"], v=t["v"], S=S, Z=Z, slots=sl,
            o=torch.empty_like(t["q"]), commit_slots=sl[ci].contiguous(),
            commit_k=t["k"][ci].contiguous(), commit_v=t["v"][ci].contiguous(),
            mean_prefix=float(w.meta["total_prefix"]) / B))
        del t["prefix_k"], t["prefix_v"]
    torch.cuda.synchronize()
    assert hb.hb_get_device_status() == 0
    return cfg, layers


GRAPH_STEPS = 600  # most steps captured into one CUDA graph


class StepGraphs:
    """CUDA graphs of consecutive steps ``fn(0), fn(1), ...`` (the layer of
    step i is i mod N_LAYERS), so that any number of steps runs as a few graph
    replays with the host out of the loop: a graph of GRAPH_STEPS steps and
    one of the remainder."""

    def __init__(self, fn, n_steps: int):
        self.fn = fn
        self.full = self._capture(GRAPH_STEPS) if n_steps >= GRAPH_STEPS else None
        rem = n_steps % GRAPH_STEPS
        self.rem = self._capture(rem) if rem else None
        self.n_full = n_steps // GRAPH_STEPS

    def _capture(self, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                self.fn(i)
        return g

    def replay(self):
        for _ in range(self.n_full):
            self.full.replay()
        if self.rem is not None:
            self.rem.replay()


def _busy(graph: "StepGraphs", seconds: float, per_replay_ms: float):
    """Replays ``graph`` for about ``seconds`` of device time (no sync), to keep
    the GPU under the step's load around a short timed region."""
    n = max(1, int(seconds * 1e3 / max(per_replay_ms, 1e-3)))
    for _ in range(n):
        graph.replay()


def _timed_replays(graph: "StepGraphs", n: int, stream) -> float:
    """Device time of ``n`` replays of ``graph`` between two events (ms)."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def run_ours(args, world, rank, local):
    import linear_attention_diffusion_feature_b300 as hb

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    cfg, layers = make_layers(device, rank)
    mean_prefix = layers[0]["mean_prefix"]
    stream = torch.cuda.current_stream()

    def step(i):
        # attend for all 64 requests, then commit of the 16 whose block is
        # finished, in one pass over the state
        ly = layers[i % N_LAYERS]
        hb.hb_block_attend_commit(cfg, ly["slots"], ly["q"], ly["k"], ly["v"], ly["S"], ly["Z"],
                                  ly["W"], ly["gate"], ly["mask"], o=ly["o"])

    def attend_only(i):
        ly = layers[i % N_LAYERS]
        hb.hb_block_attend(cfg, ly["slots"], ly["q"], ly["k"], ly["v"], ly["S"], ly["Z"],
                           ly["W"], ly["gate"], o=ly["o"])

    # Warm-up steps through the binding, then the timed K steps captured into
    # CUDA graphs (one graph of up to GRAPH_STEPS consecutive steps, layers in
    # turn), so the timed region measures the device and not Python's launch
    # overhead (~10 us per call through ctypes) and has no gaps between
    # replays. A graph of GRAPH_STEPS steps keeps the GPU under the same load
    # for ~0.3 s before and after the timed region, so that the clock samples
    # (every 50 ms) describe the conditions the timed steps ran in, however
    # short the timed region is.
    nvtx = torch.cuda.nvtx  # ranges for profilers (ncu --nvtx-include "timed/")
    nvtx.range_push("warmup")
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    timed = StepGraphs(step, args.steps)
    filler = StepGraphs(step, GRAPH_STEPS)
    timed.replay()
    filler_ms = _timed_replays(filler, 1, stream)
    nvtx.range_pop()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        _barrier(world)
        torch.cuda.synchronize()
        clocks.mark()
        t_begin = time.time()
        _busy(filler, 0.3, filler_ms)
        nvtx.range_push("timed")
        start.record(stream)
        timed.replay()
        end.record(stream)
        nvtx.range_pop()
        _busy(filler, 0.3, filler_ms)
        torch.cuda.synchronize()
        t_end = time.time()
        _barrier(world)
        step_clocks = clocks.summary(t_begin, t_end)
        total_ms = start.elapsed_time(end)
        # each step is one launch of the step kernel, so its average launch
        # duration is the timed region over K
        step_launch_ms = total_ms / args.steps

        # attend-only launches (hb_block_attend) for comparison, over >= 0.5 s
        nvtx.range_push("attend_only")
        attend_graph = StepGraphs(attend_only, GRAPH_STEPS)
        attend_graph.replay()
        one = _timed_replays(attend_graph, 1, stream)
        n_rep = max(1, int(500.0 / one) + 1)
        t0 = time.time()
        attend_only_ms = _timed_replays(attend_graph, n_rep, stream) / (n_rep * GRAPH_STEPS)
        attend_clocks = clocks.summary(t0, time.time())
        nvtx.range_pop()
        del attend_graph
    status = hb.hb_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {hb.hb_status_string(status)}")
    ms_per_step, units = aggregate(total_ms / args.steps, B * L, world)
    value = units / (ms_per_step / 1e3)

    achieved = STEP_BYTES / (step_launch_ms / 1e3) / 1e9
    attend_bytes = B * ATTEND_BYTES_PER_REQUEST + ATTEND_BYTES_W
    peak, peak_kind = _peaks()

    nvtx.range_push("e2e")
    e2e = run_e2e(args, cfg, layers, device)
    nvtx.range_pop()
    nvtx.range_push("dual_copy")
    dual = component_dual_copy(args, cfg, layers, stream)
    step_layers = component_step_layers(args, cfg, layers, stream) if world == 1 else None
    nvtx.range_pop()
    del layers
    torch.cuda.empty_cache()

    components = {
        "step_launch_ms": step_launch_ms,
        "attend_only_launch_ms": attend_only_ms,
        "attend_only_hbm_frac": attend_bytes / (attend_only_ms / 1e3) / 1e9 / peak,
        "attend_only_timing": f"{n_rep} replays of a {GRAPH_STEPS}-launch CUDA graph "
                              f"({n_rep * GRAPH_STEPS} launches, >= 0.5 s)",
        "attend_only_clocks": attend_clocks,
        "commit_cost_ms": step_launch_ms - attend_only_ms,
        "step_dual_copy": dual,
        "step_6_layers_one_launch": step_layers,
    }
    if world == 1 and not args.no_components:
        nvtx.range_push("components")
        components["stack_b256"] = component_stack(args, device)
        components["prefill_8x8192"] = component_prefill(args, device)
        components["prompt_with_outputs_8x8192"] = component_prefill_attend(args, device)
        nvtx.range_pop()

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": "continuous-batching step of one linearized layer: 64 requests, "
                        "16 heads, d=128, f=64 (F=128), L=32, prefixes 32*U{8..128} tokens as "
                        "fp32 states; attend all 64 + commit 16 (hb_block_attend_commit)",
            "batch": B, "block_len": L, "heads": H, "head_dim": D, "feat_half": FH,
            "commit_per_step": N_COMMIT, "merge": "shared_norm",
            "mean_prefix_tokens": mean_prefix,
            "l2": f"steps cycle through {N_LAYERS} independent layer instances "
                  f"({N_LAYERS} x ~{(B * ATTEND_BYTES_PER_REQUEST) / 1e6:.0f} MB > 126 MB L2)",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "kernel": "hb_block_attend_commit (k_attend_fast)", "bound": "hbm",
            "achieved": achieved, "peak": peak,
            "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
            "algorithmic_bytes_per_launch": STEP_BYTES,
            "launch_ms": step_launch_ms,
            "traffic": _traffic("hb_block_attend_commit"),
        },
        "components": components,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "timing": f"the K steps are one launch each, captured into CUDA graphs of up to "
                  f"{GRAPH_STEPS} consecutive steps (layers in turn) and timed by events around "
                  f"their replay; 0.3 s of the same steps run before and after, untimed",
        "clocks": dict(step_clocks, window="samples every 50 ms over the timed region and the "
                                           "0.3 s of identical steps on either side"),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(max_seconds=args.cpu_seconds)
    return line


def component_dual_copy(args, cfg, layers, stream):
    """The same continuous-batching step on a pool that keeps a bf16 copy of
    S beside each fp32 master: hb_block_attend_commit_s16 reads the copy for
    the 48 requests that do not commit and the master for the 16 that do,
    and writes the committing ones' new masters and copies (same output bits
    as the fp32 step). For comparison, the same step built from the attend on
    the copies plus a separate commit and copy refresh of the committing
    slots (three launches). Each timed over >= 0.5 s of graph replays."""
    import linear_attention_diffusion_feature_b300 as hb

    peak, _ = _peaks()
    for ly in layers:
        ly["S16"] = torch.empty(ly["S"].shape, dtype=torch.bfloat16, device=ly["S"].device)
        hb.hb_state_to_bf16(cfg, ly["slots"], ly["S"], ly["S16"])

    def dual_step(i):
        ly = layers[i % N_LAYERS]
        hb.hb_block_attend_commit_s16(cfg, ly["slots"], ly["q"], ly["k"], ly["v"], ly["S"],
                                      ly["S16"], ly["Z"], ly["W"], ly["gate"], ly["mask"],
                                      o=ly["o"])

    def refresh_step(i):
        ly = layers[i % N_LAYERS]
        hb.hb_block_attend_s16(cfg, ly["slots"], ly["q"], ly["k"], ly["v"], ly["S16"], ly["Z"],
                               ly["W"], ly["gate"], o=ly["o"])
        hb.hb_commit_block(cfg, ly["commit_slots"], ly["commit_k"], ly["commit_v"], ly["W"],
                           ly["S"], ly["Z"])
        hb.hb_state_to_bf16(cfg, ly["commit_slots"], ly["S"], ly["S16"])

    out = {}
    for name, fn, launches in (("fused", dual_step, 1), ("attend_commit_refresh", refresh_step, 3)):
        for i in range(args.warmup):
            fn(i)
        g = StepGraphs(fn, GRAPH_STEPS)
        g.replay()
        one = _timed_replays(g, 1, stream)
        n_rep = max(1, int(500.0 / one) + 1)
        out[name + "_ms"] = _timed_replays(g, n_rep, stream) / (n_rep * GRAPH_STEPS)
        out[name + "_launches_per_step"] = launches
        del g
    assert hb.hb_get_device_status() == 0
    for ly in layers:
        del ly["S16"]
    ms = out["fused_ms"]
    out.update({
        "tokens_per_s": B * L / (ms / 1e3),
        "algorithmic_bytes_per_launch": DUAL_STEP_BYTES,
        "hbm_frac": DUAL_STEP_BYTES / (ms / 1e3) / 1e9 / peak,
        "timing": "graphs of 600 steps (layers in turn), replayed for >= 0.5 s each",
    })
    return out


def component_step_layers(args, cfg, layers, stream):
    """The 6 layer instances' continuous-batching steps (64 requests each, 16
    committing) as one launch of hb_block_attend_commit_layers: the layers'
    requests, pools, maps, gates and commit masks side by side (copies, so the
    per-layer instances are untouched). For layers whose steps are ready
    together; in a forward pass the layers run in turn. Graphs of 100
    launches, replayed for >= 0.5 s."""
    import linear_attention_diffusion_feature_b300 as hb

    peak, _ = _peaks()
    qa, ka, va = (torch.cat([ly[n] for ly in layers]) for n in ("q", "k", "v"))
    Wa = torch.stack([ly["W"] for ly in layers])
    ga = torch.stack([ly["gate"] for ly in layers])
    Sa = torch.cat([ly["S"] for ly in layers])
    Za = torch.cat([ly["Z"] for ly in layers])
    n_sl = layers[0]["S"].shape[0]
    sla = torch.cat([ly["slots"] + i * n_sl for i, ly in enumerate(layers)]).to(torch.int32)
    ma = torch.cat([ly["mask"] for ly in layers])
    oa = torch.empty_like(qa)

    def step():
        hb.hb_block_attend_commit_layers(cfg, sla, qa, ka, va, Sa, Za, Wa, ga, ma, o=oa)

    for _ in range(args.warmup):
        step()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(100):
            step()
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    n_rep = max(1, int(500.0 / a.elapsed_time(b)) + 1)
    a.record(stream)
    for _ in range(n_rep):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (n_rep * 100)
    assert hb.hb_get_device_status() == 0
    nbytes = N_LAYERS * STEP_BYTES  # each layer's W is read once, as in one layer's step
    del g, qa, ka, va, Wa, ga, Sa, Za, sla, ma, oa
    torch.cuda.empty_cache()
    return {"workload": "6 layers x (64 requests, 16 committing) in one launch",
            "ms": ms, "per_layer_ms": ms / N_LAYERS,
            "tokens_per_s": N_LAYERS * B * L / (ms / 1e3),
            "algorithmic_bytes_per_launch": nbytes,
            "hbm_frac": nbytes / (ms / 1e3) / 1e9 / peak,
            "timing": "graphs of 100 launches, replayed for >= 0.5 s"}


def component_stack(args, device, nB: int = 256, P: int = 2048):
    """The largest single-GPU stack configuration: 6 linearized layers at 256
    requests with 2,048-token prefixes, one stack step = 6 hb_block_attend
    launches, against hb_softmax_kv_attend of the same 6 layers over the same
    prefixes kept as a KV cache; each stack step is one CUDA graph, timed over
    many replays."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    cfg = hb.Config(H, D, FH, L)
    stream = torch.cuda.current_stream()
    peak, _ = _peaks()
    layers = []
    for layer in range(N_LAYERS):
        w = inputs.stack_layer(layer, nB, device=device, P=P)
        t = w.tensors
        S = torch.empty((nB, H, F, D), dtype=torch.float32, device=device)
        Z = torch.empty((nB, H, F), dtype=torch.float32, device=device)
        sl = torch.arange(nB, dtype=torch.int32, device=device)
        hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"], P, t["W"], S, Z)
        need = hb.hb_softmax_kv_workspace_size(cfg, nB, P)
        layers.append(dict(t=t, S=S, Z=Z, sl=sl, o=torch.empty_like(t["q"]),
                           ws=torch.empty(max(need, 16), dtype=torch.uint8, device=device)))
    torch.cuda.synchronize()

    def hybrid():
        for ly in layers:
            t = ly["t"]
            hb.hb_block_attend(cfg, ly["sl"], t["q"], t["k"], t["v"], ly["S"], ly["Z"], t["W"],
                               t["gate"], o=ly["o"])

    def softmax():
        for ly in layers:
            t = ly["t"]
            hb.hb_softmax_kv_attend(cfg, t["prefix_k"], t["prefix_v"], t["cu_prefix"], P, t["q"],
                                    t["k"], t["v"], o=ly["o"], workspace=ly["ws"])

    # the same 6 layers as one launch (attend only), side by side
    qa, ka, va = (torch.cat([ly["t"][n] for ly in layers]) for n in ("q", "k", "v"))
    Wa = torch.stack([ly["t"]["W"] for ly in layers])
    ga = torch.stack([ly["t"]["gate"] for ly in layers])
    Sa = torch.cat([ly["S"] for ly in layers])
    Za = torch.cat([ly["Z"] for ly in layers])
    sla = torch.arange(N_LAYERS * nB, dtype=torch.int32, device=device)
    oa = torch.empty_like(qa)

    def hybrid_layers():
        hb.hb_block_attend_commit_layers(cfg, sla, qa, ka, va, Sa, Za, Wa, ga, None, o=oa)

    h_ms = _graph_ms(hybrid, 1, 800, args.warmup, stream)       # ~0.3 s
    hl_ms = _graph_ms(hybrid_layers, 1, 800, args.warmup, stream)
    s_ms = _graph_ms(softmax, 1, 80, args.warmup, stream)       # ~0.3 s
    assert hb.hb_get_device_status() == 0
    hb_bytes = N_LAYERS * (nB * ATTEND_BYTES_PER_REQUEST + ATTEND_BYTES_W)
    sm_bytes = N_LAYERS * nB * ((P + L) * H * D * 2 * 2 + 2 * L * H * D * 2)
    del layers, qa, ka, va, Wa, ga, Sa, Za, oa
    torch.cuda.empty_cache()
    return {"workload": f"6-layer stack, B={nB}, P={P}", "hybrid_ms": h_ms,
            "hybrid_layers_ms": hl_ms,
            "hybrid_layers_hbm_frac": hb_bytes / (hl_ms / 1e3) / 1e9 / peak,
            "hybrid_tokens_per_s": nB * L / (h_ms / 1e3),
            "hybrid_hbm_frac": hb_bytes / (h_ms / 1e3) / 1e9 / peak,
            "softmax_kv_ms": s_ms, "softmax_kv_tokens_per_s": nB * L / (s_ms / 1e3),
            "softmax_kv_hbm_frac": sm_bytes / (s_ms / 1e3) / 1e9 / peak,
            "speedup": s_ms / h_ms,
            "timing": "one stack step (6 launches, or one for hybrid_layers) per CUDA graph; "
                      "800 (hybrid) and 80 (softmax) replays between two events"}


def component_prefill(args, device):
    """Prompt ingestion (8 prompts x 8,192 tokens), one hb_prefill_state call
    per CUDA graph, timed over ~0.3 s of replays."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    w = inputs.prompt_ingestion(device=device)
    t = w.tensors
    nB, T = w.meta["B"], w.meta["T"]
    cfg = hb.Config(H, D, FH, L)
    S = torch.empty((nB, H, F, D), dtype=torch.float32, device=device)
    Z = torch.empty((nB, H, F), dtype=torch.float32, device=device)
    sl = torch.arange(nB, dtype=torch.int32, device=device)
    need = hb.hb_prefill_workspace_size(cfg, nB, T)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)

    def call():
        hb.hb_prefill_state(cfg, sl, t["k"], t["v"], t["cu_seqlens"], T, t["W"], S, Z,
                            workspace=ws)

    ms = _graph_ms(call, 1, 2000, args.warmup, torch.cuda.current_stream())
    assert hb.hb_get_device_status() == 0
    tokens = nB * T
    nbytes = 2 * tokens * H * D * 2 + nB * H * (F * D + F) * 4 + H * D * FH * 2
    flops = tokens * H * (2 * D * FH + 2 * 2 * F * D)
    peak, _ = _peaks()
    tpeak, _ = _tensor_peak()
    del w, t, S, Z, ws
    torch.cuda.empty_cache()
    return {"workload": "hb_prefill_state, 8 prompts x 8,192 tokens, overwrite", "ms": ms,
            "tokens_per_s": tokens / (ms / 1e3),
            "hbm_frac": nbytes / (ms / 1e3) / 1e9 / peak,
            "tensor_frac": flops / (ms / 1e3) / 1e12 / tpeak,
            "timing": "one call per CUDA graph, 2000 replays between two events"}


def component_prefill_attend(args, device):
    """Prompt processing with outputs (8 prompts x 8,192 tokens, from empty
    states): one hb_prefill_attend call per CUDA graph, 20 replays."""
    r = _prefill_attend(args, device, 8, 8192, 20)
    return {"workload": "hb_prefill_attend, 8 prompts x 8,192 tokens, from empty states",
            "ms": r["ms"], "tokens_per_s": r["tokens"] / (r["ms"] / 1e3),
            "hbm_frac": r["achieved"] / r["peak"], "traffic": _traffic("hb_prefill_attend"),
            "timing": "one call (a state reset and the prompt kernel) per CUDA graph, "
                      "20 replays between two events"}


def run_e2e(args, cfg, layers, device):
    """Same step through the binding with pinned host buffers: every step
    copies that step's activations and per-request metadata host->device and
    reads o back. As a serving loop would, the copies run on their own
    streams, so step i's kernel overlaps step i+1's upload and step i-1's
    download (device inputs and host outputs are double-buffered); the timed
    region spans every copy and kernel of every step. A layer's output buffer
    is written again only after the download of its previous contents."""
    import linear_attention_diffusion_feature_b300 as hb

    ly0 = layers[0]
    # the step's block tokens and its per-request metadata (state slots and
    # the commit mask) come from the host each step
    names = ("q", "k", "v", "slots", "mask")
    host = {name: ly0[name].cpu().pin_memory() for name in names}
    host_o = [torch.empty_like(host["q"]).pin_memory() for _ in range(2)]
    dev = [{name: torch.empty_like(ly0[name]) for name in names} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host_o[0].numel() * host_o[0].element_size()
    up, comp, down = torch.cuda.Stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device)
    n_steps = min(args.steps, 200)
    total = args.warmup + n_steps
    uploaded = [torch.cuda.Event() for _ in range(total)]
    computed = [torch.cuda.Event() for _ in range(total)]
    downloaded = [torch.cuda.Event() for _ in range(total)]

    def step(i):
        ly = layers[i % N_LAYERS]
        buf = dev[i % 2]
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(computed[i - 2])  # the kernel that read this buffer is done
            for name in names:
                buf[name].copy_(host[name], non_blocking=True)
            uploaded[i].record(up)
        with torch.cuda.stream(comp):
            comp.wait_event(uploaded[i])
            if i >= N_LAYERS:
                # the previous download of this layer's output buffer is done
                comp.wait_event(downloaded[i - N_LAYERS])
            hb.hb_block_attend_commit(cfg, buf["slots"], buf["q"], buf["k"], buf["v"], ly["S"],
                                      ly["Z"], ly["W"], ly["gate"], buf["mask"], o=ly["o"])
            computed[i].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(computed[i])
            if i >= 2:
                down.wait_event(downloaded[i - 2])  # host buffer i % 2 is free again
            host_o[i % 2].copy_(ly["o"], non_blocking=True)
            downloaded[i].record(down)

    torch.cuda.synchronize()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(up)
    comp.wait_event(start)
    down.wait_event(start)
    for i in range(args.warmup, total):
        step(i)
    end.record(down)  # after the last download, which waits on every stream's last work
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / n_steps
    last = total - 1
    # the last download holds that step's own output
    assert torch.equal(host_o[last % 2], layers[last % N_LAYERS]["o"].cpu())
    return {"value": B * L / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "overlap": "upload, kernel and download on separate streams"}


# ------------------------------------------------------ other workloads

def _timed(fn, steps, warmup, stream):
    """CUDA-event time of each of ``steps`` calls of ``fn`` after ``warmup``
    untimed calls; returns the per-call times in ms."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def _graph_ms(fn, per_graph, replays, warmup, stream):
    """Device time per call of ``fn`` with the host out of the loop: ``fn`` is
    called ``warmup`` times, then ``per_graph`` calls are captured into one CUDA
    graph, which is replayed ``replays`` times between two events."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            fn()
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(replays):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (replays * per_graph)


def _median(xs):
    ys = sorted(xs)
    return ys[len(ys) // 2]


def _tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1800.0, "fallback"


def run_prefill(args):
    """Prompt ingestion: 8 prompts x 8,192 tokens, 16 heads, d=128, f=64,
    overwrite S/Z (k, v are 537 MB, well above the 126 MB L2)."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = inputs.prompt_ingestion(device=device)
    t = w.tensors
    nB, T = w.meta["B"], w.meta["T"]
    cfg = hb.Config(H, D, FH, L)
    S = torch.empty((nB, H, F, D), dtype=torch.float32, device=device)
    Z = torch.empty((nB, H, F), dtype=torch.float32, device=device)
    sl = torch.arange(nB, dtype=torch.int32, device=device)
    need = hb.hb_prefill_workspace_size(cfg, nB, T)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def call():
        hb.hb_prefill_state(cfg, sl, t["k"], t["v"], t["cu_seqlens"], T, t["W"], S, Z,
                            workspace=ws)

    with ClockSampler(0) as clocks:
        ms = _timed(call, args.steps, args.warmup, stream)
    assert hb.hb_get_device_status() == 0
    med = _median(ms)
    tokens = nB * T
    nbytes = 2 * tokens * H * D * 2 + nB * H * (F * D + F) * 4 + H * D * FH * 2
    # tensor work as issued: U = K W (2 d f) and phi^T V with phi split hi + lo
    # (Z = sum of phi is summed on the CUDA cores)
    flops = tokens * H * (2 * D * FH + 2 * 2 * F * D)
    peak, kind = _peaks()
    tpeak, tkind = _tensor_peak()
    achieved = nbytes / (med / 1e3) / 1e9
    line = {
        "metric": "prompt-ingestion tokens/s and HBM GB/s", "value": tokens / (med / 1e3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": med, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prompt ingestion: hb_prefill_state, 8 prompts x 8,192 tokens, "
                               "16 heads, d=128, f=64, overwrite", "l2": "inputs 537 MB > L2"},
        "roofline": {"kernel": "hb_prefill_state", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_kind": kind,
                     "algorithmic_bytes_per_launch": nbytes, "launch_ms": med,
                     "traffic": _traffic("hb_prefill_state"),
                     "tensor": {"flops_per_launch": flops,
                                "achieved_tflops": flops / (med / 1e3) / 1e12,
                                "peak_tflops": tpeak, "peak_kind": tkind,
                                "frac": flops / (med / 1e3) / 1e12 / tpeak}},
        "gpu_launches": args.steps * (2 if need else 1),
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(max_seconds=args.cpu_seconds)
    return line


def run_decode(args):
    """Single-layer decode, 1 request, 16 heads, 2,048-token state. The step
    timed is the block's last denoising step: hb_block_attend_commit (attend
    and commit of the finished block in one launch). Also reported: the
    attend alone (every other denoising step of a block) and the same commit
    as two launches (hb_block_attend, then hb_commit_block)."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = inputs.single_layer(device=device)
    t = w.tensors
    cfg = hb.Config(H, D, FH, L)
    S = torch.zeros((1, H, F, D), dtype=torch.float32, device=device)
    Z = torch.zeros((1, H, F), dtype=torch.float32, device=device)
    sl = torch.zeros(1, dtype=torch.int32, device=device)
    for blk in range(t["commit_k"].shape[0]):
        hb.hb_commit_block(cfg, sl, t["commit_k"][blk], t["commit_v"][blk], t["W"], S, Z)
    o = torch.empty_like(t["q"])
    stream = torch.cuda.current_stream()
    one = torch.ones(1, dtype=torch.int32, device=device)
    S1, Z1 = S.clone(), Z.clone()
    S2, Z2 = S.clone(), Z.clone()

    def fused():
        hb.hb_block_attend_commit(cfg, sl, t["q"], t["k"], t["v"], S1, Z1, t["W"], t["gate"], one,
                                  o=o)

    def attend():
        hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"], o=o)

    def two_launches():
        hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S2, Z2, t["W"], t["gate"], o=o)
        hb.hb_commit_block(cfg, sl, t["k"], t["v"], t["W"], S2, Z2)

    # launch-to-launch device time: 50 calls per CUDA graph, host out of the loop
    reps = max(1, args.steps // 50)
    f_ms = _graph_ms(fused, 50, reps, args.warmup, stream)
    a_ms = _graph_ms(attend, 50, reps, args.warmup, stream)
    t_ms = _graph_ms(two_launches, 50, reps, args.warmup, stream)
    # the same call issued one by one from Python, for context
    f_host = _median(_timed(fused, min(args.steps, 200), args.warmup, stream))
    assert hb.hb_get_device_status() == 0
    nbytes = ATTEND_BYTES_PER_REQUEST + ATTEND_BYTES_W + H * (F * D + F) * 4
    peak, kind = _peaks()
    return {
        "metric": "single-layer decode: active-block tokens/s (committing step latency)",
        "value": L / (f_ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": f_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "single-layer decode: 1 request, 16 heads, d=128, f=64, L=32, "
                               "2,048-token state from 64 commits; step = attend + commit of "
                               "the finished block (hb_block_attend_commit)",
                   "l2": "state 1 MB stays L2-resident between calls (latency measurement)"},
        "roofline": {"kernel": "hb_block_attend_commit", "bound": "hbm",
                     "achieved": nbytes / (f_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": nbytes / (f_ms / 1e3) / 1e9 / peak, "peak_kind": kind,
                     "algorithmic_bytes_per_launch": nbytes, "launch_ms": f_ms,
                     "traffic": None},
        "components": {"attend_commit_fused_us": f_ms * 1e3, "attend_only_us": a_ms * 1e3,
                       "attend_then_commit_two_launches_us": t_ms * 1e3,
                       "fused_us_eager_python": f_host * 1e3,
                       "timing": "CUDA graph of 50 back-to-back calls, replayed"},
        "gpu_launches": 4 * 50 * reps,
    }


def run_feature_map(args):
    """Standalone feature map of one prompt-sized batch of keys: 65,536 tokens
    x 16 heads, d=128, f=64 -> phi fp32 (x 268 MB in, phi 537 MB out)."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    n = 65536
    cfg = hb.Config(H, D, FH, L)
    x = inputs.draw(11, (n, H, D), torch.bfloat16, device="cuda")
    W = inputs.draw(12, (H, D, FH), torch.bfloat16, device="cuda", std=D ** -0.5)
    phi = torch.empty((n, H, F), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    with ClockSampler(0) as clocks:
        ms = _timed(lambda: hb.hb_feature_map(cfg, x, W, phi), args.steps, args.warmup, stream)
    assert hb.hb_get_device_status() == 0
    med = _median(ms)
    nbytes = n * H * D * 2 + n * H * F * 4 + H * D * FH * 2
    peak, kind = _peaks()
    achieved = nbytes / (med / 1e3) / 1e9
    return {
        "metric": "feature-map tokens/s and HBM GB/s", "value": n / (med / 1e3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": med, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "hb_feature_map: 65,536 tokens x 16 heads, d=128, f=64, "
                               "bf16 in, fp32 phi out", "l2": "805 MB per call > L2"},
        "roofline": {"kernel": "hb_feature_map", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_kind": kind,
                     "algorithmic_bytes_per_launch": nbytes, "launch_ms": med,
                     "traffic": _traffic("hb_feature_map")},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }


def run_stack(args):
    """6 linearized layers, P=2,048-token prefixes, B in {1, 16, 64, 256}:
    one stack step = hb_block_attend of all 6 layers, timed against
    hb_softmax_kv_attend of the same 6 layers over the same prefixes kept as
    a KV cache, against hb_block_attend_s16 on bf16 copies of the same
    states (bit-identical output, half the state bytes), and against
    hb_block_attend_s8 on fp8 copies (a quarter of the state bytes; lossy)."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    cfg = hb.Config(H, D, FH, L)
    stream = torch.cuda.current_stream()
    peak, kind = _peaks()
    sweep = []
    P = 2048
    for nB in args.stack_batches:
        layers = []
        for layer in range(N_LAYERS):
            w = inputs.stack_layer(layer, nB, device=device, P=P)
            t = w.tensors
            S = torch.empty((nB, H, F, D), dtype=torch.float32, device=device)
            Z = torch.empty((nB, H, F), dtype=torch.float32, device=device)
            sl = torch.arange(nB, dtype=torch.int32, device=device)
            hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"], P,
                                t["W"], S, Z)
            S16 = torch.empty((nB, H, F, D), dtype=torch.bfloat16, device=device)
            hb.hb_state_to_bf16(cfg, sl, S, S16)
            S8 = torch.empty((nB, H, F, D), dtype=torch.uint8, device=device)
            sc8 = torch.empty((nB, H), dtype=torch.float32, device=device)
            hb.hb_state_to_fp8(cfg, sl, S, S8, sc8)
            need = hb.hb_softmax_kv_workspace_size(cfg, nB, P)
            layers.append(dict(t=t, S=S, S16=S16, S8=S8, sc8=sc8, Z=Z, sl=sl,
                               o=torch.empty_like(t["q"]),
                               ws=torch.empty(max(need, 16), dtype=torch.uint8, device=device)))
        torch.cuda.synchronize()

        def hybrid():
            for ly in layers:
                t = ly["t"]
                hb.hb_block_attend(cfg, ly["sl"], t["q"], t["k"], t["v"], ly["S"], ly["Z"],
                                   t["W"], t["gate"], o=ly["o"])

        def hybrid_s16():
            for ly in layers:
                t = ly["t"]
                hb.hb_block_attend_s16(cfg, ly["sl"], t["q"], t["k"], t["v"], ly["S16"], ly["Z"],
                                       t["W"], t["gate"], o=ly["o"])

        def hybrid_s8():
            for ly in layers:
                t = ly["t"]
                hb.hb_block_attend_s8(cfg, ly["sl"], t["q"], t["k"], t["v"], ly["S8"], ly["sc8"],
                                      ly["Z"], t["W"], t["gate"], o=ly["o"])

        def softmax():
            for ly in layers:
                t = ly["t"]
                hb.hb_softmax_kv_attend(cfg, t["prefix_k"], t["prefix_v"], t["cu_prefix"], P,
                                        t["q"], t["k"], t["v"], o=ly["o"], workspace=ly["ws"])

        # the same 6 layers as one launch (hb_block_attend_commit_layers,
        # attend only): the layers' requests, states, maps and gates side by side
        qa, ka, va = (torch.cat([ly["t"][n] for ly in layers]) for n in ("q", "k", "v"))
        Wa = torch.stack([ly["t"]["W"] for ly in layers])
        ga = torch.stack([ly["t"]["gate"] for ly in layers])
        Sa = torch.cat([ly["S"] for ly in layers])
        Za = torch.cat([ly["Z"] for ly in layers])
        sla = torch.arange(N_LAYERS * nB, dtype=torch.int32, device=device)
        oa = torch.empty_like(qa)

        def hybrid_layers():
            hb.hb_block_attend_commit_layers(cfg, sla, qa, ka, va, Sa, Za, Wa, ga, None, o=oa)

        hybrid()
        hybrid_layers()
        torch.cuda.synchronize()
        assert torch.equal(oa, torch.cat([ly["o"] for ly in layers]))

        reps = max(3, min(args.steps, 200))
        h_ms = _graph_ms(hybrid, 1, reps, args.warmup, stream)
        hl_ms = _graph_ms(hybrid_layers, 1, reps, args.warmup, stream)
        h16_ms = _graph_ms(hybrid_s16, 1, reps, args.warmup, stream)
        h8_ms = _graph_ms(hybrid_s8, 1, reps, args.warmup, stream)
        s_ms = _graph_ms(softmax, 1, max(3, reps // 4), args.warmup, stream)
        assert hb.hb_get_device_status() == 0
        hb_bytes = N_LAYERS * (nB * ATTEND_BYTES_PER_REQUEST + ATTEND_BYTES_W)
        # the bf16 copy halves the state read: S is H * F * d * 2 bytes per request
        hb16_bytes = hb_bytes - N_LAYERS * nB * H * F * D * 2
        # the fp8 copy: S is H * F * d bytes per request, plus a 4-byte scale per head
        hb8_bytes = hb_bytes - N_LAYERS * nB * H * (F * D * 3 - 4)
        sm_bytes = N_LAYERS * nB * ((P + L) * H * D * 2 * 2 + 2 * L * H * D * 2)
        sweep.append({
            "batch": nB, "hybrid_ms": h_ms, "softmax_kv_ms": s_ms,
            "hybrid_tokens_per_s": nB * L / (h_ms / 1e3),
            "softmax_kv_tokens_per_s": nB * L / (s_ms / 1e3),
            "speedup": s_ms / h_ms,
            "hybrid_gbs": hb_bytes / (h_ms / 1e3) / 1e9,
            "softmax_kv_gbs": sm_bytes / (s_ms / 1e3) / 1e9,
            "hybrid_frac": hb_bytes / (h_ms / 1e3) / 1e9 / peak,
            "softmax_kv_frac": sm_bytes / (s_ms / 1e3) / 1e9 / peak,
            "hybrid_layers_ms": hl_ms, "hybrid_layers_tokens_per_s": nB * L / (hl_ms / 1e3),
            "hybrid_layers_frac": hb_bytes / (hl_ms / 1e3) / 1e9 / peak,
            "layers_speedup": h_ms / hl_ms,
            "layers_note": "the 6 layers' attends as one launch (hb_block_attend_commit_layers), "
                           "output bit-identical to the 6 launches",
            "hybrid_s16_ms": h16_ms, "hybrid_s16_tokens_per_s": nB * L / (h16_ms / 1e3),
            "hybrid_s16_frac": hb16_bytes / (h16_ms / 1e3) / 1e9 / peak,
            "s16_speedup": h_ms / h16_ms,
            "s16_note": "attend only, on copies written once before timing; the refresh a "
                        "commit makes necessary (hb_state_to_bf16) is not in this number",
            "hybrid_s8_ms": h8_ms, "hybrid_s8_tokens_per_s": nB * L / (h8_ms / 1e3),
            "hybrid_s8_frac": hb8_bytes / (h8_ms / 1e3) / 1e9 / peak,
            "s8_speedup": h_ms / h8_ms,
            "s8_note": "attend only, on fp8 copies written once before timing (lossy: the "
                       "output is the attend on the dequantised state)",
        })
        del layers, qa, ka, va, Wa, ga, Sa, Za, oa
        torch.cuda.empty_cache()
    top = sweep[-1]
    return {
        "metric": "6-layer hybrid stack: active-block tokens/s vs softmax over KV cache",
        "value": top["hybrid_tokens_per_s"], "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": top["hybrid_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "6 linearized layers x 16 heads, d=128, f=64, L=32, 2,048-token "
                               "prefixes; stack step = 6 attends", "batches": args.stack_batches,
                   "timing": "each stack step captured as one CUDA graph and replayed",
                   "l2": "6 layers' states and KV caches exceed L2 from B=16 on"},
        "roofline": {"kernel": "hb_block_attend", "bound": "hbm", "achieved": top["hybrid_gbs"],
                     "peak": peak, "unit": "GB/s", "frac": top["hybrid_frac"],
                     "peak_kind": kind, "traffic": None},
        "sweep": sweep,
        "memory_per_request": _stack_memory(),
        "gpu_launches": N_LAYERS * args.steps,
    }


def _stack_memory():
    """What one request of the stack holds in device memory: the 6 layers'
    states against the KV cache the same 6 layers would keep as softmax
    layers (2,048 cached tokens and the active block, 32-token pages)."""
    from linear_attention_diffusion_feature_b300 import capacity

    tokens = 2048 + L
    kv = capacity.kv_cache_bytes(tokens, N_LAYERS, H, D)
    st = capacity.state_bytes(N_LAYERS, H, FH, D)
    return {"tokens": tokens, "kv_cache_bytes": kv, "state_bytes": st, "ratio": kv / st,
            "break_even_tokens": capacity.break_even_tokens(H, D, FH)}


def run_psweep(args):
    """One linearized layer, B in {1, 64}, prefix P = 1,024 .. 32,768 tokens:
    hb_block_attend (reads the fixed-size state, whatever P) against
    hb_softmax_kv_attend over the same prefix kept as a KV cache (reads all
    of it), packed per request and, through hb_softmax_kv_attend_paged, in
    32-token pages scattered over a shared pool. This is the shape of the
    pages' comparison over generation lengths."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    cfg = hb.Config(H, D, FH, L)
    stream = torch.cuda.current_stream()
    peak, kind = _peaks()
    sweep = []
    reps = max(3, min(args.steps, 100))
    for nB in args.psweep_batches:
        for P in args.psweep_prefixes:
            w = inputs.stack_layer(0, nB, device=device, P=P)
            t = w.tensors
            S = torch.empty((nB, H, F, D), dtype=torch.float32, device=device)
            Z = torch.empty((nB, H, F), dtype=torch.float32, device=device)
            sl = torch.arange(nB, dtype=torch.int32, device=device)
            pws = torch.empty(max(hb.hb_prefill_workspace_size(cfg, nB, P), 16), dtype=torch.uint8,
                              device=device)
            hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"], P, t["W"],
                                S, Z, workspace=pws)
            ws = torch.empty(max(hb.hb_softmax_kv_workspace_size(cfg, nB, P), 16),
                             dtype=torch.uint8, device=device)
            o = torch.empty_like(t["q"])
            kp, vp, table, plen = inputs.paged_cache(P, t["prefix_k"], t["prefix_v"], [P] * nB,
                                                     32)

            def hybrid():
                hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"], o=o)

            def softmax():
                hb.hb_softmax_kv_attend(cfg, t["prefix_k"], t["prefix_v"], t["cu_prefix"], P,
                                        t["q"], t["k"], t["v"], o=o, workspace=ws)

            def softmax_paged():
                hb.hb_softmax_kv_attend_paged(cfg, kp, vp, table, plen, P, t["q"], t["k"],
                                              t["v"], o=o, workspace=ws)

            h_ms = _graph_ms(hybrid, 10, reps, args.warmup, stream)
            s_ms = _graph_ms(softmax, 2, max(3, reps // 4), args.warmup, stream)
            sp_ms = _graph_ms(softmax_paged, 2, max(3, reps // 4), args.warmup, stream)
            assert hb.hb_get_device_status() == 0
            hb_bytes = nB * ATTEND_BYTES_PER_REQUEST + ATTEND_BYTES_W
            sm_bytes = nB * ((P + L) * H * D * 2 * 2 + 2 * L * H * D * 2)
            sweep.append({
                "batch": nB, "prefix": P, "hybrid_ms": h_ms, "softmax_kv_ms": s_ms,
                "speedup": s_ms / h_ms, "softmax_kv_paged_ms": sp_ms,
                "paged_over_packed": sp_ms / s_ms,
                "hybrid_gbs": hb_bytes / (h_ms / 1e3) / 1e9,
                "softmax_kv_gbs": sm_bytes / (s_ms / 1e3) / 1e9,
                "hybrid_frac": hb_bytes / (h_ms / 1e3) / 1e9 / peak,
                "softmax_kv_frac": sm_bytes / (s_ms / 1e3) / 1e9 / peak,
            })
            del w, t, S, Z, ws, pws, o, kp, vp, table, plen
            torch.cuda.empty_cache()
    top = sweep[-1]
    return {
        "metric": "prefix-length sweep: active-block tokens/s, hybrid vs softmax over KV cache",
        "value": top["batch"] * L / (top["hybrid_ms"] / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": top["hybrid_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "one linearized layer x 16 heads, d=128, f=64, L=32; "
                               f"B in {args.psweep_batches}; prefix P in {args.psweep_prefixes}",
                   "timing": "10 (hybrid) or 2 (softmax) calls per CUDA graph, graph replayed",
                   "paged": "softmax over 32-token pages at seeded positions of one pool",
                   "l2": "back-to-back calls on one layer: the hybrid's bytes (1.8 MB at B=1, "
                         "101 MB at B=64) and the softmax caches below ~100 MB stay partly in "
                         "the 126 MB L2 between calls; the step and stack workloads rotate "
                         "layers to avoid that"},
        "roofline": {"kernel": "hb_block_attend", "bound": "hbm", "achieved": top["hybrid_gbs"],
                     "peak": peak, "unit": "GB/s", "frac": top["hybrid_frac"],
                     "peak_kind": kind, "traffic": None},
        "sweep": sweep,
        "gpu_launches": 10 * reps,
    }


def _prefill_attend(args, device, nB, T, reps):
    """Times hb_prefill_attend on nB prompts of T tokens (the prompt-ingestion
    shape, q drawn beside it), one call per CUDA graph."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    cfg = hb.Config(H, D, FH, L)
    g = inputs.prompt_ingestion(device=device, B=nB, T=T)
    k = g.tensors["k"].view(nB, T, H, D)
    v = g.tensors["v"].view(nB, T, H, D)
    q = inputs.draw(41, (nB, T, H, D), torch.bfloat16, device=device)
    W = g.tensors["W"]
    gate = g.tensors["gate"]
    S = torch.empty((nB, H, F, D), dtype=torch.float32, device=device)
    Z = torch.empty((nB, H, F), dtype=torch.float32, device=device)
    sl = torch.arange(nB, dtype=torch.int32, device=device)
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def call():
        hb.hb_prefill_attend(cfg, sl, q, k, v, S, Z, W, gate, o=o)

    with ClockSampler(0) as clocks:
        ms = _graph_ms(call, 1, reps, args.warmup, stream)
    assert hb.hb_get_device_status() == 0
    tokens = nB * T
    # the formulation's minimum: read q, k, v, write o and the final state
    nbytes = 4 * tokens * H * D * 2 + nB * H * (F * D + F) * 4 + H * D * FH * 2
    peak, kind = _peaks()
    del g, k, v, q, S, Z, o
    torch.cuda.empty_cache()
    return {"ms": ms, "tokens": tokens, "nbytes": nbytes, "achieved": nbytes / (ms / 1e3) / 1e9,
            "peak": peak, "kind": kind, "clocks": clocks.summary()}


def run_prefill_attend(args):
    """Prompt processing with outputs: 8 prompts x 8,192 tokens, 16 heads,
    d=128, f=64 (the prompt-ingestion shape), every 32-token block attending
    to the state of the blocks before it and then committed
    (hb_prefill_attend: one CTA per prompt and head walks the prompt in
    128-token segments with the state kept on chip)."""
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    nB, T = args.pa_batch, args.pa_len
    reps = max(3, min(args.steps, 20))
    r = _prefill_attend(args, device, nB, T, reps)
    ms, tokens, nbytes = r["ms"], r["tokens"], r["nbytes"]
    return {
        "metric": "prompt processing with outputs: prompt tokens/s", "value": tokens / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": 1, "steps": reps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"hb_prefill_attend: {nB} prompts x {T} tokens, 16 heads, "
                               "d=128, f=64, L=32, from empty states",
                   "timing": "one call (a state reset and one prompt kernel) per CUDA graph, "
                             "replayed",
                   "l2": f"q, k, v, o {4 * nB * T * H * D * 2 / 1e9:.2f} GB"},
        "roofline": {"kernel": "hb_prefill_attend (k_prompt_tc)",
                     "bound": "hbm", "achieved": r["achieved"], "peak": r["peak"], "unit": "GB/s",
                     "frac": r["achieved"] / r["peak"], "peak_kind": r["kind"],
                     "algorithmic_bytes_per_call": nbytes,
                     "traffic": _traffic("hb_prefill_attend") if (nB, T) == (8, 8192) else None},
        "gpu_launches": reps * 2,
        "clocks": r["clocks"],
    }


def run_blocklen(args):
    """The continuous-batching step (64 requests, 16 committing, hb_block_attend_commit)
    at block lengths L = 16, 32 and 64: L = 32 and 16 take the persistent
    attend kernel (16-token blocks in its 32-row tiles), 64 the segment
    kernel on a one-block prompt. Six layer instances in turn, graphs of 600
    steps replayed for >= 0.5 s."""
    import linear_attention_diffusion_feature_b300 as hb
    from linear_attention_diffusion_feature_b300 import inputs

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()
    peak, kind = _peaks()
    out = []
    for Lb in args.block_lens:
        cfg = hb.Config(H, D, FH, Lb)
        layers = []
        for layer in range(N_LAYERS):
            w = inputs.continuous_batching(seed=50 + layer, device=device, B=B, n_commit=N_COMMIT)
            t = w.tensors
            S = torch.empty((B, H, F, D), dtype=torch.float32, device=device)
            Z = torch.empty((B, H, F), dtype=torch.float32, device=device)
            sl = torch.arange(B, dtype=torch.int32, device=device)
            hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                                w.meta["max_prefix"], t["W"], S, Z)
            qkv = [inputs.draw(60 + 3 * layer + j, (B, Lb, H, D), torch.bfloat16, device)
                   for j in range(3)]
            mask = torch.zeros(B, dtype=torch.int32, device=device)
            mask[t["commit_idx"]] = 1
            layers.append(dict(S=S, Z=Z, sl=sl, W=t["W"], gate=t["gate"], q=qkv[0], k=qkv[1],
                               v=qkv[2], mask=mask, o=torch.empty_like(qkv[0])))
            del t, w
        torch.cuda.synchronize()

        def step(i):
            ly = layers[i % N_LAYERS]
            hb.hb_block_attend_commit(cfg, ly["sl"], ly["q"], ly["k"], ly["v"], ly["S"], ly["Z"],
                                      ly["W"], ly["gate"], ly["mask"], o=ly["o"])

        for i in range(args.warmup):
            step(i)
        g = StepGraphs(step, GRAPH_STEPS)
        g.replay()
        one = _timed_replays(g, 1, stream)
        n_rep = max(1, int(500.0 / one) + 1)
        ms = _timed_replays(g, n_rep, stream) / (n_rep * GRAPH_STEPS)
        assert hb.hb_get_device_status() == 0
        nbytes = (B * (H * (F * D * 4 + F * 4) + 4 * Lb * H * D * 2) + H * D * FH * 2
                  + N_COMMIT * H * (F * D * 4 + F * 4))
        out.append({"block_len": Lb, "ms": ms, "tokens_per_s": B * Lb / (ms / 1e3),
                    "algorithmic_bytes": nbytes, "hbm_frac": nbytes / (ms / 1e3) / 1e9 / peak,
                    "achieved_gbs": nbytes / (ms / 1e3) / 1e9,
                    "kernel": {32: "k_attend_fast (persistent)",
                               16: "k_attend_fast (persistent, 16-token blocks in 32-row tiles)"}
                    .get(Lb, "k_prompt_tc")})
        del layers, g
        torch.cuda.empty_cache()
    top = out[0]
    return {
        "metric": "continuous-batching step at several block lengths: active-block tokens/s",
        "value": top["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": top["ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "hb_block_attend_commit, 64 requests x 16 heads, d=128, f=64, "
                               "16 committing, prefixes 32*U{8..128}", "block_lens": args.block_lens,
                   "timing": "graphs of 600 steps over 6 layer instances, >= 0.5 s of replays"},
        "roofline": {"kernel": top["kernel"], "bound": "hbm", "achieved": top["achieved_gbs"],
                     "peak": peak, "unit": "GB/s", "frac": top["hbm_frac"], "peak_kind": kind,
                     "traffic": None},
        "sweep": out,
        "gpu_launches": None,
    }


def run_serve(args):
    """Continuous-batching simulation on the library's own calls (the pages'
    end-to-end protocol on synthetic layers): the same stream of requests
    (2,048 generated tokens each, prompts of 128-512 tokens, 8 denoising
    steps per block) served by the hybrid layers (fixed-size states) and by
    the same layers as softmax over a paged KV cache, at each concurrency cap
    of the sweep, under one attention-memory budget for the 20-layer model."""
    from linear_attention_diffusion_feature_b300 import serving

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    sweep = []
    for C in args.serve_concurrency:
        cfg = serving.ServeConfig(n_requests=max(2 * C, 4), max_concurrency=C,
                                  memory_budget=args.serve_budget_gib << 30)
        res = serving.compare(cfg, device)
        res["max_concurrency"] = C
        res["n_requests"] = cfg.n_requests
        sweep.append(res)
        torch.cuda.empty_cache()
    import linear_attention_diffusion_feature_b300 as hb

    assert hb.hb_get_device_status() == 0
    top = sweep[-1]
    return {
        "metric": "continuous-batching simulation: generated tokens/s, hybrid vs softmax "
                  "attention layers", "value": top["hybrid"]["tokens_per_s_wall"],
        "unit": "tokens/s", "n_gpus": 1, "steps": top["hybrid"]["steps"], "warmup": 0,
        "ms_per_step": top["hybrid"]["wall_s"] * 1e3 / max(top["hybrid"]["steps"], 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "6 attention layers (16 heads, d=128, f=64, L=32) served with "
                               "continuous batching; 2,048 generated tokens per request, prompts "
                               "32*U{4..16} tokens, 8 denoising steps per block; memory model: "
                               "20-layer model, 6 linearized",
                   "memory_budget_gib": args.serve_budget_gib,
                   "concurrency": args.serve_concurrency,
                   "timing": "wall clock around the whole stream (host scheduling included) "
                             "and the sum of per-step CUDA-event times"},
        "sweep": sweep,
        "gpu_launches": None,
    }


def cpu_baseline_prefill(max_seconds: float = 15.0, T: int = 256):
    """The oracle's prefill on one 256-token prompt of the same shape."""
    import numpy as np

    import oracle.block_hybrid as ob
    from linear_attention_diffusion_feature_b300 import inputs

    w = inputs.prompt_ingestion(device="cpu", B=1, T=T)
    k = w.tensors["k"].to(torch.float64).numpy()
    v = w.tensors["v"].to(torch.float64).numpy()
    W = w.tensors["W"].to(torch.float64).numpy()
    t0 = time.perf_counter()
    reps = 0
    while True:
        ob.prefill(k, v, W)
        reps += 1
        el = time.perf_counter() - t0
        if el >= max_seconds or reps >= 1000:
            break
    del np
    return {"value": reps * T / el, "unit": "tokens/s", "cores": _blas_threads(),
            "kind": "oracle",
            "sample": f"{reps} x one {T}-token prompt, 16 heads, fp64 numpy oracle, {el:.1f} s"}


# ----------------------------------------------------------- CPU oracle arm

def _oracle_sample(n_req: int, seed: int = 2):
    """A bounded sample of the step for the oracle: ``n_req`` requests of the
    same workload recipe, their states from the oracle's own prefill (outside
    the timed region), and a quarter of them committing."""
    import numpy as np

    import oracle.block_hybrid as ob
    from linear_attention_diffusion_feature_b300 import inputs

    w = inputs.continuous_batching(seed=seed, device="cpu", B=n_req,
                                   n_commit=max(1, n_req // 4))
    t = {k: (v.to(torch.float64).numpy() if v.is_floating_point() else v.numpy())
         for k, v in w.tensors.items()}
    cu = t["cu_prefix"]
    states = [ob.prefill(t["prefix_k"][cu[b]:cu[b + 1]], t["prefix_v"][cu[b]:cu[b + 1]], t["W"])
              for b in range(n_req)]
    commit = set(np.asarray(t["commit_idx"]).tolist())
    return ob, t, states, commit


def _oracle_step(ob, t, states, commit):
    from oracle import host_baseline

    host_baseline.one_step(t, states, commit)


def _oracle_all_cores(t, states, commit, seconds: float):
    """The same sample on one process per host core (started by spawn, each
    with a single BLAS thread); returns (steps per second summed over the
    processes, processes)."""
    import concurrent.futures
    import multiprocessing

    from oracle import host_baseline

    n = os.cpu_count() or 1
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                             "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        ctx = multiprocessing.get_context("spawn")
        with concurrent.futures.ProcessPoolExecutor(max_workers=n, mp_context=ctx) as ex:
            res = list(ex.map(host_baseline.timed_steps, [(t, states, commit, seconds)] * n))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return sum(reps / el for reps, el in res), n


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:  # noqa: BLE001
        return 1


def cpu_baseline(max_seconds: float = 15.0, n_req: int = 8):
    ob, t, states, commit = _oracle_sample(n_req)
    t0 = time.perf_counter()
    reps = 0
    while True:
        _oracle_step(ob, t, states, commit)
        reps += 1
        el = time.perf_counter() - t0
        if el >= max_seconds or reps >= 1000:
            break
    tokens = reps * n_req * L
    one_proc = tokens / el
    rate, n = _oracle_all_cores(t, states, commit, max_seconds)
    return {"value": rate * n_req * L, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"the step restricted to {n_req} requests ({len(commit)} committing), "
                      f"fp64 numpy oracle, one process per core for {max_seconds:.0f} s",
            "one_process": {"value": one_proc, "cores": _blas_threads(),
                            "sample": f"{reps} repetitions in {el:.1f} s"}}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    n_req = 8
    ob, t, states, commit = _oracle_sample(n_req)
    for _ in range(args.warmup):
        _oracle_step(ob, t, states, commit)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(ob, t, states, commit)
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    value = n_req * L / (ms / 1e3)
    cores = _blas_threads()
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "continuous-batching step (oracle sample)", "batch": n_req,
                   "block_len": L, "heads": H, "head_dim": D, "feat_half": FH},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: {n_req} requests' attend + {len(commit)} commits"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-components", action="store_true",
                    help="skip the stack (B=256) and prompt-ingestion components of the "
                         "default line")
    ap.add_argument("--workload", choices=["step", "decode", "prefill", "stack", "feature_map", "psweep",
                             "prefill_attend", "serve", "blocklen"],
                    default="step",
                    help="step: continuous-batching step (default); decode: single-layer "
                         "latency; prefill: prompt ingestion; stack: 6-layer sweep vs "
                         "softmax over a KV cache; feature_map: standalone phi")
    ap.add_argument("--stack-batches", type=int, nargs="+", default=[1, 16, 64, 256])
    ap.add_argument("--block-lens", type=int, nargs="+", default=[16, 32, 64])
    ap.add_argument("--pa-batch", type=int, default=8, help="prefill_attend: prompts")
    ap.add_argument("--pa-len", type=int, default=8192, help="prefill_attend: tokens each")
    ap.add_argument("--serve-concurrency", type=int, nargs="+", default=[1, 16, 64, 128])
    ap.add_argument("--serve-budget-gib", type=int, default=40)
    ap.add_argument("--psweep-batches", type=int, nargs="+", default=[1, 64])
    ap.add_argument("--psweep-prefixes", type=int, nargs="+",
                    default=[1024, 2048, 4096, 8192, 16384, 32768])
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = _dist()
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: for N > 1 GPUs launch one "
                 f"process per GPU with torchrun (python -m torch.distributed.run "
                 f"--nproc-per-node N ... bench.py --gpus N)")
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if args.workload != "step":
        if world > 1:
            ap.error("--workload other than step runs on one GPU")
        runner = {"decode": run_decode, "prefill": run_prefill, "stack": run_stack,
                  "feature_map": run_feature_map, "psweep": run_psweep,
                  "prefill_attend": run_prefill_attend, "serve": run_serve,
                  "blocklen": run_blocklen}
        print(json.dumps(runner[args.workload](args)), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    line = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Continuous-batching simulator of blockwise diffusion decoding, run on this
library's own calls.

It reproduces the shape of the pages' two end-to-end claims on synthetic
layers (gist.science technical summary, "Experimental Results / Throughput
and Concurrency": higher decoding throughput under continuous batching, and
more concurrent requests before memory runs out; pith.science, "Editorial
extensions / If this is right": 1.50-1.73x throughput, about 1.3x more
concurrent requests). Two servers run the same request stream:

* ``HybridBackend`` — the linearized layers: a prompt is ingested into a
  state slot (``hb_prefill_state``); every denoising step runs one
  ``hb_block_attend_commit`` per layer for all active requests, with the
  commit mask set for the requests whose block is finished.
* ``SoftmaxBackend`` — the same layers kept as softmax attention: a prompt
  is written into 32-token pages of a shared KV pool; every step runs one
  ``hb_softmax_kv_attend_paged`` per layer; a finished block is appended to
  its request's pages.

Only the attention of the ``layers`` simulated layers runs; the rest of the
model (projections, MLPs, the other softmax layers) has no weights here.
Memory, however, is accounted for the whole attention stack of the pages'
model (20 layers, 6 of them linearized) with ``capacity``: a request is
admitted only if its attention memory at its final length fits the budget
(reserved at admission), so the budget caps each server's concurrency.

Values the pages do not fix and this module chooses (each is a field of
``ServeConfig``): prompt lengths uniform over multiples of 32 in [128, 512],
8 denoising steps per 32-token block, the attention-memory budget, and that
prompts are ingested as context only (no prompt outputs on either side).

The scheduler (``Scheduler``) is plain host logic with no device access, so
that its bookkeeping can be tested on its own.
"""

from __future__ import annotations

import collections
import time
from dataclasses import dataclass, field

import torch

from . import capacity


@dataclass
class ServeConfig:
    n_requests: int = 256          # prompts in the stream
    max_concurrency: int = 128     # the serving engine's cap on active requests
    gen_tokens: int = 2048         # tokens generated per request (the pages' protocol)
    block_len: int = 32            # L
    steps_per_block: int = 8       # denoising steps per block (not fixed by the pages)
    prompt_min: int = 128          # prompt lengths: multiples of 32 in [min, max]
    prompt_max: int = 512
    memory_budget: int = 40 << 30  # attention memory of all layers, bytes
    model_layers: int = 20         # attention layers of the model (memory model)
    linear_layers: int = 6         # linearized layers of the hybrid model
    layers: int = 6                # layers whose attention is actually run
    H: int = 16
    d: int = 128
    f: int = 64
    seed: int = 0

    @property
    def gen_blocks(self) -> int:
        return self.gen_tokens // self.block_len


@dataclass
class Request:
    rid: int
    prompt_len: int
    slot: int = -1
    blocks_done: int = 0
    step_in_block: int = 0
    reserved: int = 0  # bytes of the memory budget held


@dataclass
class StepPlan:
    admitted: list            # requests admitted before this step (ingest first)
    active: list              # requests in batch order
    commit: list              # per active request: its block is finished this step


class Scheduler:
    """Admission, slot recycling and block bookkeeping of a continuous
    batch. ``hybrid`` selects the memory model: 14 softmax layers + 6
    linearized ones, or all 20 layers softmax."""

    def __init__(self, cfg: ServeConfig, hybrid: bool):
        self.cfg = cfg
        self.hybrid = hybrid
        g = torch.Generator().manual_seed(cfg.seed)
        lo, hi = cfg.prompt_min // cfg.block_len, cfg.prompt_max // cfg.block_len
        lens = (torch.randint(lo, hi + 1, (cfg.n_requests,), generator=g) * cfg.block_len)
        self.waiting = collections.deque(Request(i, int(n)) for i, n in enumerate(lens.tolist()))
        self.active: list = []
        self.free_slots = list(range(cfg.max_concurrency))[::-1]
        self.used = 0
        self.finished: list = []
        self.peak_active = 0
        self.tokens_done = 0

    def request_bytes(self, r: Request) -> int:
        c = self.cfg
        tokens = r.prompt_len + c.gen_tokens
        if self.hybrid:
            return capacity.request_bytes(tokens, c.model_layers - c.linear_layers,
                                          c.linear_layers, c.H, c.d, c.f, c.block_len)
        return capacity.request_bytes(tokens, c.model_layers, 0, c.H, c.d, c.f, c.block_len)

    def capacity_limit(self) -> int:
        """Requests of the longest prompt that fit in the budget."""
        r = Request(-1, self.cfg.prompt_max)
        return self.cfg.memory_budget // self.request_bytes(r)

    def plan(self) -> StepPlan:
        admitted = []
        while self.waiting and self.free_slots:
            r = self.waiting[0]
            need = self.request_bytes(r)
            if self.used + need > self.cfg.memory_budget:
                break
            self.waiting.popleft()
            r.slot = self.free_slots.pop()
            r.reserved = need
            self.used += need
            self.active.append(r)
            admitted.append(r)
        self.peak_active = max(self.peak_active, len(self.active))
        commit = [r.step_in_block == self.cfg.steps_per_block - 1 for r in self.active]
        return StepPlan(admitted, list(self.active), commit)

    def finish(self, plan: StepPlan) -> None:
        keep = []
        for r, c in zip(plan.active, plan.commit):
            if c:
                r.blocks_done += 1
                r.step_in_block = 0
                self.tokens_done += self.cfg.block_len
            else:
                r.step_in_block += 1
            if r.blocks_done == self.cfg.gen_blocks:
                self.free_slots.append(r.slot)
                self.used -= r.reserved
                self.finished.append(r)
            else:
                keep.append(r)
        self.active = keep

    def done(self) -> bool:
        return not self.waiting and not self.active


class _Synthetic:
    """Seeded activations shared by both backends: per layer, W and gate, an
    active-block pool q, k, v [max_concurrency, L, H, d] (request b of a
    step's batch uses row b) and a prompt pool [max prompt tokens, H, d]."""

    def __init__(self, cfg: ServeConfig, device):
        from . import inputs

        self.layers = []
        C, L, H, d, f = cfg.max_concurrency, cfg.block_len, cfg.H, cfg.d, cfg.f
        for layer in range(cfg.layers):
            s = 7000 + 10 * layer + cfg.seed
            self.layers.append(dict(
                W=inputs.draw(s, (H, d, f), torch.bfloat16, device, std=d ** -0.5),
                gate=inputs.draw(s + 1, (H,), torch.float32, device),
                q=inputs.draw(s + 2, (C, L, H, d), torch.bfloat16, device),
                k=inputs.draw(s + 3, (C, L, H, d), torch.bfloat16, device),
                v=inputs.draw(s + 4, (C, L, H, d), torch.bfloat16, device),
                pk=inputs.draw(s + 5, (C * cfg.prompt_max, H, d), torch.bfloat16, device),
                pv=inputs.draw(s + 6, (C * cfg.prompt_max, H, d), torch.bfloat16, device),
                o=torch.empty((C, L, H, d), dtype=torch.bfloat16, device=device)))


class HybridBackend:
    """Linearized layers: a state slot per request and layer."""

    name = "hybrid"

    def __init__(self, cfg: ServeConfig, device, syn: _Synthetic):
        from . import hb

        self.hb = hb
        self.cfg = cfg
        self.syn = syn
        self.device = device
        self.hcfg = hb.Config(cfg.H, cfg.d, cfg.f, cfg.block_len)
        F = 2 * cfg.f
        C = cfg.max_concurrency
        self.S = [torch.zeros((C, cfg.H, F, cfg.d), dtype=torch.float32, device=device)
                  for _ in range(cfg.layers)]
        self.Z = [torch.zeros((C, cfg.H, F), dtype=torch.float32, device=device)
                  for _ in range(cfg.layers)]
        need = hb.hb_prefill_workspace_size(self.hcfg, C, cfg.prompt_max)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)

    def ingest(self, reqs) -> None:
        """Prompts as committed context: overwrite the new requests' slots."""
        lens = [r.prompt_len for r in reqs]
        cu = torch.tensor([0] + list(_cumsum(lens)), dtype=torch.int64).to(self.device)
        sl = torch.tensor([r.slot for r in reqs], dtype=torch.int32).to(self.device)
        total = sum(lens)
        for layer, ly in enumerate(self.syn.layers):
            self.hb.hb_prefill_state(self.hcfg, sl, ly["pk"][:total], ly["pv"][:total], cu,
                                     max(lens), ly["W"], self.S[layer], self.Z[layer],
                                     workspace=self.ws)

    def step(self, slots, commit) -> None:
        B = slots.shape[0]
        for layer, ly in enumerate(self.syn.layers):
            self.hb.hb_block_attend_commit(self.hcfg, slots, ly["q"][:B], ly["k"][:B],
                                           ly["v"][:B], self.S[layer], self.Z[layer], ly["W"],
                                           ly["gate"], commit, o=ly["o"][:B])


class SoftmaxBackend:
    """The same layers as softmax attention over a paged KV cache (32-token
    pages; a finished 32-token block is exactly one page)."""

    name = "softmax"

    def __init__(self, cfg: ServeConfig, device, syn: _Synthetic):
        from . import hb

        self.hb = hb
        self.cfg = cfg
        self.syn = syn
        self.device = device
        self.hcfg = hb.Config(cfg.H, cfg.d, cfg.f, cfg.block_len)
        C, pt = cfg.max_concurrency, cfg.block_len
        self.max_pages = (cfg.prompt_max + cfg.gen_tokens) // pt
        n_pages = C * self.max_pages
        self.kp = [torch.empty((n_pages, pt, cfg.H, cfg.d), dtype=torch.bfloat16, device=device)
                   for _ in range(cfg.layers)]
        self.vp = [torch.empty_like(self.kp[0]) for _ in range(cfg.layers)]
        # one page table for all layers: a request's pages have the same ids in
        # every layer's pool
        self.table = torch.zeros((C, self.max_pages), dtype=torch.int32, device=device)
        self.plen = torch.zeros(C, dtype=torch.int32, device=device)
        self.pages_of = {}  # slot -> list of page ids (host)
        self.free_pages = list(range(n_pages))[::-1]
        need = hb.hb_softmax_kv_workspace_size(self.hcfg, C, cfg.prompt_max + cfg.gen_tokens)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        self.max_prefix = cfg.prompt_max + cfg.gen_tokens

    def ingest(self, reqs) -> None:
        """Write each new request's prompt into fresh pages of every layer."""
        pt = self.cfg.block_len
        pages, rows, slots_rows = [], [], []
        off = 0
        for r in reqs:
            old = self.pages_of.pop(r.slot, [])
            self.free_pages.extend(old)
            n = r.prompt_len // pt
            ids = [self.free_pages.pop() for _ in range(n)]
            self.pages_of[r.slot] = ids
            pages += ids
            rows += list(range(off, off + r.prompt_len))
            off += r.prompt_len
            slots_rows.append((r.slot, ids, r.prompt_len))
        page_idx = torch.tensor(pages, dtype=torch.int64).to(self.device)
        for layer, ly in enumerate(self.syn.layers):
            src_k = ly["pk"][:off].view(-1, pt, self.cfg.H, self.cfg.d)
            src_v = ly["pv"][:off].view(-1, pt, self.cfg.H, self.cfg.d)
            self.kp[layer].index_copy_(0, page_idx, src_k)
            self.vp[layer].index_copy_(0, page_idx, src_v)
        for slot, ids, n in slots_rows:
            row = torch.zeros(self.max_pages, dtype=torch.int32)
            row[:len(ids)] = torch.tensor(ids, dtype=torch.int32)
            self.table[slot].copy_(row.to(self.device))
            self.plen[slot] = n

    def step(self, slots, commit) -> None:
        B = slots.shape[0]
        idx = slots.long()
        table = self.table.index_select(0, idx)
        plen = self.plen.index_select(0, idx)
        for ly, kp, vp in zip(self.syn.layers, self.kp, self.vp):
            self.hb.hb_softmax_kv_attend_paged(self.hcfg, kp, vp, table, plen, self.max_prefix,
                                               ly["q"][:B], ly["k"][:B], ly["v"][:B],
                                               o=ly["o"][:B], workspace=self.ws)

    def append(self, plan, slots_host) -> None:
        """A finished block becomes the next page of its request."""
        who = [b for b, c in enumerate(plan.commit) if c]
        if not who:
            return
        new_pages, rows, cols = [], [], []
        for b in who:
            slot = slots_host[b]
            pid = self.free_pages.pop()
            cols.append(len(self.pages_of[slot]))
            self.pages_of[slot].append(pid)
            new_pages.append(pid)
            rows.append(slot)
        pidx = torch.tensor(new_pages, dtype=torch.int64).to(self.device)
        bidx = torch.tensor(who, dtype=torch.int64).to(self.device)
        for ly, kp, vp in zip(self.syn.layers, self.kp, self.vp):
            kp.index_copy_(0, pidx, ly["k"].index_select(0, bidx))
            vp.index_copy_(0, pidx, ly["v"].index_select(0, bidx))
        r = torch.tensor(rows, dtype=torch.int64).to(self.device)
        c = torch.tensor(cols, dtype=torch.int64).to(self.device)
        self.table.index_put_((r, c), pidx.to(torch.int32))
        self.plen.index_add_(0, r, torch.full((len(who),), self.cfg.block_len,
                                              dtype=torch.int32, device=self.device))

    def release(self, reqs) -> None:
        for r in reqs:
            self.free_pages.extend(self.pages_of.pop(r.slot, []))


def _cumsum(xs):
    t = 0
    for x in xs:
        t += x
        yield t


@dataclass
class ServeResult:
    backend: str
    steps: int
    tokens: int
    wall_s: float
    device_s: float
    peak_active: int
    mean_active: float
    capacity_limit: int
    finished: int
    step_ms: list = field(default_factory=list)

    def as_dict(self) -> dict:
        return {
            "backend": self.backend, "steps": self.steps, "tokens": self.tokens,
            "wall_s": self.wall_s, "device_s": self.device_s,
            "tokens_per_s_wall": self.tokens / self.wall_s if self.wall_s else 0.0,
            "tokens_per_s_device": self.tokens / self.device_s if self.device_s else 0.0,
            "peak_active": self.peak_active, "mean_active": self.mean_active,
            "capacity_limit": self.capacity_limit, "finished": self.finished,
            "device_phases": getattr(self, "phases", None),
        }


def simulate(backend, cfg: ServeConfig, max_steps: int = None, trace: list = None) -> ServeResult:
    """Runs the request stream to completion (or ``max_steps`` steps) on
    ``backend`` and times it: wall clock around the whole loop, and the
    device time of each step's attention (CUDA events). With ``trace``, it
    appends ("ingest", rid, slot, first prompt row, prompt length) for every
    admission and ("commit", rid, slot, batch row) for every committed block,
    which is what a request's state is made of."""
    sched = Scheduler(cfg, hybrid=backend.name == "hybrid")
    dev = backend.device
    stream = torch.cuda.current_stream(dev)
    events = []
    steps = 0
    active_sum = 0
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    while not sched.done() and (max_steps is None or steps < max_steps):
        plan = sched.plan()
        if not plan.active:
            raise RuntimeError("no request fits the memory budget")
        a = torch.cuda.Event(enable_timing=True)
        m1 = torch.cuda.Event(enable_timing=True)
        m2 = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if plan.admitted:
            backend.ingest(plan.admitted)
            if trace is not None:
                row = 0
                for r in plan.admitted:
                    trace.append(("ingest", r.rid, r.slot, row, r.prompt_len))
                    row += r.prompt_len
        slots_host = [r.slot for r in plan.active]
        slots = torch.tensor(slots_host, dtype=torch.int32).to(dev, non_blocking=True)
        commit = torch.tensor(plan.commit, dtype=torch.int32).to(dev, non_blocking=True)
        m1.record(stream)
        backend.step(slots, commit)
        m2.record(stream)
        if isinstance(backend, SoftmaxBackend):
            backend.append(plan, slots_host)
        b.record(stream)
        events.append((a, m1, m2, b))
        if trace is not None:
            for b, (r, c) in enumerate(zip(plan.active, plan.commit)):
                if c:
                    trace.append(("commit", r.rid, r.slot, b))
        sched.finish(plan)
        if isinstance(backend, SoftmaxBackend):
            backend.release([r for r in plan.active if r.blocks_done == cfg.gen_blocks])
        active_sum += len(plan.active)
        steps += 1
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    step_ms = [a.elapsed_time(b) for a, m1, m2, b in events]
    phases = {"before_attend_s": sum(a.elapsed_time(m1) for a, m1, m2, b in events) / 1e3,
              "attend_s": sum(m1.elapsed_time(m2) for a, m1, m2, b in events) / 1e3,
              "after_attend_s": sum(m2.elapsed_time(b) for a, m1, m2, b in events) / 1e3}
    res = ServeResult(backend.name, steps, sched.tokens_done, wall, sum(step_ms) / 1e3,
                      sched.peak_active, active_sum / max(steps, 1), sched.capacity_limit(),
                      len(sched.finished), step_ms)
    res.phases = phases
    return res


def compare(cfg: ServeConfig, device, max_steps: int = None, warmup: bool = True) -> dict:
    """The same request stream on both servers.

    With ``warmup``, each server first runs the stream's first block
    (admission, ``steps_per_block`` steps and the commit) on a throwaway
    backend of the same shapes, untimed: the first use of a device function
    in a process (module loading, and a just-in-time compile where the
    binary holds no code for the device) can stall the host for seconds,
    and without the warm-up that stall lands in the first timed step."""
    syn = _Synthetic(cfg, device)
    out = {}
    for cls in (HybridBackend, SoftmaxBackend):
        if warmup:
            be = cls(cfg, device, syn)
            simulate(be, cfg, cfg.steps_per_block + 1)
            del be
            torch.cuda.empty_cache()
        be = cls(cfg, device, syn)
        out[be.name] = simulate(be, cfg, max_steps).as_dict()
        del be
        torch.cuda.empty_cache()
    h, s = out["hybrid"], out["softmax"]
    out["throughput_ratio_wall"] = (h["tokens_per_s_wall"] / s["tokens_per_s_wall"]
                                    if s["tokens_per_s_wall"] else None)
    out["throughput_ratio_device"] = (h["tokens_per_s_device"] / s["tokens_per_s_device"]
                                      if s["tokens_per_s_device"] else None)
    out["concurrency_ratio"] = (h["capacity_limit"] / s["capacity_limit"]
                                if s["capacity_limit"] else None)
    return out

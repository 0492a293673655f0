"""Seeded synthetic inputs shaped like the workloads on the pages.

The setting follows the pages about arXiv 2608.06628: LLaDA 2.1-mini-like
layers (16 heads of dimension 128), 6 of 20 attention layers linearized,
blocks of 32 tokens, 2,048-token prefixes, continuous batching. This module
only draws random numbers and lays them out; it holds none of the method's
arithmetic, so the fp64 oracle and the CUDA library can both be fed from it.

Recipe: every tensor is drawn in float32 from a ``torch.Generator`` seeded
with the workload's seed (on the device the caller names), in the draw order
listed per workload, then rounded to the activation dtype (round to nearest
even for bf16). Values ~ N(0, 1); W ~ N(0, 1/d) (variance 1/d); gate logits
~ N(0, 1) in fp32. Prefix lengths and the committing subset are drawn from
the same generator.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

N_LINEAR_LAYERS = 6  # layers {0, 4, 8, 12, 16, 18} of 20


@dataclass
class Workload:
    name: str
    H: int
    d: int
    f: int
    L: int
    dtype: torch.dtype
    tensors: dict = field(default_factory=dict)
    meta: dict = field(default_factory=dict)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(g, shape, dtype, device, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def _stack(blocks, shape, dtype, device) -> torch.Tensor:
    if blocks:
        return torch.stack(blocks)
    return torch.empty((0, *shape), dtype=dtype, device=device)


def _layer_params(g, H, d, f, dtype, device):
    W = _normal(g, (H, d, f), dtype, device, std=d ** -0.5)
    gate = torch.randn((H,), generator=g, dtype=torch.float32, device=device)
    return W, gate


def tiny(seed: int = 0, device="cpu", dtype=torch.float32) -> Workload:
    """1 request, 2 heads, d=16, f=8, L=4, three committed blocks.
    Draw order: W, gate, commit blocks (k then v, block by block), q, k, v."""
    H, d, f, L, B, nblk = 2, 16, 8, 4, 1, 3
    g = _gen(seed, device)
    W, gate = _layer_params(g, H, d, f, dtype, device)
    ck, cv = [], []
    for _ in range(nblk):
        ck.append(_normal(g, (B, L, H, d), dtype, device))
        cv.append(_normal(g, (B, L, H, d), dtype, device))
    q, k, v = (_normal(g, (B, L, H, d), dtype, device) for _ in range(3))
    return Workload("tiny: B=1 H=2 d=16 f=8 L=4, 3 committed blocks", H, d, f, L, dtype,
                    dict(W=W, gate=gate, commit_k=torch.stack(ck), commit_v=torch.stack(cv),
                         q=q, k=k, v=v), dict(B=B, n_blocks=nblk))


def single_layer(seed: int = 1, device="cpu", dtype=torch.bfloat16, n_blocks: int = 64) -> Workload:
    """1 request, 16 heads, d=128, f=64, L=32; 64 committed blocks (2,048
    tokens). Draw order as in ``tiny``."""
    H, d, f, L, B = 16, 128, 64, 32, 1
    g = _gen(seed, device)
    W, gate = _layer_params(g, H, d, f, dtype, device)
    ck, cv = [], []
    for _ in range(n_blocks):
        ck.append(_normal(g, (B, L, H, d), dtype, device))
        cv.append(_normal(g, (B, L, H, d), dtype, device))
    q, k, v = (_normal(g, (B, L, H, d), dtype, device) for _ in range(3))
    return Workload(f"single-layer decode: B=1 H=16 d=128 f=64 L=32, {n_blocks * L}-token prefix",
                    H, d, f, L, dtype,
                    dict(W=W, gate=gate, commit_k=_stack(ck, (B, L, H, d), dtype, device),
                         commit_v=_stack(cv, (B, L, H, d), dtype, device), q=q, k=k, v=v),
                    dict(B=B, n_blocks=n_blocks))


def continuous_batching(seed: int = 2, device="cpu", dtype=torch.bfloat16, B: int = 64,
                        lo: int = 8, hi: int = 128, n_commit: int = 16) -> Workload:
    """B requests with prefix lengths 32 * U{lo..hi} (256..4096 tokens),
    states to be built from the packed prefixes; one attend for all requests
    and a commit for ``n_commit`` of them (the first of a seeded permutation).
    Draw order: W, gate, lengths, prefix k, prefix v, q, k, v, permutation."""
    H, d, f, L = 16, 128, 64, 32
    g = _gen(seed, device)
    W, gate = _layer_params(g, H, d, f, dtype, device)
    lens = 32 * torch.randint(lo, hi + 1, (B,), generator=g, device=device)
    cu = torch.zeros(B + 1, dtype=torch.int64, device=device)
    cu[1:] = torch.cumsum(lens, 0)
    total = int(cu[-1])
    pk = _normal(g, (total, H, d), dtype, device)
    pv = _normal(g, (total, H, d), dtype, device)
    q, k, v = (_normal(g, (B, L, H, d), dtype, device) for _ in range(3))
    perm = torch.randperm(B, generator=g, device=device)
    commit_idx = perm[:n_commit].sort().values
    return Workload(f"continuous batching: B={B} H=16 d=128 f=64 L=32, prefixes 32*U{{{lo}..{hi}}},"
                    f" attend all + commit {n_commit}", H, d, f, L, dtype,
                    dict(W=W, gate=gate, prefix_k=pk, prefix_v=pv, cu_prefix=cu, q=q, k=k, v=v,
                         commit_idx=commit_idx),
                    dict(B=B, max_prefix=int(lens.max()), total_prefix=total))


def prompt_ingestion(seed: int = 3, device="cpu", dtype=torch.bfloat16, B: int = 8,
                     T: int = 8192) -> Workload:
    """B prompts of T tokens each, packed. Draw order: W, gate, k, v."""
    H, d, f, L = 16, 128, 64, 32
    g = _gen(seed, device)
    W, gate = _layer_params(g, H, d, f, dtype, device)
    k = _normal(g, (B * T, H, d), dtype, device)
    v = _normal(g, (B * T, H, d), dtype, device)
    cu = torch.arange(B + 1, dtype=torch.int64, device=device) * T
    return Workload(f"prompt ingestion: B={B} x T={T}, H=16 d=128 f=64", H, d, f, L, dtype,
                    dict(W=W, gate=gate, k=k, v=v, cu_seqlens=cu), dict(B=B, T=T))


def stack_layer(layer: int, B: int, seed: int = 4, device="cpu", dtype=torch.bfloat16,
                P: int = 2048) -> Workload:
    """One of the 6 linearized layers of the stack: B requests, each with a
    P-token prefix (state source and KV cache of the comparison path) and an
    active block. Layer l uses seed ``seed * 1000 + l``.
    Draw order: W, gate, prefix k, prefix v, q, k, v."""
    H, d, f, L = 16, 128, 64, 32
    g = _gen(seed * 1000 + layer, device)
    W, gate = _layer_params(g, H, d, f, dtype, device)
    pk = _normal(g, (B * P, H, d), dtype, device)
    pv = _normal(g, (B * P, H, d), dtype, device)
    q, k, v = (_normal(g, (B, L, H, d), dtype, device) for _ in range(3))
    cu = torch.arange(B + 1, dtype=torch.int64, device=device) * P
    return Workload(f"6-layer stack, layer {layer}: B={B}, P={P}", H, d, f, L, dtype,
                    dict(W=W, gate=gate, prefix_k=pk, prefix_v=pv, cu_prefix=cu, q=q, k=k, v=v),
                    dict(B=B, P=P, layer=layer))


def draw(seed: int, shape, dtype=torch.bfloat16, device="cpu", std: float = 1.0) -> torch.Tensor:
    """One seeded N(0, std^2) tensor, drawn in float32 and rounded to dtype
    (for ad-hoc shapes: ragged lengths, edge cases)."""
    return _normal(_gen(seed, device), tuple(shape), dtype, device, std=std)


def paged_cache(seed: int, k_cache: torch.Tensor, v_cache: torch.Tensor, lens,
                page_tokens: int, spare_pages: int = 3, fill: float = float("nan")):
    """Lays a packed per-request cache ``[sum P, H, d]`` out as a paged cache:
    each request's tokens go, ``page_tokens`` at a time, into pages at seeded
    random positions of one pool, with ``spare_pages`` pages that no request
    uses. Returns ``k_pages``, ``v_pages`` ``[num_pages, page_tokens, H, d]``,
    ``page_table`` ``[B, max_pages]`` int32 (entries past a request's last
    page are -1) and ``prefix_len`` ``[B]`` int32, on the cache's device.
    Unused pages and the slots past a request's last token hold ``fill``."""
    pt = int(page_tokens)
    n_pages = [-(-int(P) // pt) for P in lens]
    num_pages = sum(n_pages) + spare_pages
    perm = torch.randperm(num_pages, generator=_gen(seed, "cpu")).tolist()
    H, d = k_cache.shape[1:]
    dev, dt = k_cache.device, k_cache.dtype
    k_pages = torch.full((num_pages, pt, H, d), fill, dtype=dt, device=dev)
    v_pages = torch.full((num_pages, pt, H, d), fill, dtype=dt, device=dev)
    table = torch.full((len(lens), max(n_pages + [1])), -1, dtype=torch.int32)
    rows, used = [], 0
    for b, P in enumerate(lens):
        table[b, :n_pages[b]] = torch.tensor(perm[used:used + n_pages[b]], dtype=torch.int32)
        used += n_pages[b]
        t = torch.arange(int(P))
        rows.append(table[b, t // pt].long() * pt + t % pt)  # pool row of each token
    if rows:
        rows = torch.cat(rows).to(dev)
        k_pages.view(num_pages * pt, H, d)[rows] = k_cache
        v_pages.view(num_pages * pt, H, d)[rows] = v_cache
    prefix_len = torch.tensor([int(P) for P in lens], dtype=torch.int32)
    return k_pages, v_pages, table.to(dev), prefix_len.to(dev)

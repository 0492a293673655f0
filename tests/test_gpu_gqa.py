"""Grouped-query heads and separate query/key maps (GPU), through
hb_block_attend_ex and hb_prefill_attend_ex, against the oracle's attend_gqa
and prefill_attend on the same seeded inputs: every request's outputs, and
the committed states per key/value head."""

import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from tests.parity import (TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, assert_status_ok, f64, out_err,
                          unit_err)

pytestmark = pytest.mark.gpu

MERGES = {"shared_norm": hb.MERGE_SHARED_NORM, "convex": hb.MERGE_CONVEX}


def _problem(B, H, Hkv, dt, d=128, f=64, L=32, seed=0, same_maps=False, max_prefix=48):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, L, H, d), generator=g).to(dt)
    k = torch.randn((B, L, Hkv, d), generator=g).to(dt)
    v = torch.randn((B, L, Hkv, d), generator=g).to(dt)
    Wk = (torch.randn((Hkv, d, f), generator=g) * d ** -0.5).to(dt)
    if same_maps:
        Wq = Wk.repeat_interleave(H // Hkv, dim=0)
    else:
        Wq = (torch.randn((H, d, f), generator=g) * d ** -0.5).to(dt)
    gate = torch.randn((H,), generator=g)
    lens = torch.randint(0, max_prefix + 1, (B,), generator=g).tolist()
    states = []
    for n in lens:
        pk = torch.randn((n, Hkv, d), generator=g).to(dt)
        pv = torch.randn((n, Hkv, d), generator=g).to(dt)
        states.append(ob.prefill(f64(pk), f64(pv), f64(Wk)))
    slot_of = torch.randperm(B + 3, generator=g)[:B]
    commit = (torch.rand(B, generator=g) < 0.4).to(torch.int32)
    return dict(q=q, k=k, v=v, Wq=Wq, Wk=Wk, gate=gate, states=states, slot_of=slot_of,
                commit=commit, B=B, H=H, Hkv=Hkv, d=d, f=f, L=L)


def _pool(c, dev):
    S = torch.zeros((c["B"] + 3, c["Hkv"], 2 * c["f"], c["d"]), dtype=torch.float32)
    Z = torch.zeros((c["B"] + 3, c["Hkv"], 2 * c["f"]), dtype=torch.float32)
    for b in range(c["B"]):
        S[int(c["slot_of"][b])] = torch.as_tensor(c["states"][b][0], dtype=torch.float32)
        Z[int(c["slot_of"][b])] = torch.as_tensor(c["states"][b][1], dtype=torch.float32)
    return S.to(dev), Z.to(dev)


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("Hkv", [1, 4, 8, 16])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("with_commit", [False, True])
def test_attend_ex_matches_oracle(cuda_device, merge, Hkv, dt, with_commit):
    """16 query heads over 1, 4, 8 or 16 key/value heads, separate maps;
    bf16 takes the tensor-core attend, fp32 the generic kernel. With commits,
    the committing slots' per-key/value-head states match the oracle's
    commit with the key map, the others stay untouched."""
    c = _problem(12, 16, Hkv, dt, seed=Hkv + (100 if dt == torch.float32 else 0))
    cfg = hb.Config(16, 128, 64, 32, dtype=hb.DTYPE_BF16 if dt == torch.bfloat16 else hb.DTYPE_FP32,
                    merge=MERGES[merge])
    S, Z = _pool(c, cuda_device)
    S0, Z0 = S.clone(), Z.clone()
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    o = hb.hb_block_attend_ex(cfg, Hkv, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S, Z,
                              dev(c["Wq"]), dev(c["gate"]), Wk=dev(c["Wk"]),
                              commit=dev(c["commit"]) if with_commit else None)
    assert_status_ok()
    tol = TOL_OUT_BF16 if dt == torch.bfloat16 else TOL_OUT_FP32
    for b in range(c["B"]):
        S_old, Z_old = c["states"][b]
        ref = ob.attend_gqa(f64(c["q"][b]), f64(c["k"][b]), f64(c["v"][b]), S_old, Z_old,
                            f64(c["Wq"]), f64(c["gate"]), MERGES[merge])
        assert out_err(f64(o[b]), ref) <= tol, b
        slot = int(c["slot_of"][b])
        if with_commit and int(c["commit"][b]):
            S_new, Z_new = ob.commit(S_old, Z_old, f64(c["k"][b]), f64(c["v"][b]), f64(c["Wk"]))
            assert unit_err(f64(S[slot]), S_new, 1) <= TOL_STATE, b
            assert unit_err(f64(Z[slot]), Z_new, 1) <= TOL_STATE, b
        else:
            assert torch.equal(S[slot], S0[slot]) and torch.equal(Z[slot], Z0[slot]), b


def test_attend_ex_one_map_equals_fused_step(cuda_device):
    """With H_kv = H and one map, the extended call is the fused step: same
    output bits and states as hb_block_attend_commit."""
    c = _problem(20, 16, 16, torch.bfloat16, seed=5, same_maps=True)
    cfg = hb.Config(16, 128, 64, 32)
    S, Z = _pool(c, cuda_device)
    S2, Z2 = S.clone(), Z.clone()
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    W = dev(c["Wq"])
    o1 = hb.hb_block_attend_ex(cfg, 16, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S, Z, W,
                               dev(c["gate"]), Wk=W, commit=dev(c["commit"]))
    o2 = hb.hb_block_attend_commit(cfg, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S2, Z2, W,
                                   dev(c["gate"]), dev(c["commit"]))
    assert_status_ok()
    assert torch.equal(o1, o2) and torch.equal(S, S2) and torch.equal(Z, Z2)


def test_attend_ex_gqa_full_batch(cuda_device):
    """The continuous-batching batch (64 requests) with 16 query heads over 4
    key/value heads: every CTA runs several units of each group."""
    c = _problem(64, 16, 4, torch.bfloat16, seed=64, max_prefix=32)
    cfg = hb.Config(16, 128, 64, 32)
    S, Z = _pool(c, cuda_device)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    o = hb.hb_block_attend_ex(cfg, 4, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S, Z,
                              dev(c["Wq"]), dev(c["gate"]))
    assert_status_ok()
    o64 = f64(o)
    for b in range(64):
        ref = ob.attend_gqa(f64(c["q"][b]), f64(c["k"][b]), f64(c["v"][b]), *c["states"][b],
                            f64(c["Wq"]), f64(c["gate"]))
        assert out_err(o64[b], ref) <= TOL_OUT_BF16, b


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("Hkv", [16, 4])
@pytest.mark.parametrize("accumulate", [False, True])
def test_prefill_attend_ex_matches_oracle(cuda_device, merge, Hkv, accumulate):
    """Prompts of 6 blocks with separate maps: with H_kv = H one sequential
    launch keeps the key map on chip beside the state; with 4 key/value heads
    an attend and a commit launch per block. Every block's outputs and the
    final states against the oracle's prefill_attend."""
    B, T, H, d, f, L = 3, 192, 16, 128, 64, 32
    g = torch.Generator().manual_seed(Hkv + 7 * accumulate)
    q = torch.randn((B, T, H, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, T, Hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, T, Hkv, d), generator=g).to(torch.bfloat16)
    Wq = (torch.randn((H, d, f), generator=g) * d ** -0.5).to(torch.bfloat16)
    Wk = (torch.randn((Hkv, d, f), generator=g) * d ** -0.5).to(torch.bfloat16)
    gate = torch.randn((H,), generator=g)
    ctx = [(torch.randn((n, Hkv, d), generator=g).to(torch.bfloat16),
            torch.randn((n, Hkv, d), generator=g).to(torch.bfloat16)) for n in (0, 40, 7)]
    cfg = hb.Config(H, d, f, L, merge=MERGES[merge])
    S = torch.full((B + 1, Hkv, 2 * f, d), 5.0)
    Z = torch.full((B + 1, Hkv, 2 * f), 5.0)
    starts = []
    for b, (ck, cv) in enumerate(ctx):
        S0, Z0 = ob.prefill(f64(ck), f64(cv), f64(Wk))
        starts.append((S0, Z0) if accumulate else (None, None))
        if accumulate:
            S[b + 1] = torch.as_tensor(S0, dtype=torch.float32)
            Z[b + 1] = torch.as_tensor(Z0, dtype=torch.float32)
    S, Z = S.to(cuda_device), Z.to(cuda_device)
    sl = torch.tensor([1, 2, 3], dtype=torch.int32, device=cuda_device)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    o = hb.hb_prefill_attend_ex(cfg, Hkv, sl, dev(q), dev(k), dev(v), S, Z, dev(Wq), dev(Wk),
                                dev(gate), accumulate=accumulate)
    assert_status_ok()
    for b in range(B):
        o_ref, S_ref, Z_ref = ob.prefill_attend(f64(q[b]), f64(k[b]), f64(v[b]), f64(Wq),
                                                f64(gate), L, MERGES[merge], S0=starts[b][0],
                                                Z0=starts[b][1], Wk=f64(Wk))
        for j0 in range(0, T, L):
            assert out_err(f64(o[b, j0:j0 + L]), o_ref[j0:j0 + L]) <= TOL_OUT_BF16, (b, j0)
        assert unit_err(f64(S[b + 1]), S_ref, 1) <= TOL_STATE, b
        assert unit_err(f64(Z[b + 1]), Z_ref, 1) <= TOL_STATE, b
    assert bool((S[0] == 5.0).all())

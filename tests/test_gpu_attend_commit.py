"""hb_block_attend_commit (GPU): the output uses the state as it was before
the call, and the committing requests' states then hold the oracle's commit
of the same block; other slots are untouched. Also checked against the two
separate calls (hb_block_attend, then hb_commit_block on the subset)."""

import functools

import numpy as np
import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from linear_attention_diffusion_feature_b300 import inputs
from tests.parity import (TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, assert_status_ok, f64, new_pool,
                          out_err, slots, unit_err)

pytestmark = pytest.mark.gpu

MERGES = {"shared_norm": hb.MERGE_SHARED_NORM, "convex": hb.MERGE_CONVEX}


def _case(dt, d=128, f=64, L=32, H=16):
    prefix = [64, 96, 0, 32, 128, 160]
    commit = [1, 0, 1, 1, 0, 0]
    slot_of = [3, 0, 5, 1, 4, 2]
    B = len(prefix)
    W = inputs.draw(61, (H, d, f), dt, std=d ** -0.5)
    gate = inputs.draw(62, (H,), torch.float32)
    q, k, v = (inputs.draw(63 + i, (B, L, H, d), dt) for i in range(3))
    states = []
    for b, n in enumerate(prefix):
        pk = inputs.draw(70 + 2 * b, (n, H, d), dt)
        pv = inputs.draw(71 + 2 * b, (n, H, d), dt)
        states.append(ob.prefill(f64(pk), f64(pv), f64(W)))
    return dict(W=W, gate=gate, q=q, k=k, v=v, states=states, commit=commit, slot_of=slot_of,
                B=B, H=H, d=d, f=f, L=L)


def _pool(c, cfg, dev, num_slots=7):
    S, Z = new_pool(cfg, num_slots, dev)
    fill = inputs.draw(80, S.shape, torch.float32)  # slots no request names
    S.copy_(fill.to(dev))
    Z.copy_(fill[..., 0].abs().to(dev))
    for b, sl in enumerate(c["slot_of"]):
        S[sl] = torch.as_tensor(c["states"][b][0], dtype=torch.float32, device=dev)
        Z[sl] = torch.as_tensor(c["states"][b][1], dtype=torch.float32, device=dev)
    return S, Z


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_attend_commit_matches_oracle(cuda_device, merge, dt):
    c = _case(dt)
    cfg = hb.Config(c["H"], c["d"], c["f"], c["L"],
                    dtype=hb.DTYPE_BF16 if dt == torch.bfloat16 else hb.DTYPE_FP32,
                    merge=MERGES[merge])
    S, Z = _pool(c, cfg, cuda_device)
    S0, Z0 = S.clone(), Z.clone()
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    o = hb.hb_block_attend_commit(cfg, slots(c["slot_of"], cuda_device), dev(c["q"]), dev(c["k"]),
                                  dev(c["v"]), S, Z, dev(c["W"]), dev(c["gate"]),
                                  slots(c["commit"], cuda_device))
    assert_status_ok()
    tol = TOL_OUT_BF16 if dt == torch.bfloat16 else TOL_OUT_FP32
    W64 = f64(c["W"])
    for b, sl in enumerate(c["slot_of"]):
        S_old, Z_old = c["states"][b]
        ref = ob.attend(f64(c["q"][b]), f64(c["k"][b]), f64(c["v"][b]), S_old, Z_old, W64,
                        f64(c["gate"]), MERGES[merge])
        assert out_err(f64(o[b]), ref) <= tol, b
        if c["commit"][b]:
            S_new, Z_new = ob.commit(S_old, Z_old, f64(c["k"][b]), f64(c["v"][b]), W64)
        else:
            S_new, Z_new = f64(S0[sl]), f64(Z0[sl])
        assert unit_err(f64(S[sl]), S_new, 1) <= TOL_STATE, b
        assert unit_err(f64(Z[sl]), Z_new, 1) <= TOL_STATE, b
    assert torch.equal(S[6], S0[6]) and torch.equal(Z[6], Z0[6])


def test_attend_commit_equals_two_calls_at_full_size(cuda_device):
    """64 requests, 16 committing (the continuous-batching step): the output
    is the same bits as hb_block_attend's, the states match hb_commit_block's."""
    w = inputs.continuous_batching(seed=7, device=cuda_device, B=64, n_commit=16)
    t = w.tensors
    cfg = hb.Config(16, 128, 64, 32)
    sl = torch.arange(64, dtype=torch.int32, device=cuda_device)
    S, Z = new_pool(cfg, 64, cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                        w.meta["max_prefix"], t["W"], S, Z)
    S2, Z2 = S.clone(), Z.clone()
    mask = torch.zeros(64, dtype=torch.int32, device=cuda_device)
    mask[t["commit_idx"]] = 1
    o1 = hb.hb_block_attend_commit(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"], mask)
    o2 = hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S2, Z2, t["W"], t["gate"])
    ci = t["commit_idx"]
    hb.hb_commit_block(cfg, sl[ci].contiguous(), t["k"][ci].contiguous(), t["v"][ci].contiguous(),
                       t["W"], S2, Z2)
    assert_status_ok()
    assert torch.equal(o1, o2)
    assert unit_err(f64(S), f64(S2), 2) <= TOL_STATE
    assert unit_err(f64(Z), f64(Z2), 2) <= TOL_STATE
    untouched = torch.ones(64, dtype=torch.bool, device=cuda_device)
    untouched[ci] = False
    assert torch.equal(S[untouched], S2[untouched])


@pytest.mark.parametrize("pattern", ["none", "all"])
def test_attend_commit_mask_extremes(cuda_device, pattern):
    c = _case(torch.bfloat16)
    c["commit"] = [0] * c["B"] if pattern == "none" else [1] * c["B"]
    cfg = hb.Config(c["H"], c["d"], c["f"], c["L"])
    S, Z = _pool(c, cfg, cuda_device)
    S0 = S.clone()
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    hb.hb_block_attend_commit(cfg, slots(c["slot_of"], cuda_device), dev(c["q"]), dev(c["k"]),
                              dev(c["v"]), S, Z, dev(c["W"]), dev(c["gate"]),
                              slots(c["commit"], cuda_device))
    assert_status_ok()
    W64 = f64(c["W"])
    for b, sl in enumerate(c["slot_of"]):
        if pattern == "none":
            assert torch.equal(S[sl], S0[sl])
        else:
            S_new, _ = ob.commit(*c["states"][b], f64(c["k"][b]), f64(c["v"][b]), W64)
            assert unit_err(f64(S[sl]), S_new, 1) <= TOL_STATE


def test_attend_commit_bad_slot_is_skipped_and_flagged(cuda_device):
    c = _case(torch.bfloat16)
    cfg = hb.Config(c["H"], c["d"], c["f"], c["L"])
    S, Z = _pool(c, cfg, cuda_device)
    S0 = S.clone()
    bad = list(c["slot_of"])
    bad[2] = 99  # a committing request with a slot outside the pool
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    o = torch.full_like(dev(c["q"]), 7.0)
    hb.hb_block_attend_commit(cfg, slots(bad, cuda_device), dev(c["q"]), dev(c["k"]), dev(c["v"]),
                              S, Z, dev(c["W"]), dev(c["gate"]), slots(c["commit"], cuda_device),
                              o=o)
    st = hb.hb_get_device_status()
    assert st == 5  # HB_ERR_DEVICE_BOUNDS
    assert bool((o[2] == 7.0).all())  # no output for the skipped request
    W64 = f64(c["W"])
    for b, sl in enumerate(c["slot_of"]):
        if b == 2:
            continue
        if c["commit"][b]:
            S_new, _ = ob.commit(*c["states"][b], f64(c["k"][b]), f64(c["v"][b]), W64)
            assert unit_err(f64(S[sl]), S_new, 1) <= TOL_STATE
        else:
            assert torch.equal(S[sl], S0[sl])
    assert torch.equal(S[5], S0[5])  # the skipped request's real slot


@pytest.mark.parametrize("pattern", ["every_third", "last_only", "first_window_none"])
def test_attend_commit_schedules_any_mask(cuda_device, pattern):
    """The kernel orders committing requests' units first; with 100 requests
    (four 32-request windows of the mask) and permuted slots, any mask gives
    the two separate calls' result."""
    B, H = 100, 16
    cfg = hb.Config(H, 128, 64, 32)
    g = torch.Generator().manual_seed(5)
    q, k, v = (inputs.draw(90 + i, (B, 32, H, 128), torch.bfloat16).to(cuda_device)
               for i in range(3))
    W = inputs.draw(93, (H, 128, 64), torch.bfloat16, std=128 ** -0.5).to(cuda_device)
    gate = inputs.draw(94, (H,), torch.float32).to(cuda_device)
    perm = torch.randperm(B, generator=g).to(torch.int32).to(cuda_device)
    flags = {"every_third": [b % 3 == 0 for b in range(B)],
             "last_only": [b == B - 1 for b in range(B)],
             "first_window_none": [b >= 32 and b % 2 == 1 for b in range(B)]}[pattern]
    mask = torch.tensor(flags, dtype=torch.int32, device=cuda_device)
    S, Z = new_pool(cfg, B, cuda_device)
    S.copy_(inputs.draw(95, S.shape, torch.float32).to(cuda_device) * 1e-2)
    Z.copy_(inputs.draw(96, Z.shape, torch.float32).abs().to(cuda_device) + 1.0)
    S2, Z2 = S.clone(), Z.clone()
    o1 = hb.hb_block_attend_commit(cfg, perm, q, k, v, S, Z, W, gate, mask)
    o2 = hb.hb_block_attend(cfg, perm, q, k, v, S2, Z2, W, gate)
    ci = torch.nonzero(mask).flatten()
    hb.hb_commit_block(cfg, perm[ci].contiguous(), k[ci].contiguous(), v[ci].contiguous(), W,
                       S2, Z2)
    assert_status_ok()
    assert torch.equal(o1, o2)
    assert unit_err(f64(S), f64(S2), 2) <= TOL_STATE
    assert unit_err(f64(Z), f64(Z2), 2) <= TOL_STATE
    untouched = torch.ones(B, dtype=torch.bool, device=cuda_device)
    untouched[perm[ci].long()] = False
    assert torch.equal(S[untouched], S2[untouched])


def test_attend_commit_many_units_per_cta(cuda_device):
    """700 requests: every CTA runs more than 64 units, so the kernel's unit
    table moves through several 32-unit windows; the result is still that of
    the two separate calls."""
    B, H = 700, 16
    cfg = hb.Config(H, 128, 64, 32)
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn((B, 32, H, 128), generator=g).to(torch.bfloat16).to(cuda_device)
               for _ in range(3))
    W = (torch.randn((H, 128, 64), generator=g) * 128 ** -0.5).to(torch.bfloat16).to(cuda_device)
    gate = torch.randn((H,), generator=g).to(cuda_device)
    perm = torch.randperm(B, generator=g).to(torch.int32).to(cuda_device)
    mask = (torch.rand(B, generator=g) < 0.3).to(torch.int32).to(cuda_device)
    S, Z = new_pool(cfg, B, cuda_device)
    S.copy_(torch.randn(S.shape, generator=g).to(cuda_device) * 1e-2)
    Z.copy_(torch.rand(Z.shape, generator=g).to(cuda_device) + 1.0)
    S2, Z2 = S.clone(), Z.clone()
    o1 = hb.hb_block_attend_commit(cfg, perm, q, k, v, S, Z, W, gate, mask)
    o2 = hb.hb_block_attend(cfg, perm, q, k, v, S2, Z2, W, gate)
    ci = torch.nonzero(mask).flatten()
    hb.hb_commit_block(cfg, perm[ci].contiguous(), k[ci].contiguous(), v[ci].contiguous(), W,
                       S2, Z2)
    assert_status_ok()
    assert torch.equal(o1, o2)
    assert unit_err(f64(S), f64(S2), 2) <= TOL_STATE
    assert unit_err(f64(Z), f64(Z2), 2) <= TOL_STATE


@functools.lru_cache(maxsize=2)
def _oracle_inputs(B, H, seed, commit_frac=0.25, spare=5, max_prefix=64):
    """Host side of a batch of B requests of the production shape: seeded
    activations, states the oracle builds from short seeded prefixes
    (0 .. max_prefix tokens), permuted slots of a pool with ``spare`` unused
    slots, and a seeded commit mask (shared by both merges' tests)."""
    d, f, L = 128, 64, 32
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn((H, d, f), generator=g) * d ** -0.5).to(torch.bfloat16)
    gate = torch.randn((H,), generator=g)
    q, k, v = (torch.randn((B, L, H, d), generator=g).to(torch.bfloat16) for _ in range(3))
    lens = torch.randint(0, max_prefix + 1, (B,), generator=g).tolist()
    W64 = f64(W)
    states = []
    for n in lens:
        pk = torch.randn((n, H, d), generator=g).to(torch.bfloat16)
        pv = torch.randn((n, H, d), generator=g).to(torch.bfloat16)
        states.append(ob.prefill(f64(pk), f64(pv), W64))
    slot_of = torch.randperm(B + spare, generator=g)[:B]
    commit = (torch.rand(B, generator=g) < commit_frac).to(torch.int32)
    fill_S = torch.randn((B + spare, H, 2 * f, d), generator=g)  # slots no request names
    fill_Z = torch.rand((B + spare, H, 2 * f), generator=g) + 1.0
    return dict(W=W, gate=gate, q=q, k=k, v=v, states=states, slot_of=slot_of, commit=commit,
                fill_S=fill_S, fill_Z=fill_Z, B=B, spare=spare)


def _oracle_pool(c, device):
    S = c["fill_S"].clone()
    Z = c["fill_Z"].clone()
    for b in range(c["B"]):
        S[int(c["slot_of"][b])] = torch.as_tensor(c["states"][b][0], dtype=torch.float32)
        Z[int(c["slot_of"][b])] = torch.as_tensor(c["states"][b][1], dtype=torch.float32)
    return S.to(device), Z.to(device)


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("B", [64, 320])
def test_attend_commit_every_request_matches_oracle(cuda_device, merge, B):
    """The fused step against the oracle on every request, not a sample: at 64
    requests (the continuous-batching step) and at 320 requests, where every
    CTA runs more than 32 units, so the unit table moves to a second window
    and both ring stages wrap many times. Each output is checked against the
    oracle's attend on the state as it was before the call; each committing
    slot's S and Z against the oracle's commit; the other slots must be
    untouched."""
    c = _oracle_inputs(B, 16, seed=300 + B)
    cfg = hb.Config(16, 128, 64, 32, merge=MERGES[merge])
    S, Z = _oracle_pool(c, cuda_device)
    S0, Z0 = S.clone(), Z.clone()
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    o = hb.hb_block_attend_commit(cfg, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S, Z,
                                  dev(c["W"]), dev(c["gate"]), dev(c["commit"]))
    assert_status_ok()
    W64, g64 = f64(c["W"]), f64(c["gate"])
    o64, S64, Z64 = f64(o), f64(S), f64(Z)
    named = set(int(x) for x in c["slot_of"])
    for b in range(B):
        S_old, Z_old = c["states"][b]
        q64, k64, v64 = f64(c["q"][b]), f64(c["k"][b]), f64(c["v"][b])
        ref = ob.attend(q64, k64, v64, S_old, Z_old, W64, g64, MERGES[merge])
        assert out_err(o64[b], ref) <= TOL_OUT_BF16, b
        slot = int(c["slot_of"][b])
        if int(c["commit"][b]):
            S_new, Z_new = ob.commit(S_old, Z_old, k64, v64, W64)
            assert unit_err(S64[slot], S_new, 1) <= TOL_STATE, b
            assert unit_err(Z64[slot], Z_new, 1) <= TOL_STATE, b
        else:
            assert torch.equal(S[slot], S0[slot]) and torch.equal(Z[slot], Z0[slot]), b
    for slot in range(B + c["spare"]):
        if slot not in named:
            assert torch.equal(S[slot], S0[slot]) and torch.equal(Z[slot], Z0[slot]), slot

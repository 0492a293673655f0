"""hb_block_attend_s16 on the bf16 copy of the states (GPU): the copy written
by hb_state_to_bf16 is torch's round-to-nearest conversion of the fp32
states bit for bit, and the attend's output on it is bit-identical to
hb_block_attend's on the fp32 states, hence to the oracle within the bf16
bound."""

import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from linear_attention_diffusion_feature_b300 import inputs
from tests.parity import TOL_OUT_BF16, assert_status_ok, config, f64, new_pool, out_err

pytestmark = pytest.mark.gpu

MERGES = {"shared_norm": hb.MERGE_SHARED_NORM, "convex": hb.MERGE_CONVEX}


def _scattered_slots(B, spare, seed, device):
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(B + spare, generator=g)[:B].to(torch.int32).to(device)


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("B", [64, 100])
def test_attend_s16_is_bit_identical(cuda_device, merge, B):
    w = inputs.continuous_batching(device=cuda_device, B=B, n_commit=0)
    cfg = config(w, MERGES[merge])
    t = w.tensors
    S, Z = new_pool(cfg, B + 5, cuda_device)
    sl = _scattered_slots(B, 5, 11, cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                        w.meta["max_prefix"], t["W"], S, Z)
    S16 = torch.zeros(S.shape, dtype=torch.bfloat16, device=cuda_device)
    hb.hb_state_to_bf16(cfg, sl, S, S16)
    assert_status_ok()
    idx = sl.long()
    assert torch.equal(S16[idx], S[idx].to(torch.bfloat16))
    unused = torch.ones(B + 5, dtype=torch.bool, device=cuda_device)
    unused[idx] = False
    assert bool((S16[unused] == 0).all())
    o32 = hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"])
    o16 = hb.hb_block_attend_s16(cfg, sl, t["q"], t["k"], t["v"], S16, Z, t["W"], t["gate"])
    assert_status_ok()
    assert torch.equal(o16, o32)
    cu = t["cu_prefix"].cpu()
    for b in (0, B - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        S_ref, Z_ref = ob.prefill(f64(t["prefix_k"][a:e]), f64(t["prefix_v"][a:e]), f64(t["W"]))
        ref = ob.attend(f64(t["q"][b]), f64(t["k"][b]), f64(t["v"][b]), S_ref, Z_ref,
                        f64(t["W"]), f64(t["gate"]), MERGES[merge])
        assert out_err(f64(o16[b]), ref) <= TOL_OUT_BF16


def test_attend_s16_bad_slot_flagged(cuda_device):
    w = inputs.continuous_batching(device=cuda_device, B=4, lo=8, hi=9, n_commit=0)
    cfg = config(w)
    t = w.tensors
    S, Z = new_pool(cfg, 4, cuda_device)
    sl = torch.arange(4, dtype=torch.int32, device=cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                        w.meta["max_prefix"], t["W"], S, Z)
    S16 = torch.zeros(S.shape, dtype=torch.bfloat16, device=cuda_device)
    hb.hb_state_to_bf16(cfg, torch.tensor([0, 1, 2, 9], dtype=torch.int32, device=cuda_device),
                        S, S16)
    assert hb.hb_get_device_status() == 5
    assert bool((S16[3] == 0).all())
    hb.hb_state_to_bf16(cfg, sl, S, S16)
    assert_status_ok()
    o = torch.full_like(t["q"], 7.0)
    bad = torch.tensor([0, 4, 2, -1], dtype=torch.int32, device=cuda_device)
    hb.hb_block_attend_s16(cfg, bad, t["q"], t["k"], t["v"], S16, Z, t["W"], t["gate"], o=o)
    assert hb.hb_get_device_status() == 5
    assert bool((o[1] == 7.0).all()) and bool((o[3] == 7.0).all())
    ref = hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"])
    assert torch.equal(o[0], ref[0]) and torch.equal(o[2], ref[2])


def test_attend_s16_after_commits_and_refresh(cuda_device):
    """The copy's life cycle in a decoding loop: the fp32 master changes
    through hb_block_attend_commit (one subset of requests) and then through
    hb_commit_block (another subset); after each change only the changed
    slots' copies are refreshed, and the attend on the copies stays
    bit-identical to the attend on the masters for every request."""
    B = 64
    w = inputs.continuous_batching(device=cuda_device, B=B, n_commit=16)
    cfg = config(w)
    t = w.tensors
    S, Z = new_pool(cfg, B + 5, cuda_device)
    sl = _scattered_slots(B, 5, 13, cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                        w.meta["max_prefix"], t["W"], S, Z)
    S16 = torch.zeros(S.shape, dtype=torch.bfloat16, device=cuda_device)
    hb.hb_state_to_bf16(cfg, sl, S, S16)
    # the fused step commits the first subset
    ci = t["commit_idx"]
    mask = torch.zeros(B, dtype=torch.int32, device=cuda_device)
    mask[ci] = 1
    S_before = S.clone()
    hb.hb_block_attend_commit(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"], mask)
    assert not torch.equal(S[sl[ci].long()], S_before[sl[ci].long()])
    hb.hb_state_to_bf16(cfg, sl[ci].contiguous(), S, S16)
    o32 = hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"])
    o16 = hb.hb_block_attend_s16(cfg, sl, t["q"], t["k"], t["v"], S16, Z, t["W"], t["gate"])
    assert_status_ok()
    assert torch.equal(o16, o32)
    # a separate commit of another subset (requests 1, 3, 5, ...)
    other = torch.arange(1, B, 2, device=cuda_device)
    hb.hb_commit_block(cfg, sl[other].contiguous(), t["q"][other].contiguous(),
                       t["v"][other].contiguous(), t["W"], S, Z)
    hb.hb_state_to_bf16(cfg, sl[other].contiguous(), S, S16)
    o32 = hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"])
    o16 = hb.hb_block_attend_s16(cfg, sl, t["q"], t["k"], t["v"], S16, Z, t["W"], t["gate"])
    assert_status_ok()
    assert torch.equal(o16, o32)
    assert torch.equal(S16[sl.long()], S[sl.long()].to(torch.bfloat16))


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("B", [64, 320])
def test_attend_commit_s16_equals_fp32_step(cuda_device, merge, B):
    """The dual-copy step (copies read for requests that do not commit,
    masters read and both written for committing ones) gives the fp32 step's
    output, masters and Z bit for bit, leaves every listed slot's copy equal
    to the round-to-nearest of its new master, and keeps doing so over a
    second step with another commit mask. 320 requests make every CTA run
    more than 32 units."""
    w = inputs.continuous_batching(device=cuda_device, B=B, n_commit=B // 4, lo=2, hi=16)
    cfg = config(w, MERGES[merge])
    t = w.tensors
    S, Z = new_pool(cfg, B + 5, cuda_device)
    sl = _scattered_slots(B, 5, 17, cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                        w.meta["max_prefix"], t["W"], S, Z)
    S16 = torch.full(S.shape, 3.0, dtype=torch.bfloat16, device=cuda_device)
    hb.hb_state_to_bf16(cfg, sl, S, S16)
    S_ref, Z_ref = S.clone(), Z.clone()
    g = torch.Generator().manual_seed(B)
    idx = sl.long()
    unused = torch.ones(B + 5, dtype=torch.bool, device=cuda_device)
    unused[idx] = False
    for step in range(2):
        mask = (torch.rand(B, generator=g) < 0.25).to(torch.int32).to(cuda_device)
        o_ref = hb.hb_block_attend_commit(cfg, sl, t["q"], t["k"], t["v"], S_ref, Z_ref, t["W"],
                                          t["gate"], mask)
        o = hb.hb_block_attend_commit_s16(cfg, sl, t["q"], t["k"], t["v"], S, S16, Z, t["W"],
                                          t["gate"], mask)
        assert_status_ok()
        assert torch.equal(o, o_ref), step
        assert torch.equal(S, S_ref), step
        assert torch.equal(Z, Z_ref), step
        assert torch.equal(S16[idx], S[idx].to(torch.bfloat16)), step
        assert bool((S16[unused] == 3.0).all()), step


@pytest.mark.parametrize("merge", sorted(MERGES))
def test_attend_commit_s16_matches_oracle(cuda_device, merge):
    """The dual-copy step against the oracle on every one of 64 requests:
    outputs from the state before the call, and the committing slots' new
    master and its copy from the oracle's commit."""
    from tests.parity import TOL_STATE, unit_err
    from tests.test_gpu_attend_commit import _oracle_inputs, _oracle_pool

    c = _oracle_inputs(64, 16, seed=364)
    cfg = hb.Config(16, 128, 64, 32, merge=MERGES[merge])
    S, Z = _oracle_pool(c, cuda_device)
    S16 = S.to(torch.bfloat16)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    o = hb.hb_block_attend_commit_s16(cfg, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S, S16, Z,
                                      dev(c["W"]), dev(c["gate"]), dev(c["commit"]))
    assert_status_ok()
    W64, g64 = f64(c["W"]), f64(c["gate"])
    o64, S64, S1664 = f64(o), f64(S), f64(S16)
    for b in range(64):
        S_old, Z_old = c["states"][b]
        q64, k64, v64 = f64(c["q"][b]), f64(c["k"][b]), f64(c["v"][b])
        ref = ob.attend(q64, k64, v64, S_old, Z_old, W64, g64, MERGES[merge])
        assert out_err(o64[b], ref) <= TOL_OUT_BF16, b
        if int(c["commit"][b]):
            slot = int(c["slot_of"][b])
            S_new, _ = ob.commit(S_old, Z_old, k64, v64, W64)
            assert unit_err(S64[slot], S_new, 1) <= TOL_STATE, b
            # the copy is the master rounded to bf16: within 2^-8 relative
            assert unit_err(S1664[slot], S_new, 1) <= 2.0 ** -8, b

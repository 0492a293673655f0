"""hb_block_attend against the oracle (GPU), end to end: the GPU state comes
from the library's own commit/prefill, the oracle's from its own sums."""

import numpy as np
import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from linear_attention_diffusion_feature_b300 import inputs
from tests.parity import (TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, assert_status_ok, config, f64,
                          new_pool, out_err, slots, unit_err)

pytestmark = pytest.mark.gpu

MERGES = {"shared_norm": hb.MERGE_SHARED_NORM, "convex": hb.MERGE_CONVEX}


def _tol(w):
    return TOL_OUT_BF16 if w.dtype == torch.bfloat16 else TOL_OUT_FP32


def _committed_single(w, cuda_device, cfg):
    """Commits the workload's blocks through the library and the oracle."""
    S, Z = new_pool(cfg, 2, cuda_device)
    W = w.tensors["W"].to(cuda_device)
    S_ref = np.zeros((w.H, 2 * w.f, w.d))
    Z_ref = np.zeros((w.H, 2 * w.f))
    ck, cv = w.tensors["commit_k"], w.tensors["commit_v"]
    for blk in range(ck.shape[0]):
        hb.hb_commit_block(cfg, slots([1], cuda_device), ck[blk].to(cuda_device),
                           cv[blk].to(cuda_device), W, S, Z)
        S_ref, Z_ref = ob.commit(S_ref, Z_ref, f64(ck[blk][0]), f64(cv[blk][0]),
                                 f64(w.tensors["W"]))
    return S, Z, S_ref, Z_ref


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("maker", ["tiny", "single_layer", "single_layer_fp32"])
def test_attend_single_request(cuda_device, merge, maker):
    w = {"tiny": inputs.tiny, "single_layer": inputs.single_layer,
         "single_layer_fp32": lambda: inputs.single_layer(dtype=torch.float32)}[maker]()
    cfg = config(w, MERGES[merge])
    S, Z, S_ref, Z_ref = _committed_single(w, cuda_device, cfg)
    t = {k: x.to(cuda_device) for k, x in w.tensors.items()}
    o = hb.hb_block_attend(cfg, slots([1], cuda_device), t["q"], t["k"], t["v"], S, Z, t["W"],
                           t["gate"])
    assert_status_ok()
    ref = ob.attend(f64(w.tensors["q"][0]), f64(w.tensors["k"][0]), f64(w.tensors["v"][0]),
                    S_ref, Z_ref, f64(w.tensors["W"]), f64(w.tensors["gate"]), MERGES[merge])
    assert out_err(f64(o[0]), ref) <= _tol(w)


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_attend_empty_state_is_softmax_attention(cuda_device, merge, dt):
    w = inputs.single_layer(dtype=dt, n_blocks=0)
    cfg = config(w, MERGES[merge])
    S, Z = new_pool(cfg, 1, cuda_device)
    t = {k: x.to(cuda_device) for k, x in w.tensors.items() if not k.startswith("commit")}
    o = hb.hb_block_attend(cfg, slots([0], cuda_device), t["q"], t["k"], t["v"], S, Z, t["W"],
                           t["gate"])
    assert_status_ok()
    ref = ob.softmax_kv_attend(np.zeros((0, w.H, w.d)), np.zeros((0, w.H, w.d)),
                               f64(w.tensors["q"][0]), f64(w.tensors["k"][0]),
                               f64(w.tensors["v"][0]))
    assert out_err(f64(o[0]), ref) <= _tol(w)


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("g", [-30.0, -4.0, 0.0, 4.0, 30.0])
def test_attend_gate_range(cuda_device, merge, g):
    """Gate logits from nearly-pure linear to nearly-pure softmax."""
    w = inputs.single_layer(n_blocks=8)
    cfg = config(w, MERGES[merge])
    S, Z, S_ref, Z_ref = _committed_single(w, cuda_device, cfg)
    gate = torch.full((w.H,), g, dtype=torch.float32)
    t = {k: x.to(cuda_device) for k, x in w.tensors.items()}
    o = hb.hb_block_attend(cfg, slots([1], cuda_device), t["q"], t["k"], t["v"], S, Z, t["W"],
                           gate.to(cuda_device))
    assert_status_ok()
    ref = ob.attend(f64(w.tensors["q"][0]), f64(w.tensors["k"][0]), f64(w.tensors["v"][0]),
                    S_ref, Z_ref, f64(w.tensors["W"]), f64(gate), MERGES[merge])
    assert out_err(f64(o[0]), ref) <= TOL_OUT_BF16


@pytest.mark.parametrize("merge", sorted(MERGES))
def test_continuous_batching_step(cuda_device, merge):
    """64 requests with ragged prefixes: states by prefill, one attend for all,
    then a commit for 16 of them; sampled requests are checked by the oracle
    (attend output and the committed state)."""
    w = inputs.continuous_batching(device=cuda_device)
    cfg = config(w, MERGES[merge])
    t = w.tensors
    B = w.meta["B"]
    num_slots = B + 7
    perm_slots = torch.randperm(num_slots, generator=torch.Generator().manual_seed(5))[:B]
    sl = perm_slots.to(torch.int32).to(cuda_device)
    S, Z = new_pool(cfg, num_slots, cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                        w.meta["max_prefix"], t["W"], S, Z)
    o = hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"])
    ci = t["commit_idx"]
    ck = t["k"][ci].contiguous()
    cv = t["v"][ci].contiguous()
    S_before = S.clone()
    Z_before = Z.clone()
    hb.hb_commit_block(cfg, sl[ci], ck, cv, t["W"], S, Z)
    assert_status_ok()
    cu = t["cu_prefix"].cpu()
    W64 = f64(t["W"])
    committing = set(ci.cpu().tolist())
    for b in [0, 1, 17, 40, 63] + sorted(committing)[:2]:
        a, e = int(cu[b]), int(cu[b + 1])
        S_ref, Z_ref = ob.prefill(f64(t["prefix_k"][a:e]), f64(t["prefix_v"][a:e]), W64)
        ref = ob.attend(f64(t["q"][b]), f64(t["k"][b]), f64(t["v"][b]), S_ref, Z_ref, W64,
                        f64(t["gate"]), MERGES[merge])
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16, b
        slot = int(perm_slots[b])
        if b in committing:
            S2, Z2 = ob.commit(S_ref, Z_ref, f64(t["k"][b]), f64(t["v"][b]), W64)
            assert unit_err(f64(S[slot]), S2, 1) <= TOL_STATE
            assert unit_err(f64(Z[slot]), Z2, 1) <= TOL_STATE
        else:
            assert torch.equal(S[slot], S_before[slot]) and torch.equal(Z[slot], Z_before[slot])


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("B", [1, 16, 256])
def test_stack_layer(cuda_device, B, merge):
    """One layer of the 6-layer stack shape (2,048-token prefixes), up to the
    largest batch the stack is timed at (256 requests), in both merges,
    sampled at the first, middle and last request."""
    w = inputs.stack_layer(2, B, device=cuda_device)
    cfg = config(w, MERGES[merge])
    t = w.tensors
    S, Z = new_pool(cfg, B, cuda_device)
    sl = slots(range(B), cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"], w.meta["P"], t["W"],
                        S, Z)
    o = hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"])
    assert_status_ok()
    P = w.meta["P"]
    for b in sorted({0, B // 2, B - 1}):
        S_ref, Z_ref = ob.prefill(f64(t["prefix_k"][b * P:(b + 1) * P]),
                                  f64(t["prefix_v"][b * P:(b + 1) * P]), f64(t["W"]))
        ref = ob.attend(f64(t["q"][b]), f64(t["k"][b]), f64(t["v"][b]), S_ref, Z_ref,
                        f64(t["W"]), f64(t["gate"]), MERGES[merge])
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16


def test_attend_deterministic(cuda_device):
    w = inputs.continuous_batching(device=cuda_device, B=8, lo=8, hi=16, n_commit=0)
    cfg = config(w)
    t = w.tensors
    S, Z = new_pool(cfg, 8, cuda_device)
    sl = slots(range(8), cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                        w.meta["max_prefix"], t["W"], S, Z)
    o1 = hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"])
    o2 = hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"])
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("merge", sorted(MERGES))
def test_separate_query_and_key_feature_maps(cuda_device, merge):
    """Separate feature maps for queries (Wq) and keys (Wk) through the
    unfused calls: the state is built with Wk (hb_prefill_state, then
    hb_commit_block of the active block) and read with Wq (hb_block_attend,
    whose W only maps the queries). The oracle is the token-by-token sum with
    weights phi_Wq(q) . phi_Wk(k_t)."""
    B = 4
    w = inputs.continuous_batching(device=cuda_device, B=B, lo=8, hi=16, n_commit=0)
    cfg = config(w, MERGES[merge])
    t = w.tensors
    Wq = t["W"]
    Wk = inputs.draw(77, tuple(Wq.shape), device=cuda_device, std=128 ** -0.5)
    S, Z = new_pool(cfg, B, cuda_device)
    sl = slots(range(B), cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                        w.meta["max_prefix"], Wk, S, Z)
    q2 = inputs.draw(78, tuple(t["q"].shape), device=cuda_device)
    k2 = inputs.draw(79, tuple(t["k"].shape), device=cuda_device)
    v2 = inputs.draw(80, tuple(t["v"].shape), device=cuda_device)
    hb.hb_commit_block(cfg, sl, t["k"], t["v"], Wk, S, Z)  # the block before the active one
    o = hb.hb_block_attend(cfg, sl, q2, k2, v2, S, Z, Wq, t["gate"])
    assert_status_ok()
    cu = t["cu_prefix"].cpu()
    for b in (0, B - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        k_prev = np.concatenate([f64(t["prefix_k"][a:e]), f64(t["k"][b])])
        v_prev = np.concatenate([f64(t["prefix_v"][a:e]), f64(t["v"][b])])
        ref = ob.attend_bruteforce(f64(q2[b]), f64(k2[b]), f64(v2[b]), k_prev, v_prev, f64(Wq),
                                   f64(t["gate"]), MERGES[merge], Wk=f64(Wk))
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16, b

"""hb_commit_block, hb_prefill_state and hb_state_zero against the oracle's
state sums (GPU). S and Z must match within 1e-4 (worst head, relative to
that head's largest entry)."""

import numpy as np
import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from linear_attention_diffusion_feature_b300 import inputs
from tests.parity import TOL_STATE, assert_status_ok, config, f64, new_pool, slots, unit_err

pytestmark = pytest.mark.gpu


def _state_err(S_gpu, Z_gpu, S_ref, Z_ref):
    return max(unit_err(S_gpu, S_ref, 1), unit_err(Z_gpu, Z_ref, 1))


@pytest.mark.parametrize("maker", ["tiny", "single_layer", "single_layer_fp32"])
def test_commit_blocks_one_by_one(cuda_device, maker):
    if maker == "tiny":
        w = inputs.tiny()
    elif maker == "single_layer":
        w = inputs.single_layer()
    else:
        w = inputs.single_layer(dtype=torch.float32)
    cfg = config(w)
    S, Z = new_pool(cfg, 3, cuda_device)
    sl = slots([1], cuda_device)
    W = w.tensors["W"].to(cuda_device)
    ck, cv = w.tensors["commit_k"], w.tensors["commit_v"]
    S_ref = np.zeros((w.H, 2 * w.f, w.d))
    Z_ref = np.zeros((w.H, 2 * w.f))
    for blk in range(ck.shape[0]):
        hb.hb_commit_block(cfg, sl, ck[blk].to(cuda_device), cv[blk].to(cuda_device), W, S, Z)
        S_ref, Z_ref = ob.commit(S_ref, Z_ref, f64(ck[blk][0]), f64(cv[blk][0]), f64(w.tensors["W"]))
    assert_status_ok()
    assert _state_err(f64(S[1]), f64(Z[1]), S_ref, Z_ref) <= TOL_STATE
    assert float(S[0].abs().max()) == 0.0 and float(S[2].abs().max()) == 0.0


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_commit_batch_into_scattered_slots(cuda_device, dt):
    H, d, f, L, B = 4, 128, 64, 32, 5
    cfg = hb.Config(H, d, f, L, dtype=hb.DTYPE_BF16 if dt == torch.bfloat16 else hb.DTYPE_FP32)
    S, Z = new_pool(cfg, 9, cuda_device)
    S0 = inputs.draw(1, S.shape, torch.float32)
    Z0 = inputs.draw(2, Z.shape, torch.float32).abs()
    S.copy_(S0)
    Z.copy_(Z0)
    W = inputs.draw(3, (H, d, f), dt, std=d ** -0.5)
    k = inputs.draw(4, (B, L, H, d), dt)
    v = inputs.draw(5, (B, L, H, d), dt)
    idx = [7, 0, 3, 8, 5]
    hb.hb_commit_block(cfg, slots(idx, cuda_device), k.to(cuda_device), v.to(cuda_device),
                       W.to(cuda_device), S, Z)
    assert_status_ok()
    for b, sl in enumerate(idx):
        S_ref, Z_ref = ob.commit(f64(S0[sl]), f64(Z0[sl]), f64(k[b]), f64(v[b]), f64(W))
        assert _state_err(f64(S[sl]), f64(Z[sl]), S_ref, Z_ref) <= TOL_STATE
    for sl in (1, 2, 4, 6):  # untouched slots
        assert torch.equal(S[sl].cpu(), S0[sl]) and torch.equal(Z[sl].cpu(), Z0[sl])


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("accumulate", [False, True])
def test_prefill_ragged(cuda_device, dt, accumulate):
    H, d, f = 4, 128, 64
    lens = [0, 1, 31, 32, 129, 700]
    B = len(lens)
    cfg = hb.Config(H, d, f, 32, dtype=hb.DTYPE_BF16 if dt == torch.bfloat16 else hb.DTYPE_FP32)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    total = int(cu[-1])
    k = inputs.draw(6, (total, H, d), dt)
    v = inputs.draw(7, (total, H, d), dt)
    W = inputs.draw(8, (H, d, f), dt, std=d ** -0.5)
    S, Z = new_pool(cfg, B + 2, cuda_device)
    S0 = inputs.draw(9, S.shape, torch.float32)
    Z0 = inputs.draw(10, Z.shape, torch.float32).abs()
    S.copy_(S0)
    Z.copy_(Z0)
    idx = [2, 4, 6, 1, 3, 5]
    hb.hb_prefill_state(cfg, slots(idx, cuda_device), k.to(cuda_device), v.to(cuda_device),
                        cu.to(cuda_device), max(lens), W.to(cuda_device), S, Z,
                        accumulate=accumulate)
    assert_status_ok()
    for b, sl in enumerate(idx):
        a, e = int(cu[b]), int(cu[b + 1])
        S_ref, Z_ref = ob.prefill(f64(k[a:e]), f64(v[a:e]), f64(W))
        if accumulate:
            S_ref = S_ref + f64(S0[sl])
            Z_ref = Z_ref + f64(Z0[sl])
        assert _state_err(f64(S[sl]), f64(Z[sl]), S_ref, Z_ref) <= TOL_STATE
    assert torch.equal(S[0].cpu(), S0[0])


def test_prefill_prompt_ingestion_full_size(cuda_device):
    """8 prompts x 8,192 tokens at full size; the oracle checks a sample of
    (request, head) units."""
    w = inputs.prompt_ingestion(device=cuda_device)
    cfg = config(w)
    S, Z = new_pool(cfg, 8, cuda_device)
    t = w.tensors
    hb.hb_prefill_state(cfg, slots(range(8), cuda_device), t["k"], t["v"], t["cu_seqlens"],
                        w.meta["T"], t["W"], S, Z)
    assert_status_ok()
    T = w.meta["T"]
    for b, h in [(0, 0), (3, 7), (7, 15), (5, 2)]:
        kk = f64(t["k"][b * T:(b + 1) * T, h:h + 1])
        vv = f64(t["v"][b * T:(b + 1) * T, h:h + 1])
        S_ref, Z_ref = ob.prefill(kk, vv, f64(t["W"][h:h + 1]))
        assert _state_err(f64(S[b, h:h + 1]), f64(Z[b, h:h + 1]), S_ref, Z_ref) <= TOL_STATE
        # invariant that holds at any size: sum_i Z_i = 2T
        assert abs(float(Z[b, h].double().sum()) - 2 * T) <= 1e-4 * 2 * T


def test_commit_equals_prefill_of_same_tokens(cuda_device):
    """Order-free sums: committing 4 blocks one by one and ingesting the same
    128 tokens as one prompt give the same state (up to fp32 rounding)."""
    w = inputs.single_layer(n_blocks=4)
    cfg = config(w)
    S, Z = new_pool(cfg, 2, cuda_device)
    W = w.tensors["W"].to(cuda_device)
    for blk in range(4):
        hb.hb_commit_block(cfg, slots([0], cuda_device), w.tensors["commit_k"][blk].to(cuda_device),
                           w.tensors["commit_v"][blk].to(cuda_device), W, S, Z)
    k = w.tensors["commit_k"][:, 0].reshape(128, w.H, w.d).to(cuda_device)
    v = w.tensors["commit_v"][:, 0].reshape(128, w.H, w.d).to(cuda_device)
    cu = torch.tensor([0, 128], dtype=torch.int64, device=cuda_device)
    hb.hb_prefill_state(cfg, slots([1], cuda_device), k, v, cu, 128, W, S, Z)
    assert_status_ok()
    assert unit_err(f64(S[0]), f64(S[1]), 1) <= 1e-5
    assert unit_err(f64(Z[0]), f64(Z[1]), 1) <= 1e-5


def test_state_zero(cuda_device):
    cfg = hb.Config(16, 128, 64, 32)
    S, Z = new_pool(cfg, 4, cuda_device)
    S.fill_(3.0)
    Z.fill_(2.0)
    hb.hb_state_zero(cfg, slots([3, 1], cuda_device), S, Z)
    assert_status_ok()
    assert float(S[1].abs().max()) == 0 and float(S[3].abs().max()) == 0
    assert float(Z[1].abs().max()) == 0 and float(Z[3].abs().max()) == 0
    assert float(S[0].min()) == 3.0 and float(Z[2].min()) == 2.0


def test_state_deterministic(cuda_device):
    w = inputs.prompt_ingestion(device=cuda_device, B=2, T=1000)
    cfg = config(w)
    t = w.tensors
    outs = []
    for _ in range(2):
        S, Z = new_pool(cfg, 2, cuda_device)
        hb.hb_prefill_state(cfg, slots([0, 1], cuda_device), t["k"], t["v"], t["cu_seqlens"], 1000,
                            t["W"], S, Z)
        outs.append((S, Z))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("H,d,f", [(4, 128, 64), (2, 64, 16)])
def test_state_copy_between_slots(cuda_device, H, d, f):
    """hb_state_copy moves S and Z of each source slot to its destination bit
    for bit and leaves every other slot alone; a pair with a slot outside the
    pool is skipped and flagged while the other pairs are copied."""
    cfg = hb.Config(H, d, f, 32)
    S, Z = new_pool(cfg, 6, cuda_device)
    S.copy_(inputs.draw(90, tuple(S.shape), torch.float32, device=cuda_device))
    Z.copy_(inputs.draw(91, tuple(Z.shape), torch.float32, device=cuda_device))
    S0, Z0 = S.clone(), Z.clone()
    hb.hb_state_copy(cfg, slots([0, 3, 2], cuda_device), slots([4, 1, 2], cuda_device), S, Z)
    assert_status_ok()
    S_exp, Z_exp = S0.clone(), Z0.clone()
    S_exp[4], Z_exp[4] = S0[0], Z0[0]
    S_exp[1], Z_exp[1] = S0[3], Z0[3]
    assert torch.equal(S, S_exp) and torch.equal(Z, Z_exp)
    S1, Z1 = S.clone(), Z.clone()
    hb.hb_state_copy(cfg, slots([5, 9], cuda_device), slots([0, 3], cuda_device), S, Z)
    assert hb.hb_get_device_status() == 5  # HB_ERR_DEVICE_BOUNDS
    S1[0], Z1[0] = S1[5].clone(), Z1[5].clone()
    assert torch.equal(S, S1) and torch.equal(Z, Z1)

"""hb_prefill_attend (GPU): every block of a prompt gets the oracle's
block-hybrid output against the state of the blocks before it, and the slot
ends with the whole prompt's state; also within the bounds of chaining
hb_block_attend_commit block by block."""

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


def _prompts(seed, B, T, H, d, f, dt):
    W = inputs.draw(seed, (H, d, f), dt, std=d ** -0.5)
    gate = inputs.draw(seed + 1, (H,), torch.float32)
    q, k, v = (inputs.draw(seed + 2 + i, (B, T, H, d), dt) for i in range(3))
    return W, gate, q, k, v


def _check_against_oracle(dev, cfg, B, T, W, gate, q, k, v, slot_of, S, Z, merge, tol,
                          S0=None, Z0=None):
    o = hb.hb_prefill_attend(cfg, slots(slot_of, dev), q.to(dev), k.to(dev), v.to(dev), S, Z,
                             W.to(dev), gate.to(dev), accumulate=S0 is not None)
    assert_status_ok()
    for b, sl in enumerate(slot_of):
        ref_o, ref_S, ref_Z = ob.prefill_attend(
            f64(q[b]), f64(k[b]), f64(v[b]), f64(W), f64(gate), cfg.block_len, merge,
            S0=None if S0 is None else S0[b], Z0=None if Z0 is None else Z0[b])
        for j0 in range(0, T, cfg.block_len):
            blk = slice(j0, j0 + cfg.block_len)
            assert out_err(f64(o[b, blk]), ref_o[blk]) <= tol, (b, j0)
        assert unit_err(f64(S[sl]), ref_S, 1) <= TOL_STATE, b
        assert unit_err(f64(Z[sl]), ref_Z, 1) <= TOL_STATE, b


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_prefill_attend_matches_oracle(cuda_device, merge, dt):
    B, T, H, d, f, L = 3, 128, 16, 128, 64, 32
    cfg = hb.Config(H, d, f, L, dtype=hb.DTYPE_BF16 if dt == torch.bfloat16 else hb.DTYPE_FP32,
                    merge=MERGES[merge])
    W, gate, q, k, v = _prompts(200, B, T, H, d, f, dt)
    S, Z = new_pool(cfg, 5, cuda_device)
    S.fill_(3.0)  # overwritten: accumulate = 0 starts from an empty state
    Z.fill_(3.0)
    _check_against_oracle(cuda_device, cfg, B, T, W, gate, q, k, v, [4, 0, 2], S, Z,
                          MERGES[merge], TOL_OUT_BF16 if dt == torch.bfloat16 else TOL_OUT_FP32)
    assert float(S[1].sub(3.0).abs().max()) == 0.0 and float(S[3].sub(3.0).abs().max()) == 0.0


def test_prefill_attend_continues_a_context(cuda_device):
    """accumulate = 1: the prompt follows context already in the slots."""
    B, T, H, d, f, L = 2, 96, 16, 128, 64, 32
    cfg = hb.Config(H, d, f, L)
    W, gate, q, k, v = _prompts(300, B, T, H, d, f, torch.bfloat16)
    S, Z = new_pool(cfg, 2, cuda_device)
    S0, Z0 = [], []
    for b in range(B):
        pk = inputs.draw(310 + 2 * b, (64, H, d), torch.bfloat16)
        pv = inputs.draw(311 + 2 * b, (64, H, d), torch.bfloat16)
        s0, z0 = ob.prefill(f64(pk), f64(pv), f64(W))
        S0.append(s0)
        Z0.append(z0)
        S[b] = torch.as_tensor(s0, dtype=torch.float32, device=cuda_device)
        Z[b] = torch.as_tensor(z0, dtype=torch.float32, device=cuda_device)
    _check_against_oracle(cuda_device, cfg, B, T, W, gate, q, k, v, [0, 1], S, Z,
                          hb.MERGE_SHARED_NORM, TOL_OUT_BF16, S0=S0, Z0=Z0)


def test_prefill_attend_tiny_shape(cuda_device):
    """A shape outside the tensor-core kernels (H=2, d=16, f=8, L=4) in the
    fp32 mode: the generic kernels, block by block."""
    B, T, H, d, f, L = 2, 12, 2, 16, 8, 4
    cfg = hb.Config(H, d, f, L, dtype=hb.DTYPE_FP32)
    W, gate, q, k, v = _prompts(400, B, T, H, d, f, torch.float32)
    S, Z = new_pool(cfg, 2, cuda_device)
    _check_against_oracle(cuda_device, cfg, B, T, W, gate, q, k, v, [1, 0], S, Z,
                          hb.MERGE_SHARED_NORM, TOL_OUT_FP32)


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("T", [32, 160, 416, 512])
def test_prefill_attend_segments_match_oracle(cuda_device, merge, T):
    """Prompts of 1 to 16 blocks, so that the 128-token segments of the
    tensor-core kernel come full and partial (32, 160 = 128 + 32,
    416 = 3 x 128 + 32, 512 = 4 x 128 tokens), 4 prompts each with permuted
    slots holding earlier context: every block's output and the final state
    against the oracle."""
    B, H, d, f, L = 4, 16, 128, 64, 32
    cfg = hb.Config(H, d, f, L, merge=MERGES[merge])
    W, gate, q, k, v = _prompts(700 + T, B, T, H, d, f, torch.bfloat16)
    S, Z = new_pool(cfg, 6, cuda_device)
    S0, Z0 = [], []
    slot_of = [5, 1, 3, 0]
    for b in range(B):
        n = 24 * b  # 0, 24, 48, 72 tokens of earlier context
        pk = inputs.draw(800 + 2 * b, (n, H, d), torch.bfloat16)
        pv = inputs.draw(801 + 2 * b, (n, H, d), torch.bfloat16)
        s0, z0 = ob.prefill(f64(pk), f64(pv), f64(W))
        S0.append(s0)
        Z0.append(z0)
        S[slot_of[b]] = torch.as_tensor(s0, dtype=torch.float32, device=cuda_device)
        Z[slot_of[b]] = torch.as_tensor(z0, dtype=torch.float32, device=cuda_device)
    _check_against_oracle(cuda_device, cfg, B, T, W, gate, q, k, v, slot_of, S, Z,
                          MERGES[merge], TOL_OUT_BF16, S0=S0, Z0=Z0)


def test_prefill_attend_close_to_chained_steps(cuda_device):
    """8 prompts of 512 tokens: within the bf16 bound of hb_block_attend_commit
    run block by block (every request committing), and the same state within
    the state bound."""
    B, T, H, d, f, L = 8, 512, 16, 128, 64, 32
    cfg = hb.Config(H, d, f, L)
    W, gate, q, k, v = (x.to(cuda_device) for x in _prompts(500, B, T, H, d, f, torch.bfloat16))
    sl = torch.arange(B, dtype=torch.int32, device=cuda_device)
    S1, Z1 = new_pool(cfg, B, cuda_device)
    S2, Z2 = new_pool(cfg, B, cuda_device)
    o1 = hb.hb_prefill_attend(cfg, sl, q, k, v, S1, Z1, W, gate)
    ones = torch.ones(B, dtype=torch.int32, device=cuda_device)
    o2 = torch.empty_like(o1)
    for j0 in range(0, T, L):
        blk = slice(j0, j0 + L)
        o2[:, blk] = hb.hb_block_attend_commit(cfg, sl, q[:, blk].contiguous(),
                                               k[:, blk].contiguous(), v[:, blk].contiguous(),
                                               S2, Z2, W, gate, ones)
    assert_status_ok()
    for b in range(B):
        for j0 in range(0, T, L):
            assert out_err(f64(o1[b, j0:j0 + L]), f64(o2[b, j0:j0 + L])) <= TOL_OUT_BF16, (b, j0)
    assert unit_err(f64(S1), f64(S2), 2) <= TOL_STATE
    assert unit_err(f64(Z1), f64(Z2), 2) <= TOL_STATE


def test_prefill_attend_bad_slot_is_flagged(cuda_device):
    B, T, H, d, f, L = 2, 64, 16, 128, 64, 32
    cfg = hb.Config(H, d, f, L)
    W, gate, q, k, v = (x.to(cuda_device) for x in _prompts(600, B, T, H, d, f, torch.bfloat16))
    S, Z = new_pool(cfg, 2, cuda_device)
    o = torch.full_like(q, 5.0)
    hb.hb_prefill_attend(cfg, slots([1, 9], cuda_device), q, k, v, S, Z, W, gate, o=o)
    assert hb.hb_get_device_status() == 5  # HB_ERR_DEVICE_BOUNDS
    assert bool((o[1] == 5.0).all())      # nothing written for the bad request
    assert float(S[0].abs().max()) == 0.0  # untouched slot
    ref_o, _, _ = ob.prefill_attend(f64(q[0].cpu()), f64(k[0].cpu()), f64(v[0].cpu()),
                                    f64(W.cpu()), f64(gate.cpu()), L)
    assert out_err(f64(o[0]), ref_o) <= TOL_OUT_BF16

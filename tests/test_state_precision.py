"""Why the master state stays fp32 (CPU): the state after many commits, kept
in fp32 and rounded once per commit, stays within the 1e-4 bound the library
holds S to, while a bf16 master (rounded after every commit, as a bf16 pool
would store it) leaves it after a handful of commits. Both are measured
against the oracle's fp64 sums over the same seeded blocks."""

import numpy as np
import torch

import oracle.block_hybrid as ob
from tests.parity import TOL_STATE, unit_err


def _blocks(n_blocks, H=2, d=128, f=64, L=32, seed=3):
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn((H, d, f), generator=g) * d ** -0.5).to(torch.bfloat16)
    ks = [torch.randn((L, H, d), generator=g).to(torch.bfloat16) for _ in range(n_blocks)]
    vs = [torch.randn((L, H, d), generator=g).to(torch.bfloat16) for _ in range(n_blocks)]
    return W, ks, vs


def _drift(n_blocks, dtype):
    W, ks, vs = _blocks(n_blocks)
    W64 = W.to(torch.float64).numpy()
    H, d, f = W.shape
    S_exact = np.zeros((H, 2 * f, d))
    Z_exact = np.zeros((H, 2 * f))
    S_m = torch.zeros((H, 2 * f, d), dtype=dtype)
    errs = []
    for k, v in zip(ks, vs):
        k64, v64 = k.to(torch.float64).numpy(), v.to(torch.float64).numpy()
        S_next, Z_exact = ob.commit(S_exact, Z_exact, k64, v64, W64)
        dS = S_next - S_exact
        S_exact = S_next
        # the master adds the block's (exact) contribution and is stored back
        # in its own precision, once per commit
        S_m = (S_m.to(torch.float64) + torch.from_numpy(dS)).to(dtype)
        errs.append(unit_err(S_m.to(torch.float64).numpy(), S_exact, 1))
    return errs


def test_fp32_master_stays_within_the_state_bound():
    errs = _drift(64, torch.float32)
    assert max(errs) < TOL_STATE / 10


def test_bf16_master_leaves_the_state_bound():
    errs = _drift(16, torch.bfloat16)
    assert errs[0] > TOL_STATE        # one rounding already exceeds it
    assert max(errs) > 10 * TOL_STATE  # and it does not come back

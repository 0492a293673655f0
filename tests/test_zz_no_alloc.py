"""hb_prefill_state_noalloc against hb_prefill_state (GPU).

The no-allocation entry point serves callers that cannot call cudaMalloc (a
plug-in whose host engine owns all device memory, a serving loop that must
not risk an allocation's device synchronisation). It keeps the split partial
sums in the library's fixed device array instead of a caller workspace. Here
two calls in a row, with different prompts and batch sizes (the second one
accumulating), must leave the same S and Z as the same two calls through the
workspace entry point, within the state tolerance of the other tests.

This file is named so that pytest collects it last.
"""

import numpy as np
import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
from linear_attention_diffusion_feature_b300 import inputs
from tests.parity import TOL_STATE, assert_status_ok, f64, new_pool, slots, unit_err

pytestmark = pytest.mark.gpu

H, D, FH = 16, 128, 64


def _prompts(seed, lens, device):
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    total = int(cu[-1])
    k = inputs.draw(seed, (total, H, D), torch.bfloat16).to(device)
    v = inputs.draw(seed + 1, (total, H, D), torch.bfloat16).to(device)
    return k, v, cu.to(device), max(lens)


def test_noalloc_prefill_matches_workspace_prefill(cuda_device):
    cfg = hb.Config(H, D, FH, 32)
    W = inputs.draw(40, (H, D, FH), torch.bfloat16, std=D ** -0.5).to(cuda_device)
    calls = [  # (slots, prompt lengths, accumulate)
        ([3, 0], [700, 1500], False),
        ([0, 5, 3], [300, 2000, 64], True),
    ]
    S_a, Z_a = new_pool(cfg, 6, cuda_device)
    S_b, Z_b = new_pool(cfg, 6, cuda_device)
    for i, (idx, lens, acc) in enumerate(calls):
        assert hb.hb_prefill_workspace_size(cfg, len(idx), max(lens)) > 0  # scratch in use
        k, v, cu, mx = _prompts(50 + 10 * i, lens, cuda_device)
        sl = slots(idx, cuda_device)
        hb.hb_prefill_state_noalloc(cfg, sl, k, v, cu, mx, W, S_a, Z_a, accumulate=acc)
        hb.hb_prefill_state(cfg, sl, k, v, cu, mx, W, S_b, Z_b, accumulate=acc)
        assert_status_ok()
        for s in sorted(set(idx)):
            assert unit_err(f64(S_a[s]), f64(S_b[s]), 1) <= TOL_STATE
            assert unit_err(f64(Z_a[s]), f64(Z_b[s]), 1) <= TOL_STATE
    for s in (1, 2, 4):  # slots no call named stay untouched
        assert float(S_a[s].abs().max()) == 0.0 and float(Z_a[s].abs().max()) == 0.0

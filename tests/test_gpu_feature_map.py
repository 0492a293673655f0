"""hb_feature_map against the oracle's phi (GPU)."""

import numpy as np
import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from linear_attention_diffusion_feature_b300 import inputs
from tests.parity import TOL_PHI, f64, unit_err

pytestmark = pytest.mark.gpu

DTYPES = {"bf16": (torch.bfloat16, hb.DTYPE_BF16), "fp32": (torch.float32, hb.DTYPE_FP32)}


@pytest.mark.parametrize("dt", sorted(DTYPES))
@pytest.mark.parametrize("d,f", [(16, 8), (48, 24), (128, 64)])
@pytest.mark.parametrize("n", [1, 17, 1000])
def test_feature_map_matches_oracle(cuda_device, dt, d, f, n):
    tdt, code = DTYPES[dt]
    H = 3
    x = inputs.draw(10 + n, (n, H, d), tdt)
    W = inputs.draw(20 + d, (H, d, f), tdt, std=d ** -0.5)
    cfg = hb.Config(H, d, f, 32, dtype=code)
    phi = hb.hb_feature_map(cfg, x.to(cuda_device), W.to(cuda_device))
    ref = ob.feature_map_heads(f64(x), f64(W))
    assert unit_err(f64(phi), ref, 2) <= TOL_PHI
    halves = f64(phi).reshape(n, H, 2, f).sum(-1)
    np.testing.assert_allclose(halves, 1.0, atol=1e-5)


def test_feature_map_empty(cuda_device):
    cfg = hb.Config(2, 16, 8, 4, dtype=hb.DTYPE_FP32)
    x = torch.empty((0, 2, 16), device=cuda_device)
    W = inputs.draw(1, (2, 16, 8), torch.float32).to(cuda_device)
    phi = hb.hb_feature_map(cfg, x, W)
    assert phi.shape == (0, 2, 16)


def test_feature_map_prompt_sized(cuda_device):
    """All keys of the prompt-ingestion workload (8 x 8192 tokens, 16 heads);
    the oracle checks a sample of rows."""
    w = inputs.prompt_ingestion(device=cuda_device)
    cfg = hb.Config(w.H, w.d, w.f, w.L)
    k = w.tensors["k"]
    phi = hb.hb_feature_map(cfg, k, w.tensors["W"])
    rows = torch.tensor([0, 1, 4095, 8191, 8192, 33333, 65534, 65535])
    ref = ob.feature_map_heads(f64(k[rows.to(cuda_device)]), f64(w.tensors["W"]))
    assert unit_err(f64(phi[rows.to(cuda_device)]), ref, 2) <= TOL_PHI

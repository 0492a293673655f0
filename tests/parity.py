"""Helpers shared by the GPU parity tests: device set-up of workloads through
the C ABI, conversions to float64 for the oracle, and the error metric.

Error metric (the reading of "max relative error"): per (request, head) unit,
max |gpu - oracle| / max |oracle| over that unit's elements; the test bound
applies to the worst unit. Elementwise relative error is ill-posed where the
oracle value is near zero.
"""

from __future__ import annotations

import numpy as np
import torch

import linear_attention_diffusion_feature_b300 as hb

TOL_OUT_BF16 = 1e-2   # bf16 outputs
TOL_OUT_FP32 = 1e-4   # fp32-everything mode
TOL_STATE = 1e-4      # S and Z, both modes
TOL_PHI = 1e-5        # feature map (fp32 output from exact inputs)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def unit_err(gpu: np.ndarray, ref: np.ndarray, unit_axes: int) -> float:
    """Worst unit of max|gpu-ref|/max|ref|; the first ``unit_axes`` axes
    index units, the rest are the unit's elements."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    n = int(np.prod(gpu.shape[:unit_axes])) if unit_axes else 1
    g = gpu.reshape(n, -1)
    r = ref.reshape(n, -1)
    if g.shape[1] == 0:
        return 0.0
    assert np.isfinite(g).all(), "non-finite GPU output"
    num = np.abs(g - r).max(axis=1)
    den = np.maximum(np.abs(r).max(axis=1), 1e-30)
    return float((num / den).max())


def out_err(o_gpu: np.ndarray, o_ref: np.ndarray) -> float:
    """Outputs [L, H, d] of one request (units = heads)."""
    return unit_err(np.transpose(o_gpu, (1, 0, 2)), np.transpose(o_ref, (1, 0, 2)), 1)


def config(w, merge=hb.MERGE_SHARED_NORM) -> hb.Config:
    dt = hb.DTYPE_BF16 if w.dtype == torch.bfloat16 else hb.DTYPE_FP32
    return hb.Config(w.H, w.d, w.f, w.L, dtype=dt, merge=merge)


def new_pool(cfg: hb.Config, slots: int, device) -> tuple:
    S = torch.zeros((slots, cfg.num_heads, cfg.F, cfg.head_dim), dtype=torch.float32,
                    device=device)
    Z = torch.zeros((slots, cfg.num_heads, cfg.F), dtype=torch.float32, device=device)
    return S, Z


def slots(idx, device) -> torch.Tensor:
    return torch.as_tensor(idx, dtype=torch.int32, device=device)


def assert_status_ok():
    st = hb.hb_get_device_status()
    assert st == 0, hb.hb_status_string(st)

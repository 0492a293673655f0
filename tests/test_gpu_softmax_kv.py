"""hb_softmax_kv_attend (comparison path) against the oracle (GPU)."""

import numpy as np
import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from linear_attention_diffusion_feature_b300 import inputs
from tests.parity import TOL_OUT_BF16, TOL_OUT_FP32, assert_status_ok, config, f64, out_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_softmax_kv_ragged(cuda_device, dt):
    H, d, f, L = 4, 128, 64, 32
    lens = [0, 5, 64, 300, 2048]
    B = len(lens)
    cfg = hb.Config(H, d, f, L, dtype=hb.DTYPE_BF16 if dt == torch.bfloat16 else hb.DTYPE_FP32)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    total = int(cu[-1])
    kc = inputs.draw(31, (total, H, d), dt)
    vc = inputs.draw(32, (total, H, d), dt)
    q, k, v = (inputs.draw(33 + i, (B, L, H, d), dt) for i in range(3))
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    o = hb.hb_softmax_kv_attend(cfg, dev(kc), dev(vc), dev(cu), max(lens), dev(q), dev(k), dev(v))
    assert_status_ok()
    tol = TOL_OUT_BF16 if dt == torch.bfloat16 else TOL_OUT_FP32
    for b in range(B):
        a, e = int(cu[b]), int(cu[b + 1])
        ref = ob.softmax_kv_attend(f64(kc[a:e]), f64(vc[a:e]), f64(q[b]), f64(k[b]), f64(v[b]))
        assert out_err(f64(o[b]), ref) <= tol, b


@pytest.mark.parametrize("B", [1, 16, 32])
def test_softmax_kv_stack_layer(cuda_device, B):
    w = inputs.stack_layer(1, B, device=cuda_device)
    cfg = config(w)
    t = w.tensors
    o = hb.hb_softmax_kv_attend(cfg, t["prefix_k"], t["prefix_v"], t["cu_prefix"], w.meta["P"],
                                t["q"], t["k"], t["v"])
    assert_status_ok()
    P = w.meta["P"]
    for b in sorted({0, B - 1}):
        ref = ob.softmax_kv_attend(f64(t["prefix_k"][b * P:(b + 1) * P]),
                                   f64(t["prefix_v"][b * P:(b + 1) * P]), f64(t["q"][b]),
                                   f64(t["k"][b]), f64(t["v"][b]))
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16

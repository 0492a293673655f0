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


@pytest.mark.parametrize("B", [1, 16, 32, 256])
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


BOUNDS = 5


def _paged_problem(cuda_device, dt, lens, pt, H=4, seed=41):
    d, L = 128, 32
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    kc = inputs.draw(seed, (int(cu[-1]), H, d), dt)
    vc = inputs.draw(seed + 1, (int(cu[-1]), H, d), dt)
    q, k, v = (inputs.draw(seed + 2 + i, (len(lens), L, H, d), dt) for i in range(3))
    kp, vp, table, plen = inputs.paged_cache(seed + 5, kc, vc, lens, pt)
    return cu, kc, vc, q, k, v, kp, vp, table, plen


@pytest.mark.parametrize("dt,pt", [(torch.bfloat16, 32), (torch.bfloat16, 64),
                                   (torch.bfloat16, 256), (torch.bfloat16, 16),
                                   (torch.float32, 32)])
def test_softmax_kv_paged_ragged(cuda_device, dt, pt):
    """Ragged prefixes (empty, inside one page, on page and tile edges, many
    tiles) in pages scattered over a pool whose unused pages and slots hold
    NaN. With pages of a multiple of 32 tokens in bf16 the TMA kernel runs the
    packed kernel's tiles in the packed kernel's order, so the two outputs
    agree bit for bit."""
    H, d, f, L = 4, 128, 64, 32
    lens = [0, 5, 32, 64, 100, 300, 2048]
    cfg = hb.Config(H, d, f, L, dtype=hb.DTYPE_BF16 if dt == torch.bfloat16 else hb.DTYPE_FP32)
    cu, kc, vc, q, k, v, kp, vp, table, plen = _paged_problem(cuda_device, dt, lens, pt, H)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    o = hb.hb_softmax_kv_attend_paged(cfg, dev(kp), dev(vp), dev(table), dev(plen), max(lens),
                                      dev(q), dev(k), dev(v))
    assert_status_ok()
    tol = TOL_OUT_BF16 if dt == torch.bfloat16 else TOL_OUT_FP32
    kp64, vp64 = f64(kp), f64(vp)
    for b, P in enumerate(lens):
        ref = ob.softmax_kv_attend_paged(kp64, vp64, table[b].numpy(), P, f64(q[b]), f64(k[b]),
                                         f64(v[b]))
        assert out_err(f64(o[b]), ref) <= tol, b
    if dt == torch.bfloat16 and pt % 32 == 0:
        o_packed = hb.hb_softmax_kv_attend(cfg, dev(kc), dev(vc), dev(cu), max(lens), dev(q),
                                           dev(k), dev(v))
        assert_status_ok()
        assert torch.equal(o.cpu(), o_packed.cpu())


def test_softmax_kv_paged_stack_layer(cuda_device):
    """The comparison layer of the six-layer stack (64 requests, 2,048 cached
    tokens each) read from a shuffled page pool: bit-identical to the packed
    cache, and equal to the oracle on the first and last request."""
    B = 64
    w = inputs.stack_layer(1, B, device=cuda_device)
    cfg = config(w)
    t = w.tensors
    P = w.meta["P"]
    kp, vp, table, plen = inputs.paged_cache(9, t["prefix_k"], t["prefix_v"], [P] * B, 32)
    o = hb.hb_softmax_kv_attend_paged(cfg, kp, vp, table, plen, P, t["q"], t["k"], t["v"])
    assert_status_ok()
    o_packed = hb.hb_softmax_kv_attend(cfg, t["prefix_k"], t["prefix_v"], t["cu_prefix"], P,
                                       t["q"], t["k"], t["v"])
    assert_status_ok()
    assert torch.equal(o, o_packed)
    for b in (0, B - 1):
        ref = ob.softmax_kv_attend(f64(t["prefix_k"][b * P:(b + 1) * P]),
                                   f64(t["prefix_v"][b * P:(b + 1) * P]), f64(t["q"][b]),
                                   f64(t["k"][b]), f64(t["v"][b]))
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16


@pytest.mark.parametrize("pt", [32, 16])
def test_softmax_kv_paged_bad_page_flagged(cuda_device, pt):
    """A page id outside the pool is caught before any load: that request
    gets no output and the status word says so; the others are correct."""
    H = 2
    lens = [40, 64, 33]
    cfg = hb.Config(H, 128, 64, 32)
    cu, kc, vc, q, k, v, kp, vp, table, plen = _paged_problem(cuda_device, torch.bfloat16, lens,
                                                              pt, H, seed=51)
    table[1, 1] = kp.shape[0]  # one past the last page of the pool
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    o = torch.full_like(dev(q), 7.0)
    hb.hb_softmax_kv_attend_paged(cfg, dev(kp), dev(vp), dev(table), dev(plen), max(lens),
                                  dev(q), dev(k), dev(v), o=o)
    assert hb.hb_get_device_status() == BOUNDS
    assert hb.hb_get_device_status() == 0
    assert bool((o[1] == 7.0).all())
    for b in (0, 2):
        ref = ob.softmax_kv_attend_paged(f64(kp), f64(vp), table[b].numpy(), lens[b], f64(q[b]),
                                         f64(k[b]), f64(v[b]))
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16

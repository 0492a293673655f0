"""Pins of the oracle's fp8 (e4m3) state copy (CPU): its value table and
rounding against torch's own float8_e4m3fn conversion (an independent
library routine), round trips over every finite code, the quantiser's scale
and error bound, and what the copy costs the attend's output against the
exact state on the pages' shapes."""

import numpy as np
import pytest
import torch

import oracle.block_hybrid as ob
from oracle import state_fp8 as of8
from tests.parity import out_err

FINITE = [c for c in range(256) if c not in (0x7F, 0xFF)]


def test_value_table_matches_torch():
    codes = np.array(FINITE, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    np.testing.assert_array_equal(of8.e4m3_value(codes), ref)
    assert np.isnan(of8.e4m3_value(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    assert of8.e4m3_value(np.array([0x7E], dtype=np.uint8))[0] == 448.0
    assert of8.e4m3_value(np.array([0x01], dtype=np.uint8))[0] == 2.0 ** -9


def test_every_finite_code_round_trips():
    codes = np.array(FINITE, dtype=np.uint8)
    vals = of8.e4m3_value(codes)
    np.testing.assert_array_equal(of8.e4m3_round(vals), vals)
    np.testing.assert_array_equal(of8.e4m3_encode(vals), codes)


def test_rounding_matches_torch_including_ties():
    g = torch.Generator().manual_seed(8)
    parts = [torch.randn(20000, generator=g) * s for s in (1e-3, 1e-2, 0.1, 1.0, 10.0, 100.0)]
    # every midpoint between neighbouring values: ties go to the even code
    vals = np.sort(np.unique(of8.e4m3_value(np.array(FINITE, dtype=np.uint8))))
    mids = (vals[1:] + vals[:-1]) / 2
    parts.append(torch.from_numpy(mids[np.abs(mids) <= 448]).float())
    x = torch.cat(parts).float()
    x = x[x.abs() <= 448]
    ref = x.to(torch.float8_e4m3fn).float().double().numpy()
    got = of8.e4m3_round(x.numpy())
    np.testing.assert_array_equal(got, ref)


def test_saturation_and_signed_zero():
    r = of8.e4m3_round(np.array([449.0, 463.9, 470.0, 1e6, -1e6, -0.0], dtype=np.float32))
    np.testing.assert_array_equal(r[:5], [448.0, 448.0, 448.0, 448.0, -448.0])
    assert of8.e4m3_encode(r[5:])[0] == 0x80


def _state(P, H=3, d=128, f=64, seed=0):
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn((H, d, f), generator=g) * d ** -0.5).to(torch.bfloat16).double().numpy()
    k = torch.randn((P, H, d), generator=g).to(torch.bfloat16).double().numpy()
    v = torch.randn((P, H, d), generator=g).to(torch.bfloat16).double().numpy()
    return ob.prefill(k, v, W), W


@pytest.mark.parametrize("P", [1, 40, 2048])
def test_quantiser_scale_and_error_bound(P):
    (S, _), _ = _state(P, seed=P)
    S32 = S.astype(np.float32)
    codes, scales = of8.quantize_state_fp8(S32)
    for h in range(S.shape[0]):
        amax = np.float32(np.abs(S32[h]).max())
        assert scales[h] == np.float32(amax / np.float32(448.0))
        # the largest magnitude lands on +-448
        assert np.abs(of8.e4m3_value(codes[h])).max() == 448.0
    Sq = of8.dequantize_state_fp8(codes, scales)
    # half a quantum: 2^-4 relative for normal codes, 2^-10 of the scale
    # below 2^-6, plus the fp32 rounding of the quotient
    bound = np.maximum(np.abs(S32) * 2.0 ** -4, scales[:, None, None] * 2.0 ** -10) * (1 + 1e-6)
    assert (np.abs(Sq - S32) <= bound).all()


def test_zero_state_has_zero_scale_and_codes():
    codes, scales = of8.quantize_state_fp8(np.zeros((2, 128, 128), dtype=np.float32))
    assert not codes.any() and not scales.any()
    assert not of8.dequantize_state_fp8(codes, scales).any()


@pytest.mark.parametrize("merge,bound", [(ob.MERGE_SHARED_NORM, 1e-2), (ob.MERGE_CONVEX, 2e-2)])
def test_what_the_fp8_copy_costs_the_attend(merge, bound):
    """The copy is lossy: each code carries 3 mantissa bits (half a step is
    2^-4 of the value), and where phi(q) puts its weight on a few rows of S
    the output inherits that. Measured against the exact state over prefixes
    of 32 to 8,192 tokens (4 seeds each): the shared-normaliser merge (the
    pages' form) stays inside the 1e-2 bound of the bf16 outputs (worst about
    6e-3); the convex merge, whose linear branch is a ratio of two sums, goes
    above it for short prefixes (worst about 1.3e-2). A bf16 copy costs
    about 20x less (worst about 1e-3)."""
    g = torch.Generator().manual_seed(11)
    worst8 = worst16 = 0.0
    for P in (32, 256, 2048, 8192):
        for rep in range(4):
            (S, Z), W = _state(P, H=2, seed=100 + P + rep)
            q, k, v = (torch.randn((32, 2, 128), generator=g).to(torch.bfloat16).double().numpy()
                       for _ in range(3))
            gate = torch.randn((2,), generator=g).double().numpy()
            ref = ob.attend(q, k, v, S, Z, W, gate, merge)
            codes, scales = of8.quantize_state_fp8(S.astype(np.float32))
            o8 = ob.attend(q, k, v, of8.dequantize_state_fp8(codes, scales), Z, W, gate, merge)
            S16 = torch.from_numpy(S).float().to(torch.bfloat16).double().numpy()
            o16 = ob.attend(q, k, v, S16, Z, W, gate, merge)
            worst8 = max(worst8, out_err(o8, ref))
            worst16 = max(worst16, out_err(o16, ref))
    assert worst8 < bound
    assert worst16 < 2e-3 and worst8 > 4 * worst16

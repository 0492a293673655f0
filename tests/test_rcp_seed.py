"""The integer seed of the kernels' Newton-Raphson reciprocal (CPU): the
constant in the PTX helper header bounds the seed's relative error by 0.0506
over a whole octave of mantissas, the minimax value for this form of seed,
so three Newton steps reach fp32 rounding."""

import os
import re

import numpy as np

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "linear_attention_diffusion_feature_b300", "csrc", "hb_ptx.cuh")


def _seed_constant() -> int:
    text = open(HEADER).read()
    body = text[text.index("rcp2_newton"):]
    return int(re.search(r"0x([0-9A-Fa-f]{8})u", body).group(1), 16)


def _seed_error(R: int) -> float:
    m = np.arange(0, 1 << 23, dtype=np.uint32)
    xb = (np.uint32(127) << np.uint32(23)) | m  # every x in [1, 2)
    x = xb.view(np.float32).astype(np.float64)
    y = (np.uint32(R) - xb).view(np.float32).astype(np.float64)
    return float(np.abs(x * y - 1.0).max())


def test_seed_bound():
    assert _seed_error(_seed_constant()) < 0.0506


def test_seed_is_minimax_among_neighbours():
    R = _seed_constant()
    e = _seed_error(R)
    # moving the constant in either direction makes the worst case worse
    # (or ties it within 1e-8)
    for dR in (-4096, -256, -16, 16, 256, 4096):
        assert _seed_error(R + dR) >= e - 1e-8, dR


def test_three_newton_steps_reach_fp32_rounding():
    R = _seed_constant()
    rng = np.random.default_rng(0)
    x = (rng.random(100000) * 1e6 + 1e-6).astype(np.float32)
    y = (np.uint32(R) - x.view(np.uint32)).view(np.float32)
    one = np.float32(1.0)
    for _ in range(3):
        e = np.float32(one - x * y)
        y = np.float32(y + y * e)
    rel = np.abs(x.astype(np.float64) * y.astype(np.float64) - 1.0)
    assert rel.max() < 5e-7

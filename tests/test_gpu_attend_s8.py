"""The fp8 copy of the state (GPU): hb_state_to_fp8's codes and scales
against the oracle's quantiser bit for bit, and hb_block_attend_s8 against
the oracle's attend on the dequantised state for every request, at batches
where every CTA runs many units, for both merges and both block lengths of
the persistent kernel. The states are the oracle's, uploaded as fp32."""

import numpy as np
import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from oracle import state_fp8 as of8
from tests.parity import TOL_OUT_BF16, assert_status_ok, f64, out_err

pytestmark = pytest.mark.gpu

MERGES = {"shared_norm": hb.MERGE_SHARED_NORM, "convex": hb.MERGE_CONVEX}
H, D, FH, F = 16, 128, 64, 128
BOUNDS = 5  # HB_ERR_DEVICE_BOUNDS


def _case(B, L, seed, max_prefix=64, zero_every=7):
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn((H, D, FH), generator=g) * D ** -0.5).to(torch.bfloat16)
    gate = torch.randn((H,), generator=g)
    q, k, v = (torch.randn((B, L, H, D), generator=g).to(torch.bfloat16) for _ in range(3))
    S = np.zeros((B, H, F, D), dtype=np.float32)
    Z = np.zeros((B, H, F), dtype=np.float32)
    for b in range(B):
        n = 0 if b % zero_every == 3 else int(torch.randint(1, max_prefix + 1, (1,), generator=g))
        pk = torch.randn((n, H, D), generator=g).to(torch.bfloat16)
        pv = torch.randn((n, H, D), generator=g).to(torch.bfloat16)
        s0, z0 = ob.prefill(f64(pk), f64(pv), f64(W))
        S[b], Z[b] = s0, z0
    slot_of = torch.randperm(B + 3, generator=g)[:B]
    return dict(W=W, gate=gate, q=q, k=k, v=v, S=S, Z=Z, slot_of=slot_of)


def _pools(c, B, dev):
    S = torch.full((B + 3, H, F, D), 2.0, dtype=torch.float32)
    Z = torch.full((B + 3, H, F), 2.0, dtype=torch.float32)
    for b in range(B):
        S[int(c["slot_of"][b])] = torch.from_numpy(c["S"][b])
        Z[int(c["slot_of"][b])] = torch.from_numpy(c["Z"][b])
    return S.to(dev), Z.to(dev)


def test_fp8_copy_codes_and_scales_match_oracle(cuda_device):
    """Zero states, short and long prefixes; unlisted slots keep their bytes."""
    B = 40
    c = _case(B, 32, seed=801, max_prefix=2048)
    cfg = hb.Config(H, D, FH, 32)
    S, _ = _pools(c, B, cuda_device)
    S8 = torch.full((B + 3, H, F, D), 0x55, dtype=torch.uint8, device=cuda_device)
    sc = torch.full((B + 3, H), -1.0, dtype=torch.float32, device=cuda_device)
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    hb.hb_state_to_fp8(cfg, sl, S, S8, sc)
    assert_status_ok()
    for b in range(B):
        codes, scales = of8.quantize_state_fp8(c["S"][b])
        slot = int(c["slot_of"][b])
        np.testing.assert_array_equal(S8[slot].cpu().numpy(), codes, err_msg=str(b))
        np.testing.assert_array_equal(sc[slot].cpu().numpy(), scales, err_msg=str(b))
    spare = sorted(set(range(B + 3)) - set(int(x) for x in c["slot_of"]))
    for slot in spare:
        assert bool((S8[slot] == 0x55).all()) and bool((sc[slot] == -1.0).all())


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("B,L", [(64, 32), (320, 32), (64, 16)])
def test_attend_s8_matches_oracle(cuda_device, merge, B, L):
    c = _case(B, L, seed=810 + B + L, max_prefix=64 if B > 100 else 1024)
    cfg = hb.Config(H, D, FH, L, merge=MERGES[merge])
    S, Z = _pools(c, B, cuda_device)
    S8 = torch.empty((B + 3, H, F, D), dtype=torch.uint8, device=cuda_device)
    sc = torch.zeros((B + 3, H), dtype=torch.float32, device=cuda_device)
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    hb.hb_state_to_fp8(cfg, sl, S, S8, sc)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    o = hb.hb_block_attend_s8(cfg, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S8, sc, Z,
                              dev(c["W"]), dev(c["gate"]))
    assert_status_ok()
    W64, g64 = f64(c["W"]), f64(c["gate"])
    for b in range(B):
        codes, scales = of8.quantize_state_fp8(c["S"][b])
        Sq = of8.dequantize_state_fp8(codes, scales)
        ref = ob.attend(f64(c["q"][b]), f64(c["k"][b]), f64(c["v"][b]), Sq,
                        c["Z"][b].astype(np.float64), W64, g64, MERGES[merge])
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16, b


def test_fp8_bad_slots_flagged(cuda_device):
    cfg = hb.Config(H, D, FH, 32)
    c = _case(4, 32, seed=830)
    S, Z = _pools(c, 4, cuda_device)
    S8 = torch.zeros((7, H, F, D), dtype=torch.uint8, device=cuda_device)
    sc = torch.zeros((7, H), dtype=torch.float32, device=cuda_device)
    bad = torch.tensor([0, 9, 2, -1], dtype=torch.int32, device=cuda_device)
    hb.hb_state_to_fp8(cfg, bad, S, S8, sc)
    assert hb.hb_get_device_status() == BOUNDS
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    hb.hb_block_attend_s8(cfg, bad, dev(c["q"]), dev(c["k"]), dev(c["v"]), S8, sc, Z,
                          dev(c["W"]), dev(c["gate"]))
    assert hb.hb_get_device_status() == BOUNDS
    assert_status_ok()

"""hb_block_attend_commit_layers (GPU): several independent layers' fused
steps in one launch. Every request's output, and every committing slot's new
S and Z, against the oracle with that request's layer's feature map and gate;
and bit for bit against one hb_block_attend_commit (or hb_block_attend) call
per layer, since each (request, head) unit is computed the same way whichever
CTA runs it."""

import numpy as np
import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from linear_attention_diffusion_feature_b300 import inputs
from tests.parity import (TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, assert_status_ok, f64,
                          new_pool, out_err, unit_err)

pytestmark = pytest.mark.gpu

MERGES = {"shared_norm": hb.MERGE_SHARED_NORM, "convex": hb.MERGE_CONVEX}


def _case(dt, n_layers, B, L, d=128, f=64, H=16, seed=900, max_prefix=96):
    g = torch.Generator().manual_seed(seed)
    W = inputs.draw(seed + 1, (n_layers, H, d, f), dt, std=d ** -0.5)
    gate = inputs.draw(seed + 2, (n_layers, H), torch.float32)
    R = n_layers * B
    q, k, v = (inputs.draw(seed + 3 + i, (R, L, H, d), dt) for i in range(3))
    # every request of every layer gets its own slot, in a shuffled order,
    # with two slots no request names
    slot_of = torch.randperm(R + 2, generator=g)[:R]
    commit = (torch.rand(R, generator=g) < 0.3).to(torch.int32)
    states = []
    for r in range(R):
        n = int(torch.randint(0, max_prefix + 1, (1,), generator=g))
        pk = inputs.draw(seed + 100 + 2 * r, (n, H, d), dt)
        pv = inputs.draw(seed + 101 + 2 * r, (n, H, d), dt)
        states.append(ob.prefill(f64(pk), f64(pv), f64(W[r // B])))
    return dict(W=W, gate=gate, q=q, k=k, v=v, slot_of=slot_of, commit=commit, states=states,
                n_layers=n_layers, B=B, R=R, H=H, d=d, f=f, L=L)


def _pool(c, cfg, dev):
    S, Z = new_pool(cfg, c["R"] + 2, dev)
    fill = inputs.draw(990, S.shape, torch.float32)
    S.copy_(fill.to(dev))
    Z.copy_(fill[..., 0].abs().to(dev))
    for r in range(c["R"]):
        sl = int(c["slot_of"][r])
        S[sl] = torch.as_tensor(c["states"][r][0], dtype=torch.float32, device=dev)
        Z[sl] = torch.as_tensor(c["states"][r][1], dtype=torch.float32, device=dev)
    return S, Z


def _cfg(c, dt, merge):
    return hb.Config(c["H"], c["d"], c["f"], c["L"],
                     dtype=hb.DTYPE_BF16 if dt == torch.bfloat16 else hb.DTYPE_FP32,
                     merge=MERGES[merge])


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("L", [32, 16])
def test_layers_match_oracle(cuda_device, merge, L):
    c = _case(torch.bfloat16, n_layers=6, B=12, L=L)
    cfg = _cfg(c, torch.bfloat16, merge)
    S, Z = _pool(c, cfg, cuda_device)
    S0, Z0 = S.clone(), Z.clone()
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    o = hb.hb_block_attend_commit_layers(cfg, dev(c["slot_of"].to(torch.int32)), dev(c["q"]),
                                         dev(c["k"]), dev(c["v"]), S, Z, dev(c["W"]),
                                         dev(c["gate"]), dev(c["commit"]))
    assert_status_ok()
    for r in range(c["R"]):
        lyr, sl = r // c["B"], int(c["slot_of"][r])
        W64, g64 = f64(c["W"][lyr]), f64(c["gate"][lyr])
        S_old, Z_old = c["states"][r]
        ref = ob.attend(f64(c["q"][r]), f64(c["k"][r]), f64(c["v"][r]), S_old, Z_old, W64, g64,
                        MERGES[merge])
        assert out_err(f64(o[r]), ref) <= TOL_OUT_BF16, r
        if c["commit"][r]:
            S_new, Z_new = ob.commit(S_old, Z_old, f64(c["k"][r]), f64(c["v"][r]), W64)
        else:
            S_new, Z_new = f64(S0[sl]), f64(Z0[sl])
        assert unit_err(f64(S[sl]), S_new, 1) <= TOL_STATE, r
        assert unit_err(f64(Z[sl]), Z_new, 1) <= TOL_STATE, r
    spare = sorted(set(range(c["R"] + 2)) - set(int(x) for x in c["slot_of"]))
    for sl in spare:
        assert torch.equal(S[sl], S0[sl]) and torch.equal(Z[sl], Z0[sl])


@pytest.mark.parametrize("with_commit", [True, False])
@pytest.mark.parametrize("dt,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_layers_equal_one_call_per_layer(cuda_device, with_commit, dt, d):
    """The production shape runs as one launch, the others as one call per
    layer: both must give what per-layer calls give, bit for bit. 6 layers
    of 64 requests put every CTA on many units of different layers."""
    B = 64 if d == 128 else 8
    c = _case(dt, n_layers=6, B=B, L=32, d=d, f=d // 2, seed=930, max_prefix=64)
    cfg = _cfg(c, dt, "shared_norm")
    S, Z = _pool(c, cfg, cuda_device)
    S2, Z2 = S.clone(), Z.clone()
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = dev(c["slot_of"].to(torch.int32))
    q, k, v, W, gate = dev(c["q"]), dev(c["k"]), dev(c["v"]), dev(c["W"]), dev(c["gate"])
    cm = dev(c["commit"]) if with_commit else None
    o = hb.hb_block_attend_commit_layers(cfg, sl, q, k, v, S, Z, W, gate, cm)
    assert_status_ok()
    o2 = torch.empty_like(o)
    for lyr in range(c["n_layers"]):
        r = slice(lyr * B, (lyr + 1) * B)
        if with_commit:
            hb.hb_block_attend_commit(cfg, sl[r], q[r], k[r], v[r], S2, Z2, W[lyr], gate[lyr],
                                      cm[r], o=o2[r])
        else:
            hb.hb_block_attend(cfg, sl[r], q[r], k[r], v[r], S2, Z2, W[lyr], gate[lyr], o=o2[r])
    assert_status_ok()
    assert torch.equal(o, o2)
    assert torch.equal(S, S2) and torch.equal(Z, Z2)
    if not with_commit:
        # attend only: the pools are only read
        S0, Z0 = _pool(c, cfg, cuda_device)
        assert torch.equal(S, S0) and torch.equal(Z, Z0)


@pytest.mark.parametrize("n_layers,L,mask", [(1, 32, "some"), (3, 16, "all"), (4, 32, "none")])
def test_layers_edge_cases(cuda_device, n_layers, L, mask):
    """One layer (the plain fused step), 16-token blocks with every request
    committing, and a commit mask of zeros: bit for bit what per-layer calls
    give."""
    B = 20
    c = _case(torch.bfloat16, n_layers=n_layers, B=B, L=L, seed=970 + n_layers, max_prefix=48)
    if mask == "all":
        c["commit"] = torch.ones(c["R"], dtype=torch.int32)
    elif mask == "none":
        c["commit"] = torch.zeros(c["R"], dtype=torch.int32)
    cfg = _cfg(c, torch.bfloat16, "convex")
    S, Z = _pool(c, cfg, cuda_device)
    S2, Z2 = S.clone(), Z.clone()
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = dev(c["slot_of"].to(torch.int32))
    q, k, v, W, gate = dev(c["q"]), dev(c["k"]), dev(c["v"]), dev(c["W"]), dev(c["gate"])
    cm = dev(c["commit"])
    o = hb.hb_block_attend_commit_layers(cfg, sl, q, k, v, S, Z, W, gate, cm)
    o2 = torch.empty_like(o)
    for lyr in range(n_layers):
        r = slice(lyr * B, (lyr + 1) * B)
        hb.hb_block_attend_commit(cfg, sl[r], q[r], k[r], v[r], S2, Z2, W[lyr], gate[lyr], cm[r],
                                  o=o2[r])
    assert_status_ok()
    assert torch.equal(o, o2)
    assert torch.equal(S, S2) and torch.equal(Z, Z2)


def test_layers_reject_bad_shapes(cuda_device):
    c = _case(torch.bfloat16, n_layers=2, B=4, L=32, seed=960, max_prefix=8)
    cfg = _cfg(c, torch.bfloat16, "shared_norm")
    S, Z = _pool(c, cfg, cuda_device)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = dev(c["slot_of"].to(torch.int32))
    # 8 requests do not split into 3 layers
    W3 = dev(torch.cat([c["W"], c["W"][:1]]))
    g3 = dev(torch.cat([c["gate"], c["gate"][:1]]))
    with pytest.raises(ValueError):
        hb.hb_block_attend_commit_layers(cfg, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S, Z,
                                         W3, g3)
    assert np.isfinite(S.cpu().numpy()).all()

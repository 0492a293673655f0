"""Block lengths other than 32 on the tensor-core path (GPU): a decoding step
(attend, and attend with commits) and prompts with outputs for L = 16 and
L = 64, through the same C-ABI calls, against the oracle on every request.
The oracle pins that the state a prompt leaves does not depend on the block
length; here the GPU's outputs and states follow the oracle at each L."""

import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from tests.parity import (TOL_OUT_BF16, TOL_STATE, assert_status_ok, f64, new_pool, out_err,
                          unit_err)

pytestmark = pytest.mark.gpu

MERGES = {"shared_norm": hb.MERGE_SHARED_NORM, "convex": hb.MERGE_CONVEX}
H, D, FH = 16, 128, 64


def _batch(B, L, seed, max_prefix=80):
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn((H, D, FH), generator=g) * D ** -0.5).to(torch.bfloat16)
    gate = torch.randn((H,), generator=g)
    q, k, v = (torch.randn((B, L, H, D), generator=g).to(torch.bfloat16) for _ in range(3))
    lens = torch.randint(0, max_prefix + 1, (B,), generator=g).tolist()
    states = []
    for n in lens:
        pk = torch.randn((n, H, D), generator=g).to(torch.bfloat16)
        pv = torch.randn((n, H, D), generator=g).to(torch.bfloat16)
        states.append(ob.prefill(f64(pk), f64(pv), f64(W)))
    slot_of = torch.randperm(B + 3, generator=g)[:B]
    commit = (torch.rand(B, generator=g) < 0.4).to(torch.int32)
    return dict(W=W, gate=gate, q=q, k=k, v=v, states=states, slot_of=slot_of, commit=commit)


def _pool(c, B, dev):
    cfg = hb.Config(H, D, FH, 32)
    S, Z = new_pool(cfg, B + 3, dev)
    S.fill_(2.0)
    Z.fill_(2.0)
    for b in range(B):
        S[int(c["slot_of"][b])] = torch.as_tensor(c["states"][b][0], dtype=torch.float32)
        Z[int(c["slot_of"][b])] = torch.as_tensor(c["states"][b][1], dtype=torch.float32)
    return S, Z


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("L", [16, 64])
@pytest.mark.parametrize("with_commit", [False, True])
def test_step_matches_oracle(cuda_device, merge, L, with_commit):
    B = 24
    c = _batch(B, L, seed=L + 7 * with_commit)
    cfg = hb.Config(H, D, FH, L, merge=MERGES[merge])
    S, Z = _pool(c, B, cuda_device)
    S0, Z0 = S.clone(), Z.clone()
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    if with_commit:
        o = hb.hb_block_attend_commit(cfg, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S, Z,
                                      dev(c["W"]), dev(c["gate"]), dev(c["commit"]))
    else:
        o = hb.hb_block_attend(cfg, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S, Z,
                               dev(c["W"]), dev(c["gate"]))
    assert_status_ok()
    W64 = f64(c["W"])
    for b in range(B):
        S_old, Z_old = c["states"][b]
        q64, k64, v64 = f64(c["q"][b]), f64(c["k"][b]), f64(c["v"][b])
        ref = ob.attend(q64, k64, v64, S_old, Z_old, W64, f64(c["gate"]), MERGES[merge])
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16, b
        slot = int(c["slot_of"][b])
        if with_commit and int(c["commit"][b]):
            S_new, Z_new = ob.commit(S_old, Z_old, k64, v64, W64)
            assert unit_err(f64(S[slot]), S_new, 1) <= TOL_STATE, b
            assert unit_err(f64(Z[slot]), Z_new, 1) <= TOL_STATE, b
        else:
            assert torch.equal(S[slot], S0[slot]) and torch.equal(Z[slot], Z0[slot]), b
    spare = set(range(B + 3)) - set(int(x) for x in c["slot_of"])
    for slot in spare:
        assert torch.equal(S[slot], S0[slot]), slot


@pytest.mark.parametrize("merge", sorted(MERGES))
@pytest.mark.parametrize("L,T", [(16, 48), (16, 272), (64, 64), (64, 320)])
def test_prompt_matches_oracle(cuda_device, merge, L, T):
    """Prompts cut into 16- or 64-token blocks: below one 128-token segment,
    and several segments with a partial last one; 3 prompts continuing
    earlier context at permuted slots."""
    B = 3
    cfg = hb.Config(H, D, FH, L, merge=MERGES[merge])
    g = torch.Generator().manual_seed(1000 + L + T)
    W = (torch.randn((H, D, FH), generator=g) * D ** -0.5).to(torch.bfloat16)
    gate = torch.randn((H,), generator=g)
    q, k, v = (torch.randn((B, T, H, D), generator=g).to(torch.bfloat16) for _ in range(3))
    S, Z = new_pool(cfg, B + 2, cuda_device)
    slot_of = [4, 0, 2]
    starts = []
    for b in range(B):
        n = 40 * b
        pk = torch.randn((n, H, D), generator=g).to(torch.bfloat16)
        pv = torch.randn((n, H, D), generator=g).to(torch.bfloat16)
        s0, z0 = ob.prefill(f64(pk), f64(pv), f64(W))
        starts.append((s0, z0))
        S[slot_of[b]] = torch.as_tensor(s0, dtype=torch.float32, device=cuda_device)
        Z[slot_of[b]] = torch.as_tensor(z0, dtype=torch.float32, device=cuda_device)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    o = hb.hb_prefill_attend(cfg, torch.tensor(slot_of, dtype=torch.int32, device=cuda_device),
                             dev(q), dev(k), dev(v), S, Z, dev(W), dev(gate), accumulate=True)
    assert_status_ok()
    for b in range(B):
        o_ref, S_ref, Z_ref = ob.prefill_attend(f64(q[b]), f64(k[b]), f64(v[b]), f64(W),
                                                f64(gate), L, MERGES[merge], S0=starts[b][0],
                                                Z0=starts[b][1])
        for j0 in range(0, T, L):
            assert out_err(f64(o[b, j0:j0 + L]), o_ref[j0:j0 + L]) <= TOL_OUT_BF16, (b, j0)
        assert unit_err(f64(S[slot_of[b]]), S_ref, 1) <= TOL_STATE, b
        assert unit_err(f64(Z[slot_of[b]]), Z_ref, 1) <= TOL_STATE, b


@pytest.mark.parametrize("merge", sorted(MERGES))
def test_step16_many_units_per_cta_matches_oracle(cuda_device, merge):
    """16-token blocks on the persistent attend kernel at 320 requests (every
    CTA runs more than 32 units of 32-row tiles whose upper 16 rows belong to
    the next request): every request's output and committed state against
    the oracle, and nothing written past the last request's output rows."""
    B, L = 320, 16
    c = _batch(B, L, seed=1600, max_prefix=40)
    cfg = hb.Config(H, D, FH, L, merge=MERGES[merge])
    S, Z = _pool(c, B, cuda_device)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    buf = torch.full((B + 1, L, H, D), 7.0, dtype=torch.bfloat16, device=cuda_device)
    o = hb.hb_block_attend_commit(cfg, sl, dev(c["q"]), dev(c["k"]), dev(c["v"]), S, Z,
                                  dev(c["W"]), dev(c["gate"]), dev(c["commit"]), o=buf[:B])
    assert_status_ok()
    assert bool((buf[B] == 7.0).all())
    W64 = f64(c["W"])
    for b in range(B):
        S_old, Z_old = c["states"][b]
        q64, k64, v64 = f64(c["q"][b]), f64(c["k"][b]), f64(c["v"][b])
        ref = ob.attend(q64, k64, v64, S_old, Z_old, W64, f64(c["gate"]), MERGES[merge])
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16, b
        if int(c["commit"][b]):
            S_new, Z_new = ob.commit(S_old, Z_old, k64, v64, W64)
            slot = int(c["slot_of"][b])
            assert unit_err(f64(S[slot]), S_new, 1) <= TOL_STATE, b
            assert unit_err(f64(Z[slot]), Z_new, 1) <= TOL_STATE, b


def test_step16_bf16_copies_equal_fp32(cuda_device):
    """16-token blocks: the attend that reads the bf16 copy of the states,
    and the dual-copy step, give the fp32 pool's output (and masters) bit for
    bit, as at 32 tokens."""
    B, L = 64, 16
    c = _batch(B, L, seed=1601, max_prefix=40)
    cfg = hb.Config(H, D, FH, L)
    S, Z = _pool(c, B, cuda_device)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = c["slot_of"].to(torch.int32).to(cuda_device)
    q, k, v, W, gate = (dev(c[n]) for n in ("q", "k", "v", "W", "gate"))
    S16 = S.to(torch.bfloat16)
    o_ref = hb.hb_block_attend(cfg, sl, q, k, v, S, Z, W, gate)
    o16 = hb.hb_block_attend_s16(cfg, sl, q, k, v, S16, Z, W, gate)
    assert_status_ok()
    assert torch.equal(o16, o_ref)
    S2, Z2 = S.clone(), Z.clone()
    mask = dev(c["commit"])
    o_ref = hb.hb_block_attend_commit(cfg, sl, q, k, v, S, Z, W, gate, mask)
    o_dual = hb.hb_block_attend_commit_s16(cfg, sl, q, k, v, S2, S16, Z2, W, gate, mask)
    assert_status_ok()
    assert torch.equal(o_dual, o_ref) and torch.equal(S2, S) and torch.equal(Z2, Z)
    idx = sl.long()
    assert torch.equal(S16[idx], S2[idx].to(torch.bfloat16))


@pytest.mark.parametrize("Hkv", [4, 16])
def test_step16_grouped_heads_match_oracle(cuda_device, Hkv):
    """16-token blocks with 16 query heads over Hkv key/value heads and a
    separate key map: outputs and committed per-group states."""
    B, L = 40, 16
    g = torch.Generator().manual_seed(1602 + Hkv)
    q = torch.randn((B, L, H, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, L, Hkv, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, L, Hkv, D), generator=g).to(torch.bfloat16)
    Wq = (torch.randn((H, D, FH), generator=g) * D ** -0.5).to(torch.bfloat16)
    Wk = (torch.randn((Hkv, D, FH), generator=g) * D ** -0.5).to(torch.bfloat16)
    gate = torch.randn((H,), generator=g)
    states = []
    for b in range(B):
        n = int(torch.randint(0, 41, (1,), generator=g))
        pk = torch.randn((n, Hkv, D), generator=g).to(torch.bfloat16)
        pv = torch.randn((n, Hkv, D), generator=g).to(torch.bfloat16)
        states.append(ob.prefill(f64(pk), f64(pv), f64(Wk)))
    commit = (torch.rand(B, generator=g) < 0.4).to(torch.int32)
    S = torch.stack([torch.as_tensor(s0, dtype=torch.float32) for s0, _ in states])
    Z = torch.stack([torch.as_tensor(z0, dtype=torch.float32) for _, z0 in states])
    S, Z = S.to(cuda_device), Z.to(cuda_device)
    cfg = hb.Config(H, D, FH, L)
    dev = lambda x: x.to(cuda_device)  # noqa: E731
    sl = torch.arange(B, dtype=torch.int32, device=cuda_device)
    o = hb.hb_block_attend_ex(cfg, Hkv, sl, dev(q), dev(k), dev(v), S, Z, dev(Wq), dev(gate),
                              Wk=dev(Wk), commit=dev(commit))
    assert_status_ok()
    for b in range(B):
        S_old, Z_old = states[b]
        ref = ob.attend_gqa(f64(q[b]), f64(k[b]), f64(v[b]), S_old, Z_old, f64(Wq), f64(gate),
                            hb.MERGE_SHARED_NORM)
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16, b
        if int(commit[b]):
            S_new, Z_new = ob.commit(S_old, Z_old, f64(k[b]), f64(v[b]), f64(Wk))
            assert unit_err(f64(S[b]), S_new, 1) <= TOL_STATE, b
            assert unit_err(f64(Z[b]), Z_new, 1) <= TOL_STATE, b

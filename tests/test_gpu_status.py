"""Device-side faults are reported, not trapped: an out-of-range slot or a
ragged length that does not fit its buffer skips that request's work, sets
the device status word, and leaves the rest of the call correct (GPU)."""

import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from linear_attention_diffusion_feature_b300 import inputs
from tests.parity import TOL_OUT_BF16, assert_status_ok, config, f64, new_pool, out_err, slots

pytestmark = pytest.mark.gpu

BOUNDS = 5


def test_attend_bad_slot_skips_that_request(cuda_device):
    w = inputs.continuous_batching(device=cuda_device, B=4, lo=8, hi=9, n_commit=0)
    cfg = config(w)
    t = w.tensors
    S, Z = new_pool(cfg, 4, cuda_device)
    hb.hb_prefill_state(cfg, slots(range(4), cuda_device), t["prefix_k"], t["prefix_v"],
                        t["cu_prefix"], w.meta["max_prefix"], t["W"], S, Z)
    assert_status_ok()
    o = torch.full_like(t["q"], 7.0)
    hb.hb_block_attend(cfg, slots([0, 4, 2, -1], cuda_device), t["q"], t["k"], t["v"], S, Z,
                       t["W"], t["gate"], o=o)
    assert hb.hb_get_device_status() == BOUNDS
    assert hb.hb_get_device_status() == 0  # reading clears it
    assert bool((o[1] == 7.0).all()) and bool((o[3] == 7.0).all())
    cu = t["cu_prefix"].cpu()
    for b in (0, 2):
        a, e = int(cu[b]), int(cu[b + 1])
        S_ref, Z_ref = ob.prefill(f64(t["prefix_k"][a:e]), f64(t["prefix_v"][a:e]), f64(t["W"]))
        ref = ob.attend(f64(t["q"][b]), f64(t["k"][b]), f64(t["v"][b]), S_ref, Z_ref,
                        f64(t["W"]), f64(t["gate"]))
        assert out_err(f64(o[b]), ref) <= TOL_OUT_BF16


def test_commit_bad_slot_flagged(cuda_device):
    cfg = hb.Config(2, 128, 64, 32)
    S, Z = new_pool(cfg, 2, cuda_device)
    k = inputs.draw(1, (2, 32, 2, 128), device=cuda_device)
    W = inputs.draw(2, (2, 128, 64), device=cuda_device, std=128 ** -0.5)
    hb.hb_commit_block(cfg, slots([1, 2], cuda_device), k, k, W, S, Z)
    assert hb.hb_get_device_status() == BOUNDS
    assert float(S[1].abs().sum()) > 0 and float(S[0].abs().sum()) == 0


def test_prefill_ragged_lengths_out_of_range(cuda_device):
    cfg = hb.Config(2, 128, 64, 32)
    S, Z = new_pool(cfg, 3, cuda_device)
    k = inputs.draw(3, (100, 2, 128), device=cuda_device)
    W = inputs.draw(4, (2, 128, 64), device=cuda_device, std=128 ** -0.5)
    sl = slots([0, 1, 2], cuda_device)
    # request 1 runs past the 100 packed rows; request 2 has a negative length
    cu = torch.tensor([0, 40, 120, 60], dtype=torch.int64, device=cuda_device)
    hb.hb_prefill_state(cfg, sl, k, k, cu, 80, W, S, Z)
    assert hb.hb_get_device_status() == BOUNDS
    assert float(S[0].abs().sum()) > 0
    assert float(S[1].abs().sum()) == 0 and float(S[2].abs().sum()) == 0
    # a request longer than max_seqlen is skipped as well
    cu = torch.tensor([0, 40, 100, 100], dtype=torch.int64, device=cuda_device)
    S.zero_()
    hb.hb_prefill_state(cfg, sl, k, k, cu, 50, W, S, Z)
    assert hb.hb_get_device_status() == BOUNDS
    assert float(S[0].abs().sum()) > 0 and float(S[1].abs().sum()) == 0


def test_softmax_kv_prefix_out_of_range(cuda_device):
    cfg = hb.Config(2, 128, 64, 32)
    kc = inputs.draw(5, (64, 2, 128), device=cuda_device)
    q = inputs.draw(6, (2, 32, 2, 128), device=cuda_device)
    cu = torch.tensor([0, 64, 200], dtype=torch.int64, device=cuda_device)
    o = torch.full_like(q, 7.0)
    hb.hb_softmax_kv_attend(cfg, kc, kc, cu, 200, q, q, q, o=o)
    assert hb.hb_get_device_status() == BOUNDS
    assert bool((o[1] == 7.0).all()) and not bool((o[0] == 7.0).any())


def test_host_validation_raises(cuda_device):
    cfg = hb.Config(2, 128, 64, 32)
    S, Z = new_pool(cfg, 2, cuda_device)
    q = inputs.draw(7, (1, 32, 2, 128), device=cuda_device)
    W = inputs.draw(8, (2, 128, 64), device=cuda_device)
    gate = torch.zeros(2, device=cuda_device)
    with pytest.raises(ValueError):
        hb.hb_block_attend(cfg, slots([0], cuda_device), q, q, q[:, :16], S, Z, W, gate)
    with pytest.raises(TypeError):
        hb.hb_block_attend(cfg, slots([0], cuda_device), q.float(), q, q, S, Z, W, gate)
    bad = hb.Config(2, 128, 64, 32, scale=-1.0)
    with pytest.raises(hb.HBError):
        hb.hb_block_attend(bad, slots([0], cuda_device), q, q, q, S, Z, W, gate)


def test_tensors_on_another_device_are_refused(cuda_device, monkeypatch):
    """The library launches on the current device, so the binding refuses a
    tensor or a stream that lives on another one before anything is launched
    (emulated on one GPU by reporting another current device)."""
    cfg = hb.Config(2, 128, 64, 32)
    S, Z = new_pool(cfg, 2, cuda_device)
    q = inputs.draw(7, (1, 32, 2, 128), device=cuda_device)
    W = inputs.draw(8, (2, 128, 64), device=cuda_device, std=128 ** -0.5)
    gate = torch.zeros(2, device=cuda_device)
    sl = slots([0], cuda_device)
    o = torch.full_like(q, 7.0)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: cuda_device.index + 1)
    with pytest.raises(ValueError, match="current device"):
        hb.hb_block_attend(cfg, sl, q, q, q, S, Z, W, gate, o=o)
    monkeypatch.undo()
    torch.cuda.synchronize()
    assert bool((o == 7.0).all())
    assert hb.hb_get_device_status() == 0


TIMEOUT = 6


@pytest.mark.parametrize("variant", ["attend", "attend_commit", "prefill_attend"])
def test_wait_that_runs_out_is_reported_and_the_context_survives(cuda_device, variant):
    """Failure detection without a GPU fault: with the pipeline's wait limit
    lowered to a few clocks, the waits of the attend kernels run out before
    their copies land. The call must end on its own, report HB_ERR_TIMEOUT
    through the status word, and leave the context usable: with the default
    limit back, the same call on fresh inputs gives the bits a call before
    the fault gave."""
    B = 64 if variant != "prefill_attend" else 4
    w = inputs.continuous_batching(device=cuda_device, B=B, lo=2, hi=8, n_commit=B // 4)
    cfg = config(w)
    t = w.tensors
    S0, Z0 = new_pool(cfg, B, cuda_device)
    sl = slots(range(B), cuda_device)
    hb.hb_prefill_state(cfg, sl, t["prefix_k"], t["prefix_v"], t["cu_prefix"],
                        w.meta["max_prefix"], t["W"], S0, Z0)
    mask = torch.zeros(B, dtype=torch.int32, device=cuda_device)
    mask[t["commit_idx"]] = 1
    if variant == "prefill_attend":
        g = torch.Generator().manual_seed(9)
        q, k, v = (torch.randn((B, 8 * 32, 16, 128), generator=g).to(torch.bfloat16)
                   .to(cuda_device) for _ in range(3))

    def call(S, Z):
        if variant == "attend":
            return hb.hb_block_attend(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"], t["gate"])
        if variant == "attend_commit":
            return hb.hb_block_attend_commit(cfg, sl, t["q"], t["k"], t["v"], S, Z, t["W"],
                                             t["gate"], mask)
        return hb.hb_prefill_attend(cfg, sl, q, k, v, S, Z, t["W"], t["gate"])

    S1, Z1 = S0.clone(), Z0.clone()
    ref = call(S1, Z1)
    assert_status_ok()
    hb.hb_set_wait_limit(2)
    try:
        S2, Z2 = S0.clone(), Z0.clone()
        call(S2, Z2)
        status = hb.hb_get_device_status()
    finally:
        hb.hb_set_wait_limit(0)
    assert status == TIMEOUT
    S3, Z3 = S0.clone(), Z0.clone()
    again = call(S3, Z3)
    assert_status_ok()
    assert torch.equal(again, ref)
    assert torch.equal(S3, S1) and torch.equal(Z3, Z1)

"""The continuous-batching simulator on the GPU: a small request stream runs
to completion on both servers, and after it every state slot holds exactly
the oracle's state of the last request that used it: its prompt ingested,
then each committed block folded in (so admission, slot recycling and the
commit masks drive the library's calls as the scheduler says)."""

import pytest
import torch

import linear_attention_diffusion_feature_b300 as hb
import oracle.block_hybrid as ob
from linear_attention_diffusion_feature_b300 import serving
from tests.parity import TOL_STATE, assert_status_ok, f64, unit_err

pytestmark = pytest.mark.gpu


def _cfg():
    return serving.ServeConfig(n_requests=7, max_concurrency=3, gen_tokens=96,
                               steps_per_block=2, prompt_min=32, prompt_max=96,
                               memory_budget=1 << 40, layers=2)


def test_hybrid_server_states_match_oracle(cuda_device):
    cfg = _cfg()
    syn = serving._Synthetic(cfg, cuda_device)
    be = serving.HybridBackend(cfg, cuda_device, syn)
    trace = []
    res = serving.simulate(be, cfg, trace=trace)
    assert_status_ok()
    assert res.finished == 7 and res.tokens == 7 * 96
    # the last occupant of each slot and what its state is made of
    last = {}
    for ev in trace:
        if ev[0] == "ingest":
            _, rid, slot, row, n = ev
            last[slot] = dict(rid=rid, row=row, n=n, commits=[])
        else:
            _, rid, slot, b = ev
            assert last[slot]["rid"] == rid
            last[slot]["commits"].append(b)
    assert sorted(last) == [0, 1, 2]
    for layer, ly in enumerate(syn.layers):
        W = f64(ly["W"])
        for slot, rec in last.items():
            assert len(rec["commits"]) == 3
            a, n = rec["row"], rec["n"]
            S_ref, Z_ref = ob.prefill(f64(ly["pk"][a:a + n]), f64(ly["pv"][a:a + n]), W)
            for b in rec["commits"]:
                S_ref, Z_ref = ob.commit(S_ref, Z_ref, f64(ly["k"][b]), f64(ly["v"][b]), W)
            assert unit_err(f64(be.S[layer][slot]), S_ref, 1) <= TOL_STATE, (layer, slot)
            assert unit_err(f64(be.Z[layer][slot]), Z_ref, 1) <= TOL_STATE, (layer, slot)


def test_softmax_server_pages_hold_the_committed_tokens(cuda_device):
    """The comparison server's paged cache: when a request finishes, its pages
    (in table order) hold its prompt and then its committed blocks, and its
    prefix length counts them (checked just before the pages return to the
    pool, where later requests reuse them)."""
    cfg = _cfg()
    syn = serving._Synthetic(cfg, cuda_device)
    trace = []
    checked = []

    class Checked(serving.SoftmaxBackend):
        def release(self, reqs):
            for r in reqs:
                ing = [ev for ev in trace if ev[0] == "ingest" and ev[1] == r.rid][0]
                blocks = [ev[3] for ev in trace if ev[0] == "commit" and ev[1] == r.rid]
                row, n = ing[3], ing[4]
                P = int(self.plen[r.slot])
                assert P == n + 32 * len(blocks) == n + cfg.gen_tokens
                pages = self.table[r.slot, :P // 32].long()
                for ly, kp, vp in zip(syn.layers, self.kp, self.vp):
                    for pool, src, act in ((kp, "pk", "k"), (vp, "pv", "v")):
                        got = pool.index_select(0, pages).reshape(P, cfg.H, cfg.d)
                        want = torch.cat([ly[src][row:row + n]] + [ly[act][b] for b in blocks])
                        assert torch.equal(got, want), r.rid
                checked.append(r.rid)
            super().release(reqs)

    be = Checked(cfg, cuda_device, syn)
    res = serving.simulate(be, cfg, trace=trace)
    assert_status_ok()
    assert res.finished == 7
    assert sorted(checked) == list(range(7))

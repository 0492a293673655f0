"""Plants plausible mistakes in the oracle (on the CPU) and checks that the
pins notice each one: a dropped term, a wrong sign, a wrong index or axis, a
transposed operand. A mutation counts as caught when any pin check raises."""

import numpy as np
import pytest

import oracle.block_hybrid as ob
from tests import oracle_checks


def _fm_swapped_halves(x, W):
    u = np.asarray(x, np.float64) @ np.asarray(W, np.float64)
    return np.concatenate([ob._softmax_last(-u), ob._softmax_last(u)], axis=-1)


def _fm_no_negation(x, W):
    u = np.asarray(x, np.float64) @ np.asarray(W, np.float64)
    return np.concatenate([ob._softmax_last(u), ob._softmax_last(u)], axis=-1)


def _softmax_wrong_axis(u):
    e = np.exp(u - u.max(axis=0, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


def _commit_drops_previous(S, Z, k, v, W):
    S = np.zeros_like(np.asarray(S, np.float64))
    Z = np.zeros_like(np.asarray(Z, np.float64))
    return _ORIG["commit"](S, Z, k, v, W)


def _commit_swaps_kv(S, Z, k, v, W):
    return _ORIG["commit"](S, Z, v, k, W)


def _commit_transposed(S, Z, k, v, W):
    S = np.asarray(S, np.float64).copy()
    Z = np.asarray(Z, np.float64).copy()
    for h in range(W.shape[0]):
        phi = ob.feature_map(np.asarray(k)[:, h, :], np.asarray(W)[h])
        S[h] += (np.asarray(v)[:, h, :].T @ phi).T.T  # [d, F] added into [F, d]
        Z[h] += phi.sum(axis=0)
    return S, Z


def _scale_one_over_d(d, scale):
    return 1.0 / d if (scale is None or scale == 0) else float(scale)


def _sigmoid_wrong_sign(g):
    return _ORIG["sigmoid"](-np.asarray(g, np.float64))


def _make_attend(variant):
    def attend(q, k, v, S, Z, W, gate, merge=ob.MERGE_SHARED_NORM, scale=None):
        q, k, v, S, Z, W = (np.asarray(a, np.float64) for a in (q, k, v, S, Z, W))
        L, H, d = q.shape
        sc = ob._scale(d, scale)
        w = ob.sigmoid(gate)
        o = np.empty((L, H, d))
        for h in range(H):
            s = sc * (q[:, h, :] @ k[:, h, :].T)
            e = np.exp(s)
            if variant == "softmax_over_queries":
                e = e.T
            sm_num = e @ v[:, h, :]
            sm_den = e.sum(axis=1)
            src = k if variant == "phi_of_key" else q
            phi_q = ob.feature_map(src[:, h, :], W[h])
            num = phi_q @ S[h]
            den = phi_q @ Z[h]
            if merge == ob.MERGE_SHARED_NORM:
                if variant == "gate_on_linear":
                    o[:, h, :] = (sm_num + w[h] * num) / (sm_den + w[h] * den)[:, None]
                elif variant == "gate_on_numerator_only":
                    o[:, h, :] = (w[h] * sm_num + num) / (sm_den + den)[:, None]
                else:
                    o[:, h, :] = (w[h] * sm_num + num) / (w[h] * sm_den + den)[:, None]
            else:
                o_soft = sm_num / sm_den[:, None]
                o_lin = np.where(den[:, None] > 0, num / np.where(den > 0, den, 1.0)[:, None], o_soft)
                a = (1.0 - w[h]) if variant == "convex_swapped" else w[h]
                o[:, h, :] = a * o_soft + (1.0 - a) * o_lin
        return o
    return attend


def _softmax_kv_no_block(k_prefix, v_prefix, q, k, v, scale=None):
    if np.asarray(k_prefix).shape[0] == 0:
        return _ORIG["softmax_kv_attend"](k_prefix, v_prefix, q, k, v, scale)
    return _ORIG["softmax_kv_attend"](k_prefix[:-1], v_prefix[:-1], q, k_prefix[-1:], v_prefix[-1:], scale)


def _prefill_attend_commit_first(q, k, v, W, gate, L, merge=ob.MERGE_SHARED_NORM, scale=None,
                                 S0=None, Z0=None):
    """Commits each block before it attends (the block sees itself twice)."""
    q, k, v, W = (np.asarray(a, np.float64) for a in (q, k, v, W))
    T, H, d = q.shape
    f = W.shape[2]
    S = np.zeros((H, 2 * f, d)) if S0 is None else np.asarray(S0, np.float64).copy()
    Z = np.zeros((H, 2 * f)) if Z0 is None else np.asarray(Z0, np.float64).copy()
    o = np.empty((T, H, d))
    for j0 in range(0, T, L):
        blk = slice(j0, j0 + L)
        S, Z = ob.commit(S, Z, k[blk], v[blk], W)
        o[blk] = ob.attend(q[blk], k[blk], v[blk], S, Z, W, gate, merge, scale)
    return o, S, Z


def _prefill_attend_ignores_context(q, k, v, W, gate, L, merge=ob.MERGE_SHARED_NORM, scale=None,
                                    S0=None, Z0=None):
    """Starts from an empty state even when an earlier context is given."""
    return _ORIG["prefill_attend"](q, k, v, W, gate, L, merge, scale)



def _gather_pool_order(pages, page_ids, P):
    """Reads pages in pool order instead of through the page table."""
    return _ORIG["gather_pages"](pages, np.arange(np.asarray(pages).shape[0]), P)


def _gather_page_slot_swapped(pages, page_ids, P):
    """Swaps the roles of page index and slot: page t mod p, slot t // p."""
    pages = np.asarray(pages, np.float64)
    p = pages.shape[1]
    rows = [pages[int(page_ids[t % p]), t // p] for t in range(int(P))]
    return np.stack(rows) if rows else np.zeros((0,) + pages.shape[2:])


def _gather_whole_pages(pages, page_ids, P):
    """Reads every slot of the request's pages, past token P - 1 too."""
    p = np.asarray(pages).shape[1]
    return _ORIG["gather_pages"](pages, page_ids, -(-int(P) // p) * p)


def _kv_head_modulo(h, H, H_kv):
    """Groups query heads by h mod H_kv instead of consecutive runs."""
    return h % H_kv


def _prefill_attend_commit_with_query_map(q, k, v, W, gate, L, merge=ob.MERGE_SHARED_NORM,
                                          scale=None, S0=None, Z0=None, Wk=None):
    """Builds the state with the query map, ignoring the key map."""
    if Wk is not None and np.asarray(Wk).shape == np.asarray(W).shape:
        Wk = W
    elif Wk is not None:
        Wk = np.asarray(W)[::np.asarray(W).shape[0] // np.asarray(Wk).shape[0]]
    return _ORIG["prefill_attend"](q, k, v, W, gate, L, merge, scale, S0, Z0, Wk)


_ORIG = {name: getattr(ob, name) for name in
         ("commit", "sigmoid", "softmax_kv_attend", "feature_map", "_softmax_last", "_scale", "attend",
          "prefill_attend", "gather_pages", "kv_head")}

MUTATIONS = {
    "phi halves swapped": {"feature_map": _fm_swapped_halves},
    "phi negative half not negated": {"feature_map": _fm_no_negation},
    "softmax over the wrong axis": {"_softmax_last": _softmax_wrong_axis},
    "commit drops the previous state": {"commit": _commit_drops_previous},
    "commit swaps k and v": {"commit": _commit_swaps_kv},
    "commit transposed outer product": {"commit": _commit_transposed},
    "scale 1/d instead of 1/sqrt(d)": {"_scale": _scale_one_over_d},
    "gate logistic of -g": {"sigmoid": _sigmoid_wrong_sign},
    "gate on the linear branch": {"attend": _make_attend("gate_on_linear")},
    "gate on the numerator only": {"attend": _make_attend("gate_on_numerator_only")},
    "block softmax over queries": {"attend": _make_attend("softmax_over_queries")},
    "linear read uses phi(k) of the block": {"attend": _make_attend("phi_of_key")},
    "convex weights swapped": {"attend": _make_attend("convex_swapped")},
    "comparison drops block keys": {"softmax_kv_attend": _softmax_kv_no_block},
    "prompt block committed before it attends": {"prefill_attend": _prefill_attend_commit_first},
    "prompt ignores the earlier context": {"prefill_attend": _prefill_attend_ignores_context},
    "paged gather ignores the page table": {"gather_pages": _gather_pool_order},
    "paged gather swaps page and slot": {"gather_pages": _gather_page_slot_swapped},
    "paged gather reads whole pages": {"gather_pages": _gather_whole_pages},
    "grouped heads taken modulo": {"kv_head": _kv_head_modulo},
    "prompt state built with the query map": {
        "prefill_attend": _prefill_attend_commit_with_query_map},
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    for attr, fn in MUTATIONS[name].items():
        monkeypatch.setattr(ob, attr, fn)
    failed = []
    for check in oracle_checks.ALL_CHECKS:
        try:
            check(ob)
        except Exception:  # noqa: BLE001 - any failure or shape error counts
            failed.append(check.__name__)
    assert failed, f"no pin noticed the planted mistake: {name}"

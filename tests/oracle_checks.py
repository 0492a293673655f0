"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each ``check_*`` function takes the oracle module, runs it, and raises
``AssertionError`` when the oracle disagrees with a fact fixed by the pages or
by mathematics: hand-derived values (``tests/golden``), closed forms,
invariants, limits that reduce to a library routine (scipy / torch), and an
independent token-by-token formulation. ``test_oracle_pins`` runs them on the
real oracle; ``test_oracle_mutations`` plants plausible mistakes in the oracle
and checks that at least one of them fails.
"""

from __future__ import annotations

import numpy as np
import scipy.special
import torch

from tests import golden

RTOL = 1e-12
ATOL = 1e-12


def _close(a, b, rtol=RTOL, atol=ATOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    np.testing.assert_allclose(a, b, rtol=rtol, atol=atol)


def _rand_problem(seed, L=5, H=2, d=6, f=2, N=7):
    """Small random problem with F = 2f != d so that a transposed operand
    breaks shapes instead of passing silently."""
    g = np.random.default_rng(seed)
    return dict(
        q=g.standard_normal((L, H, d)),
        k=g.standard_normal((L, H, d)),
        v=g.standard_normal((L, H, d)),
        k_prev=g.standard_normal((N, H, d)),
        v_prev=g.standard_normal((N, H, d)),
        W=g.standard_normal((H, d, f)) / np.sqrt(d),
        gate=g.standard_normal(H),
    )


def _sdpa(q, k, v, scale=None):
    """torch fp64 CPU scaled_dot_product_attention per head, no mask.
    q [L, H, d], k/v [M, H, d] -> [L, H, d]."""
    tq = torch.from_numpy(np.ascontiguousarray(np.transpose(q, (1, 0, 2))))
    tk = torch.from_numpy(np.ascontiguousarray(np.transpose(k, (1, 0, 2))))
    tv = torch.from_numpy(np.ascontiguousarray(np.transpose(v, (1, 0, 2))))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk[None], tv[None], scale=scale)[0]
    return np.transpose(out.numpy(), (1, 0, 2))


# ---------------------------------------------------------------- feature map

def check_feature_map_golden(ob):
    g = golden.load("feature_map_hand.json")
    phi = ob.feature_map(np.array(g["x"]), np.array(g["W"]))
    _close(phi, g["phi"])


def check_feature_map_vs_scipy(ob):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((9, 16))
    W = rng.standard_normal((16, 8)) / 4.0
    u = x @ W
    ref = np.concatenate([scipy.special.softmax(u, axis=1),
                          scipy.special.softmax(-u, axis=1)], axis=1)
    _close(ob.feature_map(x, W), ref)


def check_feature_map_invariants(ob):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((11, 12))
    W = rng.standard_normal((12, 5))
    phi = ob.feature_map(x, W)
    assert phi.shape == (11, 10)
    assert np.all(phi > 0)
    _close(phi[:, :5].sum(1), np.ones(11))
    _close(phi[:, 5:].sum(1), np.ones(11))
    # W = 0: both halves are the uniform distribution 1/f.
    _close(ob.feature_map(x, np.zeros((12, 5))), np.full((11, 10), 0.2))
    # Negating W swaps the halves.
    neg = ob.feature_map(x, -W)
    _close(neg[:, :5], phi[:, 5:])
    _close(neg[:, 5:], phi[:, :5])


# --------------------------------------------------------------- commit / state

def check_commit_golden(ob):
    g = golden.load("merge_hand.json")
    W = np.zeros((1, 2, 2))
    kc = np.array(g["k_committed"])[:, None, :]
    vc = np.array(g["v_committed"])[:, None, :]
    S, Z = ob.prefill(kc, vc, W)
    _close(S[0], g["S"])
    _close(Z[0], g["Z"])


def check_commit_chunking(ob):
    """The state is a plain sum over committed tokens: committing blocks one
    by one, in one chunk, or in any other chunking gives the same state."""
    p = _rand_problem(3, N=13)
    H, d, f = p["W"].shape
    S1 = np.zeros((H, 2 * f, d))
    Z1 = np.zeros((H, 2 * f))
    for t in range(13):  # token by token
        S1, Z1 = ob.commit(S1, Z1, p["k_prev"][t:t + 1], p["v_prev"][t:t + 1], p["W"])
    S2, Z2 = ob.prefill(p["k_prev"], p["v_prev"], p["W"])  # one chunk
    S3 = np.zeros((H, 2 * f, d))
    Z3 = np.zeros((H, 2 * f))
    for a, b in [(0, 4), (4, 5), (5, 13)]:  # ragged chunks
        S3, Z3 = ob.commit(S3, Z3, p["k_prev"][a:b], p["v_prev"][a:b], p["W"])
    for S, Z in ((S2, Z2), (S3, Z3)):
        _close(S, S1)
        _close(Z, Z1)


def check_commit_sum_invariants(ob):
    """Each half of phi sums to 1, so sum_i Z_i = 2N and
    sum_i S_{i,:} = 2 sum_t v_t."""
    p = _rand_problem(4, N=10)
    S, Z = ob.prefill(p["k_prev"], p["v_prev"], p["W"])
    _close(Z.sum(axis=1), np.full(Z.shape[0], 20.0))
    _close(S.sum(axis=1), 2.0 * p["v_prev"].sum(axis=0))


def check_commit_outer_products(ob):
    """S equals the sum of the rank-1 terms phi(k_t) v_t^T built one
    coordinate at a time from the scipy softmax."""
    p = _rand_problem(5, N=6)
    H, d, f = p["W"].shape
    S, Z = ob.prefill(p["k_prev"], p["v_prev"], p["W"])
    for h in range(H):
        S_ref = np.zeros((2 * f, d))
        Z_ref = np.zeros(2 * f)
        for t in range(6):
            u = p["k_prev"][t, h] @ p["W"][h]
            phi = np.concatenate([scipy.special.softmax(u), scipy.special.softmax(-u)])
            for i in range(2 * f):
                Z_ref[i] += phi[i]
                for j in range(d):
                    S_ref[i, j] += phi[i] * p["v_prev"][t, h, j]
        _close(S[h], S_ref)
        _close(Z[h], Z_ref)


# ---------------------------------------------------------------------- attend

def check_merge_golden(ob):
    g = golden.load("merge_hand.json")
    q = np.array(g["q"])[:, None, :]
    k = np.array(g["k"])[:, None, :]
    v = np.array(g["v"])[:, None, :]
    W = np.zeros((1, 2, 2))
    S, Z = ob.prefill(np.array(g["k_committed"])[:, None, :],
                      np.array(g["v_committed"])[:, None, :], W)
    gate = np.array([g["gate_logit"]])
    o_sn = ob.attend(q, k, v, S, Z, W, gate, ob.MERGE_SHARED_NORM)
    o_cv = ob.attend(q, k, v, S, Z, W, gate, ob.MERGE_CONVEX)
    _close(o_sn[:, 0, :], g["o_shared_norm"])
    _close(o_cv[:, 0, :], g["o_convex"])


def check_empty_state_is_softmax_attention(ob):
    """No committed tokens: SHARED_NORM (any gate) and CONVEX reduce to plain
    softmax attention within the block (torch fp64 SDPA)."""
    p = _rand_problem(6)
    H, d, f = p["W"].shape
    S0 = np.zeros((H, 2 * f, d))
    Z0 = np.zeros((H, 2 * f))
    ref = _sdpa(p["q"], p["k"], p["v"])
    for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
        _close(ob.attend(p["q"], p["k"], p["v"], S0, Z0, p["W"], p["gate"], merge), ref, rtol=1e-10)
    # explicit scale is honoured
    ref2 = _sdpa(p["q"], p["k"], p["v"], scale=0.3)
    _close(ob.attend(p["q"], p["k"], p["v"], S0, Z0, p["W"], p["gate"],
                     ob.MERGE_SHARED_NORM, scale=0.3), ref2, rtol=1e-10)


def check_convex_soft_limit(ob):
    """CONVEX with sigmoid(g) = 1 ignores the state entirely."""
    p = _rand_problem(7)
    S, Z = ob.prefill(p["k_prev"], p["v_prev"], p["W"])
    gate = np.full(p["gate"].shape, np.inf)
    ref = _sdpa(p["q"], p["k"], p["v"])
    _close(ob.attend(p["q"], p["k"], p["v"], S, Z, p["W"], gate, ob.MERGE_CONVEX), ref, rtol=1e-10)


def check_state_vs_bruteforce(ob):
    """The state-based output equals the token-by-token kernel sum."""
    for seed in (8, 9):
        p = _rand_problem(seed)
        S, Z = ob.prefill(p["k_prev"], p["v_prev"], p["W"])
        for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
            a = ob.attend(p["q"], p["k"], p["v"], S, Z, p["W"], p["gate"], merge)
            b = ob.attend_bruteforce(p["q"], p["k"], p["v"], p["k_prev"], p["v_prev"],
                                     p["W"], p["gate"], merge)
            _close(a, b, rtol=1e-11)


def check_pure_linear_limits(ob):
    """sigmoid = 0 leaves only the linear branch: one committed token gives
    back its value; W = 0 gives the mean of the committed values."""
    p = _rand_problem(10, N=1)
    gate = np.full(p["gate"].shape, -np.inf)
    S, Z = ob.prefill(p["k_prev"], p["v_prev"], p["W"])
    for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
        o = ob.attend(p["q"], p["k"], p["v"], S, Z, p["W"], gate, merge)
        _close(o, np.broadcast_to(p["v_prev"][0], o.shape))
    p = _rand_problem(11, N=9)
    W0 = np.zeros_like(p["W"])
    S, Z = ob.prefill(p["k_prev"], p["v_prev"], W0)
    o = ob.attend(p["q"], p["k"], p["v"], S, Z, W0, gate, ob.MERGE_CONVEX)
    _close(o, np.broadcast_to(p["v_prev"].mean(axis=0), o.shape))


def check_block_permutation(ob):
    """Bidirectional (unmasked) in-block attention: permuting the active
    block's tokens permutes the outputs the same way."""
    p = _rand_problem(12, L=6)
    S, Z = ob.prefill(p["k_prev"], p["v_prev"], p["W"])
    perm = np.array([3, 0, 5, 1, 4, 2])
    for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
        o = ob.attend(p["q"], p["k"], p["v"], S, Z, p["W"], p["gate"], merge)
        op = ob.attend(p["q"][perm], p["k"][perm], p["v"][perm], S, Z, p["W"], p["gate"], merge)
        _close(op, o[perm])


def check_convex_combination(ob):
    """All weights are positive, so every output coordinate lies within the
    range of the values it mixes; constant values come back unchanged."""
    p = _rand_problem(13)
    for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
        S, Z = ob.prefill(p["k_prev"], p["v_prev"], p["W"])
        o = ob.attend(p["q"], p["k"], p["v"], S, Z, p["W"], p["gate"], merge)
        allv = np.concatenate([p["v"], p["v_prev"]], axis=0)
        assert np.all(o <= allv.max(axis=0)[None] + 1e-12)
        assert np.all(o >= allv.min(axis=0)[None] - 1e-12)
        c = np.array([0.5, -2.0, 3.0, 1.0, 0.0, -1.5])
        vc = np.broadcast_to(c, p["v"].shape)
        vpc = np.broadcast_to(c, p["v_prev"].shape)
        S, Z = ob.prefill(p["k_prev"], vpc, p["W"])
        o = ob.attend(p["q"], p["k"], vc, S, Z, p["W"], p["gate"], merge)
        _close(o, np.broadcast_to(c, o.shape))



def check_separate_query_key_maps(ob):
    """A state built with a key map Wk and read with a query map Wq equals
    the token-by-token sum with weights phi_Wq(q) . phi_Wk(k_t), both
    merges; and it differs from using either map for both."""
    p = _rand_problem(19, N=9)
    g = np.random.default_rng(19)
    Wk = g.standard_normal(p["W"].shape) / np.sqrt(p["W"].shape[1])
    S, Z = ob.prefill(p["k_prev"], p["v_prev"], Wk)
    for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
        o = ob.attend(p["q"], p["k"], p["v"], S, Z, p["W"], p["gate"], merge)
        ref = ob.attend_bruteforce(p["q"], p["k"], p["v"], p["k_prev"], p["v_prev"], p["W"],
                                   p["gate"], merge, Wk=Wk)
        _close(o, ref, rtol=1e-10, atol=1e-12)
        same = ob.attend_bruteforce(p["q"], p["k"], p["v"], p["k_prev"], p["v_prev"], p["W"],
                                    p["gate"], merge)
        assert np.abs(o - same).max() > 1e-3


# --------------------------------------------------- softmax-over-KV comparison

def check_softmax_kv_vs_sdpa(ob):
    p = _rand_problem(14, N=11)
    o = ob.softmax_kv_attend(p["k_prev"], p["v_prev"], p["q"], p["k"], p["v"])
    ref = _sdpa(p["q"], np.concatenate([p["k_prev"], p["k"]]),
                np.concatenate([p["v_prev"], p["v"]]))
    _close(o, ref, rtol=1e-10)


def check_softmax_kv_empty_prefix(ob):
    p = _rand_problem(15)
    H, d, f = p["W"].shape
    empty = np.zeros((0, H, d))
    o = ob.softmax_kv_attend(empty, empty, p["q"], p["k"], p["v"])
    _close(o, _sdpa(p["q"], p["k"], p["v"]), rtol=1e-10)



def _paged_problem(seed, P=11, p=4, n_junk=3):
    """A request's P cached tokens cut into pages of p slots, the pages put at
    shuffled positions of a pool that also holds unused pages. Unused pages
    and the slots past token P - 1 hold NaN, so reading any of them shows."""
    g = np.random.default_rng(seed)
    prob = _rand_problem(seed, N=P)
    H, d = prob["q"].shape[1:]
    n_pages = -(-P // p)
    order = g.permutation(n_pages + n_junk)
    page_ids = order[:n_pages]
    k_pages = np.full((n_pages + n_junk, p, H, d), np.nan)
    v_pages = np.full((n_pages + n_junk, p, H, d), np.nan)
    for t in range(P):
        k_pages[page_ids[t // p], t % p] = prob["k_prev"][t]
        v_pages[page_ids[t // p], t % p] = prob["v_prev"][t]
    return prob, k_pages, v_pages, page_ids


def check_paged_gather_layout(ob):
    """Token t of a request is slot t mod p of its (t // p)-th page: the
    gather puts the scattered tokens back in order, exactly."""
    prob, k_pages, v_pages, page_ids = _paged_problem(16)
    P = prob["k_prev"].shape[0]
    np.testing.assert_array_equal(ob.gather_pages(k_pages, page_ids, P), prob["k_prev"])
    np.testing.assert_array_equal(ob.gather_pages(v_pages, page_ids, P), prob["v_prev"])
    assert ob.gather_pages(k_pages, page_ids, 0).shape == (0,) + k_pages.shape[2:]


def check_paged_softmax_kv_vs_sdpa(ob):
    """Over a shuffled page pool with NaN in every unused slot, the paged
    comparison equals torch's fp64 scaled_dot_product_attention over the
    request's tokens in order followed by its block; with an empty prefix it
    is attention within the block alone."""
    for P, p in ((11, 4), (8, 4), (1, 3), (0, 4)):
        prob, k_pages, v_pages, page_ids = _paged_problem(17 + P, P=P, p=p)
        o = ob.softmax_kv_attend_paged(k_pages, v_pages, page_ids, P, prob["q"], prob["k"],
                                       prob["v"])
        ref = _sdpa(prob["q"], np.concatenate([prob["k_prev"], prob["k"]]),
                    np.concatenate([prob["v_prev"], prob["v"]]))
        _close(o, ref, rtol=1e-10)


# ------------------------------------------------- prompt with outputs (N1)

def _prompt_problem(seed, T=12, L=4, H=2, d=6, f=2, N0=5):
    g = np.random.default_rng(seed)
    return dict(
        q=g.standard_normal((T, H, d)), k=g.standard_normal((T, H, d)),
        v=g.standard_normal((T, H, d)), k0=g.standard_normal((N0, H, d)),
        v0=g.standard_normal((N0, H, d)), W=g.standard_normal((H, d, f)) / np.sqrt(d),
        gate=g.standard_normal(H), L=L)


def check_prefill_attend_vs_bruteforce(ob):
    """Block j of a prompt attends to exactly the tokens before it: each
    block's output equals the state-free token-by-token formulation over
    the earlier tokens (and an earlier context, when one is given), and the
    final state equals the plain sum over every token, built here from
    outer products of phi(k_t) and v_t."""
    p = _prompt_problem(7)
    L = p["L"]
    for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
        for with_context in (False, True):
            if with_context:
                S0, Z0 = ob.prefill(p["k0"], p["v0"], p["W"])
                kc, vc = p["k0"], p["v0"]
            else:
                S0 = Z0 = None
                kc, vc = p["k0"][:0], p["v0"][:0]
            o, S, Z = ob.prefill_attend(p["q"], p["k"], p["v"], p["W"], p["gate"], L, merge,
                                        S0=S0, Z0=Z0)
            for j0 in range(0, p["q"].shape[0], L):
                blk = slice(j0, j0 + L)
                ref = ob.attend_bruteforce(p["q"][blk], p["k"][blk], p["v"][blk],
                                           np.concatenate([kc, p["k"][:j0]]),
                                           np.concatenate([vc, p["v"][:j0]]), p["W"], p["gate"],
                                           merge)
                _close(o[blk], ref, rtol=1e-10, atol=1e-12)
            K = np.concatenate([kc, p["k"]])
            V = np.concatenate([vc, p["v"]])
            H = p["W"].shape[0]
            for h in range(H):
                S_ref = sum(np.outer(ob.feature_map(K[t, h], p["W"][h]), V[t, h])
                            for t in range(K.shape[0]))
                Z_ref = sum(ob.feature_map(K[t, h], p["W"][h]) for t in range(K.shape[0]))
                _close(S[h], S_ref, rtol=1e-10, atol=1e-12)
                _close(Z[h], Z_ref, rtol=1e-10, atol=1e-12)


def check_prefill_attend_first_block_is_softmax(ob):
    """With nothing committed before it, the first block of a prompt is plain
    softmax attention within the block (SHARED_NORM, any gate): torch's fp64
    scaled_dot_product_attention."""
    p = _prompt_problem(8)
    L = p["L"]
    o, _, _ = ob.prefill_attend(p["q"], p["k"], p["v"], p["W"], p["gate"], L,
                                ob.MERGE_SHARED_NORM)
    _close(o[:L], _sdpa(p["q"][:L], p["k"][:L], p["v"][:L]), rtol=1e-10, atol=1e-12)


# ------------------------------------ grouped-query heads, separate key map

def _gqa_problem(seed, L=5, H=4, H_kv=2, d=6, f=2, N=7):
    g = np.random.default_rng(seed)
    return dict(
        q=g.standard_normal((L, H, d)), k=g.standard_normal((L, H_kv, d)),
        v=g.standard_normal((L, H_kv, d)), k_prev=g.standard_normal((N, H_kv, d)),
        v_prev=g.standard_normal((N, H_kv, d)), Wq=g.standard_normal((H, d, f)) / np.sqrt(d),
        Wk=g.standard_normal((H_kv, d, f)) / np.sqrt(d), gate=g.standard_normal(H))


def check_gqa_reduces_to_repeated_heads(ob):
    """Grouped-query attention with H_kv key/value heads is ordinary
    attention after each key/value head (its k, v and state) is repeated for
    the H / H_kv consecutive query heads of its group (numpy's repeat along
    the head axis); with H_kv = H it is attend itself."""
    p = _gqa_problem(31)
    G = p["q"].shape[1] // p["k"].shape[1]
    S, Z = ob.prefill(p["k_prev"], p["v_prev"], p["Wk"])
    rep = lambda x, axis: np.repeat(x, G, axis=axis)  # noqa: E731
    for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
        o = ob.attend_gqa(p["q"], p["k"], p["v"], S, Z, p["Wq"], p["gate"], merge)
        ref = ob.attend(p["q"], rep(p["k"], 1), rep(p["v"], 1), rep(S, 0), rep(Z, 0), p["Wq"],
                        p["gate"], merge)
        _close(o, ref)
        # one key/value head per query head: nothing is grouped
        S4, Z4 = ob.prefill(rep(p["k_prev"], 1), rep(p["v_prev"], 1), rep(p["Wk"], 0))
        o4 = ob.attend_gqa(p["q"], rep(p["k"], 1), rep(p["v"], 1), S4, Z4, p["Wq"], p["gate"],
                           merge)
        _close(o4, ob.attend(p["q"], rep(p["k"], 1), rep(p["v"], 1), S4, Z4, p["Wq"], p["gate"],
                             merge))


def check_gqa_vs_bruteforce(ob):
    """Query head h of a group reads the state its key/value head g = h // G
    built with the key map: its output is the token-by-token sum with
    weights phi_Wq[h](q) . phi_Wk[g](k_t) over g's committed tokens."""
    p = _gqa_problem(32)
    H, H_kv = p["q"].shape[1], p["k"].shape[1]
    G = H // H_kv
    S, Z = ob.prefill(p["k_prev"], p["v_prev"], p["Wk"])
    for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
        o = ob.attend_gqa(p["q"], p["k"], p["v"], S, Z, p["Wq"], p["gate"], merge)
        for h in range(H):
            g = h // G
            ref = ob.attend_bruteforce(p["q"][:, h:h + 1], p["k"][:, g:g + 1], p["v"][:, g:g + 1],
                                       p["k_prev"][:, g:g + 1], p["v_prev"][:, g:g + 1],
                                       p["Wq"][h:h + 1], p["gate"][h:h + 1], merge,
                                       Wk=p["Wk"][g:g + 1])
            _close(o[:, h:h + 1], ref, rtol=1e-10, atol=1e-12)


def check_prefill_attend_state_free_of_block_length(ob):
    """The state a prompt leaves is the plain sum over its tokens with the key
    map, whatever block length cuts it (1, 2, 3, 4, 6 or 12 tokens per
    block), with a separate key map and with grouped heads."""
    g = np.random.default_rng(33)
    T, H, H_kv, d, f = 12, 4, 2, 6, 2
    q = g.standard_normal((T, H, d))
    k, v = g.standard_normal((T, H_kv, d)), g.standard_normal((T, H_kv, d))
    Wq = g.standard_normal((H, d, f)) / np.sqrt(d)
    Wk = g.standard_normal((H_kv, d, f)) / np.sqrt(d)
    gate = g.standard_normal(H)
    for L in (1, 2, 3, 4, 6, 12):
        _, S, Z = ob.prefill_attend(q, k, v, Wq, gate, L, Wk=Wk)
        for h in range(H_kv):
            S_ref = sum(np.outer(ob.feature_map(k[t, h], Wk[h]), v[t, h]) for t in range(T))
            Z_ref = sum(ob.feature_map(k[t, h], Wk[h]) for t in range(T))
            _close(S[h], S_ref, rtol=1e-10, atol=1e-12)
            _close(Z[h], Z_ref, rtol=1e-10, atol=1e-12)


def check_prefill_attend_gqa_vs_bruteforce(ob):
    """A prompt with grouped heads and separate maps: block j of query head h
    attends to exactly the tokens before it of key/value head h // G, through
    phi_Wq[h] . phi_Wk[h // G]."""
    g = np.random.default_rng(34)
    T, L, H, H_kv, d, f = 8, 4, 4, 2, 6, 2
    q = g.standard_normal((T, H, d))
    k, v = g.standard_normal((T, H_kv, d)), g.standard_normal((T, H_kv, d))
    Wq = g.standard_normal((H, d, f)) / np.sqrt(d)
    Wk = g.standard_normal((H_kv, d, f)) / np.sqrt(d)
    gate = g.standard_normal(H)
    G = H // H_kv
    for merge in (ob.MERGE_SHARED_NORM, ob.MERGE_CONVEX):
        o, _, _ = ob.prefill_attend(q, k, v, Wq, gate, L, merge, Wk=Wk)
        for j0 in range(0, T, L):
            blk = slice(j0, j0 + L)
            for h in range(H):
                gg = h // G
                ref = ob.attend_bruteforce(q[blk, h:h + 1], k[blk, gg:gg + 1], v[blk, gg:gg + 1],
                                           k[:j0, gg:gg + 1], v[:j0, gg:gg + 1], Wq[h:h + 1],
                                           gate[h:h + 1], merge, Wk=Wk[gg:gg + 1])
                _close(o[blk, h:h + 1], ref, rtol=1e-10, atol=1e-12)


ALL_CHECKS = [
    check_feature_map_golden,
    check_feature_map_vs_scipy,
    check_feature_map_invariants,
    check_commit_golden,
    check_commit_chunking,
    check_commit_sum_invariants,
    check_commit_outer_products,
    check_merge_golden,
    check_empty_state_is_softmax_attention,
    check_convex_soft_limit,
    check_state_vs_bruteforce,
    check_pure_linear_limits,
    check_block_permutation,
    check_convex_combination,
    check_separate_query_key_maps,
    check_softmax_kv_vs_sdpa,
    check_softmax_kv_empty_prefix,
    check_paged_gather_layout,
    check_paged_softmax_kv_vs_sdpa,
    check_prefill_attend_vs_bruteforce,
    check_prefill_attend_first_block_is_softmax,
    check_gqa_reduces_to_repeated_heads,
    check_gqa_vs_bruteforce,
    check_prefill_attend_state_free_of_block_length,
    check_prefill_attend_gqa_vs_bruteforce,
]

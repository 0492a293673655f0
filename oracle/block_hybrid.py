"""Plain fp64 reference of block-hybrid attention (test infrastructure only).

This module is the oracle that the CUDA library is checked against. It is slow
on purpose: every function writes the defining formula out with numpy
float64 arrays and library primitives (matrix products, ``exp``), with no
blocking, fusion, reordering or numerical tricks beyond what the definition
states. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import it; the product path never does.

Sources (web pages about arXiv 2608.06628, "Retrofitting Linear Attention into
Diffusion Language Models", Kim, Roh and Kim):

* [GIST] gist.science explainer of the paper, section "Technical Summary",
  sub-section "Methodology: Block-Hybrid Attention / Architecture Design"
  (its four bullets: within-block, cross-block, state compression, merging).
* [PITH] pith.science referee report on the paper: "The reading / What
  carries the argument" (the sums S_n and Z_n and the O(Fd) read) and
  "Referee Report / minor comments", the comment on the Section 3.1 out(q)
  equation (where the learned gate sits in the merge).
* [ABS] the arXiv abstract, as reproduced on mlsanity.com.

Notation (one attention head): d = head dimension, f = width of one softmax
half of the feature map, F = 2f, L = tokens in the active block, N = committed
tokens. Per-request layouts mirror the library's: activations ``[L, H, d]``,
``W`` ``[H, d, f]``, ``S`` ``[H, F, d]``, ``Z`` ``[H, F]``, gate logits ``[H]``.

Readings of points the pages leave open (each one is also listed in the
design notes):

* Softmax scale inside the block: 1/sqrt(d) unless the caller passes one.
* The feature map applies softmax to the raw product x W (no temperature).
  The positive half comes first, then the negated half.
* One W per head serves both queries and keys.
* SHARED_NORM merge (the pages' own form, [GIST] merging bullet and [PITH]
  out(q) comment): w = sigmoid(alpha_h) scales only the softmax branch's
  numerator and denominator; the linear branch is unweighted, and both share
  one normaliser:
      o = (w * sum_j e^{s_ij} v_j + phi(q_i)^T S) / (w * sum_j e^{s_ij} + phi(q_i)^T Z)
  with the exponentials unshifted (the form is not shift-invariant).
* CONVEX merge (the alternative form the specification of this library
  fixes): o = sigmoid(g_h) * o_soft + (1 - sigmoid(g_h)) * o_lin, with
  o_soft = softmax attention within the block and
  o_lin = phi(q)^T S / phi(q)^T Z. With nothing committed (Z = 0) the linear
  branch is undefined and is dropped: o = o_soft.
* The prompt counts as committed context; ingesting it is the same sum as
  committing blocks (the sums are plain sums, so chunking does not matter).
"""

from __future__ import annotations

import numpy as np

MERGE_SHARED_NORM = 0
MERGE_CONVEX = 1

# exp() of fp64 overflows above ~709.78; the literal (unshifted) definition
# used here is only valid while every block score stays well below that.
_EXP_LIMIT = 700.0


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def sigmoid(g):
    """Logistic function 1 / (1 + e^{-g}), evaluated without overflow for
    any g including +-inf."""
    g = _f64(g)
    out = np.empty_like(g)
    pos = g >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-g[pos]))
    e = np.exp(g[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def _softmax_last(u: np.ndarray) -> np.ndarray:
    """Softmax over the last axis. Subtracting the row maximum is an exact
    identity of softmax and only keeps exp() in range."""
    e = np.exp(u - u.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def feature_map(x, W) -> np.ndarray:
    """Hedgehog feature map of one head, [GIST] cross-block bullet and
    [PITH] "What carries the argument":

        phi(x) = [softmax(x W), softmax(-x W)]

    x: [..., d]; W: [d, f]. Returns [..., 2f]: the softmax of u = x W over
    its f entries, followed by the softmax of -u.
    """
    x = _f64(x)
    W = _f64(W)
    u = x @ W
    return np.concatenate([_softmax_last(u), _softmax_last(-u)], axis=-1)


def feature_map_heads(x, W) -> np.ndarray:
    """phi for every head: x [n, H, d], W [H, d, f] -> [n, H, 2f]."""
    x = _f64(x)
    W = _f64(W)
    H = W.shape[0]
    return np.stack([feature_map(x[:, h, :], W[h]) for h in range(H)], axis=1)


def commit(S, Z, k, v, W):
    """Fold one finished block into the recurrent state, [GIST] state
    compression bullet and [PITH] "What carries the argument":

        S_n = S_{n-1} + sum_{t in B_n} phi(k_t) v_t^T      ([F, d] per head)
        Z_n = Z_{n-1} + sum_{t in B_n} phi(k_t)            ([F] per head)

    S [H, F, d], Z [H, F], k/v [T, H, d], W [H, d, f]. Returns new (S, Z);
    the inputs are left untouched. T may be any length (a block, a prompt).
    """
    S = _f64(S).copy()
    Z = _f64(Z).copy()
    k = _f64(k)
    v = _f64(v)
    W = _f64(W)
    for h in range(W.shape[0]):
        phi_k = feature_map(k[:, h, :], W[h])  # [T, F]
        S[h] += phi_k.T @ v[:, h, :]  # sum_t phi(k_t) v_t^T
        Z[h] += phi_k.sum(axis=0)  # sum_t phi(k_t)
    return S, Z


def prefill(k, v, W):
    """State of a prompt taken as committed context: the commit sums started
    from zero over all prompt tokens. k/v [T, H, d]; returns (S, Z)."""
    W = _f64(W)
    H, d, f = W.shape
    S0 = np.zeros((H, 2 * f, d))
    Z0 = np.zeros((H, 2 * f))
    return commit(S0, Z0, k, v, W)


def _scale(d: int, scale) -> float:
    return 1.0 / np.sqrt(d) if (scale is None or scale == 0) else float(scale)


def attend(q, k, v, S, Z, W, gate, merge: int = MERGE_SHARED_NORM, scale=None):
    """Block-hybrid attention for the active block of one request.

    Every query i of the active block gets (per head):
      * an exact bidirectional softmax branch over the L tokens of the block
        ([GIST] within-block bullet; no mask):
            s_ij = scale * q_i . k_j,  sm_num_i = sum_j e^{s_ij} v_j,
            sm_den_i = sum_j e^{s_ij};
      * a linear branch that reads the fixed-size state ([GIST] cross-block
        and state-compression bullets, [PITH] O(Fd) read):
            num_i = phi(q_i)^T S,  den_i = phi(q_i)^T Z;
      * the gated merge (module docstring: SHARED_NORM or CONVEX).

    q/k/v [L, H, d]; S [H, F, d]; Z [H, F]; W [H, d, f]; gate [H] logits.
    Returns o [L, H, d] in float64.
    """
    q, k, v, S, Z, W = (_f64(a) for a in (q, k, v, S, Z, W))
    gate = _f64(gate)
    L, H, d = q.shape
    sc = _scale(d, scale)
    w = sigmoid(gate)
    o = np.empty((L, H, d))
    for h in range(H):
        s = sc * (q[:, h, :] @ k[:, h, :].T)  # [L queries, L keys]
        if np.abs(s).max(initial=0.0) > _EXP_LIMIT:
            raise ValueError("block scores outside the fp64 exp range")
        e = np.exp(s)
        sm_num = e @ v[:, h, :]  # [L, d]
        sm_den = e.sum(axis=1)  # [L]
        phi_q = feature_map(q[:, h, :], W[h])  # [L, F]
        num = phi_q @ S[h]  # [L, d]
        den = phi_q @ Z[h]  # [L]
        if merge == MERGE_SHARED_NORM:
            o[:, h, :] = (w[h] * sm_num + num) / (w[h] * sm_den + den)[:, None]
        elif merge == MERGE_CONVEX:
            o_soft = sm_num / sm_den[:, None]
            o_h = o_soft.copy()
            has = den > 0
            o_lin = num[has] / den[has][:, None]
            o_h[has] = w[h] * o_soft[has] + (1.0 - w[h]) * o_lin
            o[:, h, :] = o_h
        else:
            raise ValueError(f"unknown merge mode {merge}")
    return o


def attend_bruteforce(q, k, v, k_prev, v_prev, W, gate,
                      merge: int = MERGE_SHARED_NORM, scale=None, Wk=None):
    """Second, state-free formulation of ``attend`` used to cross-check it.

    By the kernel identity phi(q)^T (sum_t phi(k_t) v_t^T) =
    sum_t (phi(q) . phi(k_t)) v_t^T, the linear branch is a weighted sum over
    the committed tokens themselves with weights a_t = phi(q) . phi(k_t).
    This function evaluates that sum token by token and never forms S or Z.
    k_prev/v_prev [N, H, d] are all committed tokens (N may be 0).
    With ``Wk`` given, the committed keys take that feature map and the
    queries ``W`` (separate query and key maps; the pages speak of the
    feature map matrices W of a layer without saying whether queries and
    keys share one); by default one map serves both.
    """
    q, k, v, k_prev, v_prev, W = (_f64(a) for a in (q, k, v, k_prev, v_prev, W))
    Wk = W if Wk is None else _f64(Wk)
    gate = _f64(gate)
    L, H, d = q.shape
    N = k_prev.shape[0]
    sc = _scale(d, scale)
    w = sigmoid(gate)
    o = np.empty((L, H, d))
    for h in range(H):
        for i in range(L):
            phi_q = feature_map(q[i, h, :], W[h])
            blk_w = np.array([np.exp(sc * np.dot(q[i, h, :], k[j, h, :])) for j in range(L)])
            lin_w = np.array([np.dot(phi_q, feature_map(k_prev[t, h, :], Wk[h])) for t in range(N)])
            blk_num = sum(blk_w[j] * v[j, h, :] for j in range(L))
            blk_den = blk_w.sum()
            lin_num = sum((lin_w[t] * v_prev[t, h, :] for t in range(N)), np.zeros(d))
            lin_den = lin_w.sum()
            if merge == MERGE_SHARED_NORM:
                o[i, h, :] = (w[h] * blk_num + lin_num) / (w[h] * blk_den + lin_den)
            else:
                o_soft = blk_num / blk_den
                if lin_den > 0:
                    o[i, h, :] = w[h] * o_soft + (1.0 - w[h]) * (lin_num / lin_den)
                else:
                    o[i, h, :] = o_soft
    return o


def kv_head(h: int, H: int, H_kv: int) -> int:
    """The key/value head that query head h reads under grouped-query
    attention: query heads come in H_kv consecutive groups of H / H_kv, and
    group g shares key/value head g. The pages do not speak of head counts
    (the specification's layers have H_kv = H); this is the usual grouping,
    in which a layer with fewer key/value heads stores one state per
    key/value head."""
    if H % H_kv != 0:
        raise ValueError("the number of key/value heads must divide the number of query heads")
    return h // (H // H_kv)


def attend_gqa(q, k, v, S, Z, Wq, gate, merge: int = MERGE_SHARED_NORM, scale=None):
    """``attend`` with grouped query heads: every query head h is ``attend``
    of that one head against key/value head g = kv_head(h, H, H_kv), that is
    the block's keys and values of head g and the state (S, Z) of head g,
    with its own query map Wq[h] and gate[h].

    q [L, H, d], Wq [H, d, f], gate [H]; k/v [L, H_kv, d], S [H_kv, F, d],
    Z [H_kv, F]. Returns o [L, H, d] in float64.
    """
    q, k, v, S, Z, Wq = (_f64(a) for a in (q, k, v, S, Z, Wq))
    gate = _f64(gate)
    L, H, d = q.shape
    H_kv = k.shape[1]
    o = np.empty((L, H, d))
    for h in range(H):
        g = kv_head(h, H, H_kv)
        o[:, h:h + 1, :] = attend(q[:, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], S[g:g + 1],
                                  Z[g:g + 1], Wq[h:h + 1], gate[h:h + 1], merge, scale)
    return o


def prefill_attend(q, k, v, W, gate, L: int, merge: int = MERGE_SHARED_NORM, scale=None,
                   S0=None, Z0=None, Wk=None):
    """A prompt processed block by block with block-hybrid attention, so that
    every prompt token gets its output ([GIST] "Methodology: Block-Hybrid
    Attention / Architecture Design": exact softmax inside the active block,
    linear attention over the committed blocks through S and Z, which change
    only when a block is committed).

    Reading taken: the prompt q/k/v [T, H, d] (T a multiple of L) is a
    sequence of T / L blocks; block j is the active block, attending to the
    state of blocks 0 .. j-1 (added to the initial state S0, Z0, zero when
    omitted), and is then committed. The pages run this form when the layers
    are trained against their softmax teacher ([GIST] "Retrofitting
    Strategy", stage 1) and give no other prefill formula.

    With ``Wk`` given, W is the query map and Wk the key map (the state is
    built with Wk); k/v may then have H_kv < H heads (grouped-query
    attention, ``attend_gqa``), with Wk [H_kv, d, f] and the state per
    key/value head.

    Returns (o [T, H, d], S [H_kv, F, d], Z [H_kv, F]) in float64.
    """
    q, k, v, W = (_f64(a) for a in (q, k, v, W))
    Wk = W if Wk is None else _f64(Wk)
    T, H, d = q.shape
    H_kv = k.shape[1]
    if T % L != 0:
        raise ValueError("prompt length must be a multiple of the block length")
    f = W.shape[2]
    S = np.zeros((H_kv, 2 * f, d)) if S0 is None else _f64(S0).copy()
    Z = np.zeros((H_kv, 2 * f)) if Z0 is None else _f64(Z0).copy()
    o = np.empty((T, H, d))
    for j0 in range(0, T, L):
        blk = slice(j0, j0 + L)
        if H_kv == H:
            o[blk] = attend(q[blk], k[blk], v[blk], S, Z, W, gate, merge, scale)
        else:
            o[blk] = attend_gqa(q[blk], k[blk], v[blk], S, Z, W, gate, merge, scale)
        S, Z = commit(S, Z, k[blk], v[blk], Wk)
    return o, S, Z


def softmax_kv_attend(k_prefix, v_prefix, q, k, v, scale=None):
    """Full-prefix softmax attention of the active block over a KV cache, the
    cost the method removes ([ABS]: each denoising step attends to all
    previous blocks; [GIST] problem statement). Comparison path only.

    Each query attends, without a mask, to the P cached keys followed by the
    L keys of the active block:
        o_i = sum_j softmax_j(scale * q_i . k_j) v_j,  j over prefix and block.
    k_prefix/v_prefix [P, H, d] (P may be 0); q/k/v [L, H, d].
    """
    k_prefix, v_prefix, q, k, v = (_f64(a) for a in (k_prefix, v_prefix, q, k, v))
    L, H, d = q.shape
    sc = _scale(d, scale)
    K = np.concatenate([k_prefix, k], axis=0)
    V = np.concatenate([v_prefix, v], axis=0)
    o = np.empty((L, H, d))
    for h in range(H):
        s = sc * (q[:, h, :] @ K[:, h, :].T)  # [L, P+L]
        p = _softmax_last(s)
        o[:, h, :] = p @ V[:, h, :]
    return o


def gather_pages(pages, page_ids, P):
    """The first P tokens of one request from a paged cache, in token order.

    A paged cache stores a request's tokens in fixed-size pages drawn from a
    shared pool (PagedAttention, Kwon et al., SOSP 2023); [GIST] "Key
    Contributions", implementation bullet: the method's serving kernel keeps
    the fixed-size state next to such paged KV caches. Token t of the request
    sits in slot t mod p of page page_ids[t // p], where p is the page size.
    pages [num_pages, p, H, d]; page_ids lists the request's pages in order.
    Slots past token P - 1 are never read.
    """
    pages = _f64(pages)
    p = pages.shape[1]
    rows = [pages[int(page_ids[t // p]), t % p] for t in range(int(P))]
    if not rows:
        return np.zeros((0,) + pages.shape[2:])
    return np.stack(rows)


def softmax_kv_attend_paged(k_pages, v_pages, page_ids, P, q, k, v, scale=None):
    """softmax_kv_attend over a paged KV cache: the request's P cached keys
    and values are gathered from their pages (gather_pages), then the
    comparison softmax is applied to them and the active block unchanged."""
    return softmax_kv_attend(gather_pages(k_pages, page_ids, P),
                             gather_pages(v_pages, page_ids, P), q, k, v, scale)

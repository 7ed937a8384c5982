"""Plain fp64 restatement of Hedgehog / Taylor causal linear attention.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.  All arithmetic is float64; inputs are promoted exactly
from whatever precision the caller holds (bf16-rounded values are exactly
representable in float64).

Sources (page title, then section / equation):

* "The Hedgehog & the Porcupine: Expressive Linear Attentions with Softmax
  Mimicry" (paper-graph-ui summary of arXiv 2402.04347), referred to below as
  *HH summary*; and the paperlayer.ai summary of the same paper, *HH digest*.

Readings taken where the pages are silent or inconsistent:

* W orientation: ``h = x @ W + b`` with ``W[k][l]`` = input k -> output l, so
  the direction w_l of Choice 1 is column l of W.
* The negated half negates the bias too: ``exp(-(xW + b))`` (Choice 3 writes
  ``exp(-w.x - b)``); the positive block comes first.
* No 1/sqrt(d) or temperature inside phi; 1/sqrt(d) only in the softmax
  target of the distillation loss.
* Causal sums include the diagonal (j <= i).
* Taylor map: ``[1, x, (x_i x_j / sqrt2) for i, j in [d]]`` with the pair
  index i-major; the 1/sqrt2 makes phi(q).phi(k) = 1 + q.k + (q.k)^2 / 2.
* Natural logarithm in the loss; the per-head result is the sum over queries.
* Softmax-over-features map (Choice 4, Eq. 5): the printed equation
  normalises exp(w_l . x) over the d learned directions and drops the bias.
  Choice 3's negation block is kept as in practice, each half normalised over
  its own d directions: phi = [softmax(x W), softmax(-x W)] (2d features).
* Entropies use the natural logarithm with 0 log 0 = 0; KL = CE - H(p).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "hedgehog_feature_map",
    "hedgehog_softmax_feature_map",
    "taylor2_feature_map",
    "taylor2_feature_dim",
    "feature_map",
    "causal_weights",
    "linattn_quadratic",
    "linattn_rows",
    "linattn_recurrent",
    "decode_step",
    "softmax_target",
    "mimicry_loss",
    "mimicry_loss_rows",
    "fwd_causal",
    "loss_causal",
    "mimicry_loss_grad",
    "loss_grad_causal",
    "attention_entropy",
    "mimicry_stats",
    "stats_causal",
]


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# Feature maps
# ---------------------------------------------------------------------------

def hedgehog_feature_map(x, W, b) -> np.ndarray:
    """Hedgehog single-layer MLP map with the negation block.

    HH summary, "The Hedgehog MLP Feature Map": Choice 1 (element-wise
    exponential of a learned affine map) and Choice 3 (negation mapping
    R^d -> R^2d).  ``x``: [..., d]; ``W``: [d, d] (input-major); ``b``: [d].
    Returns [..., 2d] = [exp(h), exp(-h)] with h = x W + b.
    """
    x, W, b = _f64(x), _f64(W), _f64(b)
    h = x @ W + b
    return np.concatenate([np.exp(h), np.exp(-h)], axis=-1)


def hedgehog_softmax_feature_map(x, W) -> np.ndarray:
    """Softmax-over-features Hedgehog map, no bias.

    HH summary, "The Hedgehog MLP Feature Map", Choice 4 (Eq. 5): feature l
    is exp(w_l . x) / sum_i exp(w_i . x) over the d learned directions (the
    columns of W); with the negation block of Choice 3 the second half is the
    same normalisation of exp(-w_l . x).  Returns [..., 2d]
    = [softmax(x W), softmax(-x W)], each half summing to one.
    """
    x, W = _f64(x), _f64(W)
    h = x @ W
    pos = np.exp(h)
    neg = np.exp(-h)
    pos = pos / pos.sum(axis=-1, keepdims=True)
    neg = neg / neg.sum(axis=-1, keepdims=True)
    return np.concatenate([pos, neg], axis=-1)


def taylor2_feature_dim(d: int) -> int:
    """d' = 1 + d + d^2 (HH summary, "The Taylor Exponential as a Bridge Result")."""
    return 1 + d + d * d


def taylor2_feature_map(x) -> np.ndarray:
    """Degree-2 Taylor map [1, x, vec(x x^T) / sqrt 2], pair index i-major.

    HH summary, "The Taylor Exponential as a Bridge Result" (the feature
    construction for 1 + q.k + (q.k)^2/2).  ``x``: [..., d] -> [..., 1+d+d^2].
    """
    x = _f64(x)
    d = x.shape[-1]
    one = np.ones(x.shape[:-1] + (1,), dtype=np.float64)
    outer = (x[..., :, None] * x[..., None, :]).reshape(x.shape[:-1] + (d * d,))
    return np.concatenate([one, x, outer / math.sqrt(2.0)], axis=-1)


def feature_map(kind: str, x, W=None, b=None) -> np.ndarray:
    """Dispatch on the map name: ``"hedgehog"``, ``"hedgehog_softmax"`` (b unused)
    or ``"taylor2"``."""
    if kind == "hedgehog":
        return hedgehog_feature_map(x, W, b)
    if kind == "hedgehog_softmax":
        return hedgehog_softmax_feature_map(x, W)
    if kind == "taylor2":
        return taylor2_feature_map(x)
    raise ValueError(f"unknown feature map {kind!r}")


# ---------------------------------------------------------------------------
# Causal linear attention
# ---------------------------------------------------------------------------

def causal_weights(phi_q, phi_k) -> np.ndarray:
    """Row-normalised linear-attention weights a_ij / sum_{m<=i} a_im, j <= i.

    HH summary, "2. Context and Motivation" (the kernel form, paper Eq. 2): the unnormalised
    weight of key j for query i is phi(q_i) . phi(k_j); entries above the
    diagonal are zero.  ``phi_q``, ``phi_k``: [n, d'] -> [n, n].
    """
    a = _f64(phi_q) @ _f64(phi_k).T
    a = np.tril(a)
    return a / a.sum(axis=-1, keepdims=True)


def linattn_quadratic(phi_q, phi_k, v) -> np.ndarray:
    """Quadratic (brute-force) causal linear attention for one head.

    HH summary, "2. Context and Motivation" and "Complexity Analysis" (paper Eq. 2):
    y_i = sum_{j<=i} (phi(q_i).phi(k_j)) v_j / sum_{j<=i} phi(q_i).phi(k_j).
    ``phi_q``, ``phi_k``: [n, d']; ``v``: [n, d] -> y [n, d].
    """
    a = np.tril(_f64(phi_q) @ _f64(phi_k).T)
    return (a @ _f64(v)) / a.sum(axis=-1, keepdims=True)


def linattn_rows(phi_q, phi_k, v, rows) -> np.ndarray:
    """The same definition evaluated one query row at a time.

    For sampled checks on long sequences: row i needs phi_k[:i+1] and
    v[:i+1] only.  Returns [len(rows), d].
    """
    phi_q, phi_k, v = _f64(phi_q), _f64(phi_k), _f64(v)
    out = np.empty((len(rows), v.shape[-1]), dtype=np.float64)
    for r, i in enumerate(rows):
        a = phi_k[: i + 1] @ phi_q[i]
        out[r] = (a @ v[: i + 1]) / a.sum()
    return out


def decode_step(phi_q_t, phi_k_t, v_t, S, z):
    """One recurrent step: fold token t into the state, then read it out.

    HH summary, "Complexity Analysis": S_t = S_{t-1} + phi(k_t)^T v_t,
    z_t = z_{t-1} + phi(k_t), y_t = phi(q_t) S_t / (phi(q_t) . z_t).  The
    state after the step includes token t (the causal sum runs to j = i).
    ``S``: [d', d]; ``z``: [d'].  Returns (y_t, S_t, z_t); inputs unchanged.
    """
    phi_q_t, phi_k_t, v_t = _f64(phi_q_t), _f64(phi_k_t), _f64(v_t)
    S = _f64(S) + np.outer(phi_k_t, v_t)
    z = _f64(z) + phi_k_t
    y = (phi_q_t @ S) / (phi_q_t @ z)
    return y, S, z


def linattn_recurrent(phi_q, phi_k, v, S0=None, z0=None):
    """Recurrent causal linear attention over a whole sequence.

    Runs :func:`decode_step` token by token from state (S0, z0) (zeros by
    default).  Returns (y [n, d], S_n [d', d], z_n [d']).
    """
    phi_q, phi_k, v = _f64(phi_q), _f64(phi_k), _f64(v)
    n, dp = phi_k.shape
    d = v.shape[-1]
    S = np.zeros((dp, d)) if S0 is None else _f64(S0).copy()
    z = np.zeros(dp) if z0 is None else _f64(z0).copy()
    y = np.empty((n, d))
    for t in range(n):
        y[t], S, z = decode_step(phi_q[t], phi_k[t], v[t], S, z)
    return y, S, z


# ---------------------------------------------------------------------------
# Attention-weight distillation (mimicry) loss
# ---------------------------------------------------------------------------

def softmax_target(q, k) -> np.ndarray:
    """Causal softmax(q k^T / sqrt d) over j <= i, max-subtracted per row.

    HH summary, "The Attention Weight Distillation Loss" (paper Eq. 4, the
    target fraction).  ``q``, ``k``: [n, d] -> [n, n].
    """
    q, k = _f64(q), _f64(k)
    n, d = q.shape
    s = (q @ k.T) / math.sqrt(d)
    mask = np.tril(np.ones((n, n), dtype=bool))
    s = np.where(mask, s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    e = np.where(mask, np.exp(s), 0.0)
    return e / e.sum(axis=-1, keepdims=True)


def mimicry_loss(q, k, phi_q, phi_k) -> np.ndarray:
    """Per-query cross-entropy L_i of paper Eq. 4 for one head.

    HH summary, "The Attention Weight Distillation Loss":
    L_i = - sum_{j<=i} p_ij log( a_ij / sum_{m<=i} a_im ),
    p = causal softmax(q k^T / sqrt d), a_ij = phi(q_i).phi(k_j).
    Natural log.  Returns [n].
    """
    p = softmax_target(q, k)
    w = causal_weights(phi_q, phi_k)
    n = p.shape[0]
    out = np.empty(n)
    for i in range(n):
        out[i] = -np.sum(p[i, : i + 1] * np.log(w[i, : i + 1]))
    return out


def mimicry_loss_rows(q, k, phi_q, phi_k, rows) -> np.ndarray:
    """Eq. 4 evaluated for selected query rows only (sampled checks)."""
    q, k, phi_q, phi_k = _f64(q), _f64(k), _f64(phi_q), _f64(phi_k)
    d = q.shape[-1]
    out = np.empty(len(rows))
    for r, i in enumerate(rows):
        s = (k[: i + 1] @ q[i]) / math.sqrt(d)
        e = np.exp(s - s.max())
        p = e / e.sum()
        a = phi_k[: i + 1] @ phi_q[i]
        out[r] = -np.sum(p * np.log(a / a.sum()))
    return out


def mimicry_loss_grad(q, k, W, b, Wk=None, bk=None, kind="hedgehog", feature_rounding=None):
    """Gradient of sum_i L_i (paper Eq. 4, one head) w.r.t. the Hedgehog map.

    HH summary, "The Attention Weight Distillation Loss": only the feature-map
    MLPs are trained; q, k (and so the softmax target p) are frozen.  With
    h = xW + b, phi = [e^h; e^-h] ("The Hedgehog MLP Feature Map", Choices 1
    and 3), a_ij = phi(q_i).phi(k_j), A_i = sum_{j<=i} a_ij and
    L_i = ln A_i - sum_j p_ij ln a_ij, the chain rule gives
        g_ij = dL/da_ij = 1/A_i - p_ij / a_ij                (j <= i, else 0)
        dL/dphi(q_i) = sum_j g_ij phi(k_j),  dL/dphi(k_j) = sum_i g_ij phi(q_i)
        dL/dh = dL/dphi_+ * e^h - dL/dphi_- * e^-h
        dL/dW = sum_x x^T dL/dh(x),  dL/db = sum_x dL/dh(x)
    over the query rows (query map) and the key rows (key map).  Returns
    (dWq, dbq, dWk, dbk); with one shared map (Wk None) the gradient with
    respect to it is dWq + dWk, dbq + dbk.

    kind="hedgehog_softmax": the map of Choice 4 (Eq. 5), h = xW (no bias),
    phi = [softmax(h); softmax(-h)].  Only the step from dL/dphi to dL/dh
    changes: the Jacobian of s = softmax(u) maps an upstream gradient y to
    s * (y - <y, s>), and the negated half enters with a minus sign, so
        dL/dh = phi_+ * (dL/dphi_+ - <dL/dphi_+, phi_+>)
              - phi_- * (dL/dphi_- - <dL/dphi_-, phi_->).
    b and bk are ignored and dbq, dbk are returned as None.

    feature_rounding: None, or a function applied to phi(q) and phi(k) right
    after the map, so that every later step uses the rounded features (an
    error-budget experiment: rounding them to the storage precision of a
    kernel's operands); the arithmetic is otherwise unchanged.
    """
    q, k = _f64(q), _f64(k)
    d = q.shape[-1]
    soft = kind == "hedgehog_softmax"
    if not soft and kind != "hedgehog":
        raise ValueError(f"no parameters to differentiate for {kind!r}")
    Wq = _f64(W)
    Wk_ = Wq if Wk is None else _f64(Wk)
    if soft:
        pq = hedgehog_softmax_feature_map(q, Wq)
        pk = hedgehog_softmax_feature_map(k, Wk_)
    else:
        bq = _f64(b)
        bk_ = bq if Wk is None else _f64(bk)
        hq = q @ Wq + bq
        hk = k @ Wk_ + bk_
        pq = np.concatenate([np.exp(hq), np.exp(-hq)], axis=-1)
        pk = np.concatenate([np.exp(hk), np.exp(-hk)], axis=-1)
    if feature_rounding is not None:
        pq, pk = _f64(feature_rounding(pq)), _f64(feature_rounding(pk))
    n = q.shape[0]
    mask = np.tril(np.ones((n, n), dtype=bool))
    a = pq @ pk.T
    A = np.where(mask, a, 0.0).sum(axis=-1)
    p = softmax_target(q, k)
    g = np.where(mask, 1.0 / A[:, None] - p / np.where(mask, a, 1.0), 0.0)
    dpq = g @ pk
    dpk = g.T @ pq
    if soft:
        dhq = _softmax_vjp(dpq[:, :d], pq[:, :d]) - _softmax_vjp(dpq[:, d:], pq[:, d:])
        dhk = _softmax_vjp(dpk[:, :d], pk[:, :d]) - _softmax_vjp(dpk[:, d:], pk[:, d:])
        return q.T @ dhq, None, k.T @ dhk, None
    dhq = dpq[:, :d] * pq[:, :d] - dpq[:, d:] * pq[:, d:]
    dhk = dpk[:, :d] * pk[:, :d] - dpk[:, d:] * pk[:, d:]
    return q.T @ dhq, dhq.sum(axis=0), k.T @ dhk, dhk.sum(axis=0)


def _softmax_vjp(y, s) -> np.ndarray:
    """Row-wise vector-Jacobian product of softmax: s * (y - sum_l y_l s_l).

    s = softmax(u) over the last axis has ds_l/du_m = s_l (delta_lm - s_m),
    so sum_l y_l ds_l/du_m = s_m (y_m - <y, s>).
    """
    return s * (y - (y * s).sum(axis=-1, keepdims=True))


def attention_entropy(weights) -> np.ndarray:
    """Per-row entropy H(a_i) = -sum_{j<=i} a_ij log a_ij of causal weights.

    HH summary, "The Two Missing Properties as Design Specifications" (the
    spikiness measure: 0 for one-hot rows, log i for uniform rows).
    ``weights``: [n, n] row-normalised, zero above the diagonal; 0 log 0 = 0.
    """
    w = _f64(weights)
    n = w.shape[0]
    out = np.empty(n)
    for i in range(n):
        row = w[i, : i + 1]
        nz = row[row > 0]
        out[i] = -np.sum(nz * np.log(nz))
    return out


def mimicry_stats(q, k, phi_q, phi_k) -> np.ndarray:
    """Per-query [CE, KL, H(p), H(w)] for one head.

    CE is paper Eq. 4 (mimicry_loss); H(p) and H(w) are the entropies of the
    softmax target and of the linear-attention weights (spikiness, as above);
    KL(p || w) = CE - H(p), the divergence named next to the cross-entropy in
    the HH digest (section A.3, attention distillation).  Returns [n, 4].
    """
    p = softmax_target(q, k)
    w = causal_weights(phi_q, phi_k)
    ce = mimicry_loss(q, k, phi_q, phi_k)
    hp = attention_entropy(p)
    hw = attention_entropy(w)
    return np.stack([ce, ce - hp, hp, hw], axis=-1)


# ---------------------------------------------------------------------------
# Batched wrappers over [B, H, n, d] inputs (per-head maps W[H], b[H])
# ---------------------------------------------------------------------------

def _map_head(kind, x, W, b, h):
    if kind == "hedgehog":
        return hedgehog_feature_map(x, W[h], b[h])
    if kind == "hedgehog_softmax":
        return hedgehog_softmax_feature_map(x, W[h])
    return taylor2_feature_map(x)


def fwd_causal(kind, q, k, v, W=None, b=None):
    """Quadratic-form outputs y [B, H, n, d] for every (batch, head)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H = q.shape[:2]
    y = np.empty(v.shape, dtype=np.float64)
    for bi in range(B):
        for h in range(H):
            pq = _map_head(kind, q[bi, h], W, b, h)
            pk = _map_head(kind, k[bi, h], W, b, h)
            y[bi, h] = linattn_quadratic(pq, pk, v[bi, h])
    return y


def loss_causal(kind, q, k, W=None, b=None):
    """Per-row losses [B, H, n] and per-head sums [B, H]."""
    q, k = _f64(q), _f64(k)
    B, H, n = q.shape[:3]
    rows = np.empty((B, H, n))
    for bi in range(B):
        for h in range(H):
            pq = _map_head(kind, q[bi, h], W, b, h)
            pk = _map_head(kind, k[bi, h], W, b, h)
            rows[bi, h] = mimicry_loss(q[bi, h], k[bi, h], pq, pk)
    return rows, rows.sum(axis=-1)


def stats_causal(kind, q, k, W=None, b=None):
    """Per-row [CE, KL, H(p), H(w)] for every (batch, head): [B, H, n, 4]."""
    q, k = _f64(q), _f64(k)
    B, H, n = q.shape[:3]
    out = np.empty((B, H, n, 4))
    for bi in range(B):
        for h in range(H):
            pq = _map_head(kind, q[bi, h], W, b, h)
            pk = _map_head(kind, k[bi, h], W, b, h)
            out[bi, h] = mimicry_stats(q[bi, h], k[bi, h], pq, pk)
    return out


def loss_grad_causal(q, k, W, b, Wk=None, bk=None, kind="hedgehog", feature_rounding=None):
    """Gradient of the loss summed over [B, H, n] w.r.t. per-head maps.

    Returns (dWq [H, d, d], dbq [H, d], dWk, dbk), each summed over the batch.
    With one shared map (Wk None) dWk and dbk are None and the query and key
    sides are added into dWq, dbq.  kind="hedgehog_softmax" (no bias): the
    bias gradients are None.
    """
    q, k = _f64(q), _f64(k)
    B, H, n, d = q.shape
    soft = kind == "hedgehog_softmax"
    dWq = np.zeros((H, d, d))
    dbq = np.zeros((H, d))
    dWk = np.zeros((H, d, d))
    dbk = np.zeros((H, d))
    for bi in range(B):
        for h in range(H):
            g = mimicry_loss_grad(q[bi, h], k[bi, h], _f64(W)[h],
                                  None if soft else _f64(b)[h],
                                  None if Wk is None else _f64(Wk)[h],
                                  None if (bk is None or soft) else _f64(bk)[h], kind=kind,
                                  feature_rounding=feature_rounding)
            dWq[h] += g[0]
            dWk[h] += g[2]
            if not soft:
                dbq[h] += g[1]
                dbk[h] += g[3]
    if soft:
        dbq = dbk = None
    if Wk is None:
        return dWq + dWk, (None if soft else dbq + dbk), None, None
    return dWq, dbq, dWk, dbk

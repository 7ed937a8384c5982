"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Each check below ties the oracle to something other than itself: hand-worked
tiny cases (tests/golden/hand_worked.json), closed forms (the Taylor kernel
1 + s + s^2/2; the Hedgehog kernel as a sum of cosh), special cases that
reduce to a known answer (identity / zero maps, constant values), invariants
(weights form a distribution; Gibbs' inequality for the loss) and the
agreement of two independent forms (quadratic vs recurrent).

``test_planted_mistakes_are_caught`` plants plausible mistakes in copies of
the oracle (on the CPU) and asserts that at least one pin fails for each.
"""

import math
import os
import types

import numpy as np
import pytest

import oracle as ORACLE

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------------------
# pin checks, written against a module-like object O so mutants can be run
# ---------------------------------------------------------------------------

def _head(O, kind, q, k, v, W=None, b=None):
    pq = O.feature_map(kind, q, W, b)
    pk = O.feature_map(kind, k, W, b)
    return pq, pk, O.linattn_quadratic(pq, pk, v), O.mimicry_loss(q, k, pq, pk)


def check_hand_worked(O, golden):
    for name in ("E1", "E2", "E3", "E4"):
        g = golden[name]
        W = np.array(g["W"]) if "W" in g else None
        b = np.array(g["b"]) if "b" in g else None
        q, k, v = (np.array(g[t]) for t in ("q", "k", "v"))
        pq, pk, y, L = _head(O, g["kind"], q, k, v, W, b)
        np.testing.assert_allclose(y, np.array(g["y"]), rtol=0, atol=2e-10, err_msg=name)
        np.testing.assert_allclose(L, np.array(g["L"]), rtol=0, atol=2e-11, err_msg=name)
    g = golden["E4"]
    pq = O.feature_map("hedgehog", np.array(g["q"]), np.array(g["W"]), np.array(g["b"]))
    pk = O.feature_map("hedgehog", np.array(g["k"]), np.array(g["W"]), np.array(g["b"]))
    assert abs(pq[3] @ pk[1] - g["pair_4_2"]) < 1e-8
    # exact closed forms of E1 / E2
    assert abs(_head(O, "hedgehog", np.array([[0.0], [0.0]]), np.array([[0.0], [math.log(2)]]),
                     np.array([[1.0], [3.0]]), np.eye(1), np.zeros(1))[2][1, 0] - 19 / 9) < 1e-14
    y2 = _head(O, "taylor2", np.array([[1.0], [0.5], [-1.0]]), np.array([[0.5], [1.0], [2.0]]),
               np.array([[1.0], [2.0], [3.0]]))[2]
    assert abs(y2[1, 0] - 145 / 93) < 1e-14 and abs(y2[2, 0] - 37 / 17) < 1e-14


def check_taylor_closed_form(O, golden):
    for d in (1, 3, 16):
        q = RNG.normal(size=(50, d))
        k = RNG.normal(size=(50, d))
        pq, pk = O.taylor2_feature_map(q), O.taylor2_feature_map(k)
        s = np.sum(q * k, axis=-1)
        np.testing.assert_allclose(np.sum(pq * pk, axis=-1), 1 + s + s * s / 2, rtol=1e-12)
        assert pq.shape[-1] == 1 + d + d * d == O.taylor2_feature_dim(d)
    g = golden["taylor_dim_d64"]
    assert O.taylor2_feature_dim(g["d"]) == g["dprime"]
    # layout: [1, x, x_i x_j / sqrt2 (i-major)]
    x = np.array([2.0, 3.0, 5.0])
    p = O.taylor2_feature_map(x)
    assert p[0] == 1 and list(p[1:4]) == [2, 3, 5]
    assert abs(p[4 + 0 * 3 + 2] - 10 / math.sqrt(2)) < 1e-14


def check_hedgehog_cosh(O, golden):
    for d in (1, 4, 16):
        W = RNG.normal(size=(d, d)) / math.sqrt(d)
        b = RNG.normal(size=d) * 0.3
        q = RNG.normal(size=(20, d))
        k = RNG.normal(size=(20, d))
        pq = O.hedgehog_feature_map(q, W, b)
        pk = O.hedgehog_feature_map(k, W, b)
        hq, hk = q @ W + b, k @ W + b
        # phi(q).phi(k) = sum_l e^{hq+hk} + e^{-(hq+hk)} = 2 sum_l cosh(hq_l + hk_l)
        np.testing.assert_allclose(np.sum(pq * pk, axis=-1),
                                   2 * np.sum(np.cosh(hq + hk), axis=-1), rtol=1e-12)
        assert pq.shape[-1] == 2 * d and np.all(pq > 0)


def check_identity_and_zero_maps(O, golden):
    d = 5
    x = RNG.normal(size=(7, d))
    np.testing.assert_allclose(O.hedgehog_feature_map(x, np.eye(d), np.zeros(d)),
                               np.concatenate([np.exp(x), np.exp(-x)], -1), rtol=1e-15)
    np.testing.assert_array_equal(O.hedgehog_feature_map(x, np.zeros((d, d)), np.zeros(d)),
                                  np.ones((7, 2 * d)))


def check_orientation(O, golden):
    # W[0][1] = 1: input dimension 0 drives output feature 1 (h = x W + b).
    W = np.zeros((3, 3))
    W[0, 1] = 1.0
    x = np.array([0.7, -0.2, 0.4])
    p = O.hedgehog_feature_map(x, W, np.array([0.0, 0.25, 0.0]))
    np.testing.assert_allclose(p, [1, math.exp(0.95), 1, 1, math.exp(-0.95), 1], rtol=1e-15)


def check_weight_rows(O, golden):
    pq = np.exp(RNG.normal(size=(33, 8)))
    pk = np.exp(RNG.normal(size=(33, 8)))
    w = O.causal_weights(pq, pk)
    assert np.all(w >= 0)
    np.testing.assert_allclose(w.sum(-1), 1.0, rtol=1e-13)
    assert np.all(np.triu(w, 1) == 0)


def check_constant_values_and_first_row(O, golden):
    d = 4
    W = RNG.normal(size=(d, d)) * 0.5
    b = RNG.normal(size=d) * 0.1
    q, k = RNG.normal(size=(2, 40, d))
    v = np.full((40, 3), -1.75)
    y = _head(O, "hedgehog", q, k, v, W, b)[2]
    np.testing.assert_allclose(y, -1.75, rtol=1e-13)
    v = RNG.normal(size=(40, 3))
    for kind in ("hedgehog", "taylor2"):
        y = _head(O, kind, q, k, v, W, b)[2]
        np.testing.assert_allclose(y[0], v[0], rtol=1e-13)


def check_uniform_cases(O, golden):
    n, d = 30, 4
    q, k = RNG.normal(size=(2, n, d))
    v = RNG.normal(size=(n, 3))
    prefix_mean = np.cumsum(v, 0) / np.arange(1, n + 1)[:, None]
    y = _head(O, "hedgehog", q, k, v, np.zeros((d, d)), np.zeros(d))[2]
    np.testing.assert_allclose(y, prefix_mean, rtol=1e-12, atol=1e-14)
    y = _head(O, "taylor2", np.zeros((n, d)), k, v)[2]
    np.testing.assert_allclose(y, prefix_mean, rtol=1e-12, atol=1e-14)


def check_quadratic_vs_recurrent(O, golden):
    for kind, d in (("hedgehog", 6), ("taylor2", 3)):
        W = RNG.normal(size=(d, d)) / math.sqrt(d)
        b = RNG.normal(size=d) * 0.1
        q, k = RNG.normal(size=(2, 45, d))
        v = RNG.normal(size=(45, d))
        pq, pk = O.feature_map(kind, q, W, b), O.feature_map(kind, k, W, b)
        yq = O.linattn_quadratic(pq, pk, v)
        yr, S, z = O.linattn_recurrent(pq, pk, v)
        np.testing.assert_allclose(yr, yq, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(S, pk.T @ v, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(z, pk.sum(0), rtol=1e-12)
        np.testing.assert_allclose(O.linattn_rows(pq, pk, v, [0, 7, 44]), yq[[0, 7, 44]], rtol=1e-12)
        # continuation: a prefill to n1, then steps from that state == the full sequence
        y1, S1, z1 = O.linattn_recurrent(pq[:20], pk[:20], v[:20])
        y2, S2, z2 = O.linattn_recurrent(pq[20:], pk[20:], v[20:], S1, z1)
        np.testing.assert_allclose(np.concatenate([y1, y2]), yq, rtol=1e-11, atol=1e-13)
        y2b = O.linattn_quadratic(pq, pk, v)[20:]
        np.testing.assert_allclose(y2, y2b, rtol=1e-11, atol=1e-13)


def check_softmax_target(O, golden):
    d = 4
    q = RNG.normal(size=(2, d))
    k = RNG.normal(size=(2, d))
    p = O.softmax_target(q, k)
    # two keys: p_21 = logistic((q2.k1 - q2.k2) / sqrt d)
    p21 = 1.0 / (1.0 + math.exp((q[1] @ k[1] - q[1] @ k[0]) / math.sqrt(d)))
    assert abs(p[1, 0] - p21) < 1e-14 and p[0, 0] == 1.0 and p[0, 1] == 0.0
    big = O.softmax_target(np.full((5, 2), 30.0), np.full((5, 2), 30.0))
    np.testing.assert_allclose(big.sum(-1), 1.0, rtol=1e-14)


def check_loss_properties(O, golden):
    n, d = 40, 4
    W = RNG.normal(size=(d, d)) * 0.7
    b = RNG.normal(size=d) * 0.2
    q, k = RNG.normal(size=(2, n, d))
    pq, pk = O.feature_map("hedgehog", q, W, b), O.feature_map("hedgehog", k, W, b)
    L = O.mimicry_loss(q, k, pq, pk)
    p = O.softmax_target(q, k)
    H = -np.sum(np.where(p > 0, p * np.log(np.where(p > 0, p, 1)), 0), axis=-1)
    assert abs(L[0]) < 1e-15
    assert np.all(H >= -1e-15) and np.all(L >= H - 1e-12)          # Gibbs
    np.testing.assert_allclose(O.mimicry_loss_rows(q, k, pq, pk, [0, 5, 39]), L[[0, 5, 39]], rtol=1e-12)
    # W = 0, b = 0: uniform prediction, L_i = ln i for any q, k
    p0 = O.feature_map("hedgehog", q, np.zeros((d, d)), np.zeros(d))
    L0 = O.mimicry_loss(q, k, p0, p0)
    np.testing.assert_allclose(L0, np.log(np.arange(1, n + 1)), rtol=1e-13, atol=1e-15)


def check_loss_grad_finite_differences(O, golden):
    """The loss gradient w.r.t. W, b against central differences of the loss."""
    rng = np.random.default_rng(11)
    n, d, eps = 6, 3, 1e-6

    def total(Wq, bq, Wk, bk, q, k):
        pq = O.hedgehog_feature_map(q, Wq, bq)
        pk = O.hedgehog_feature_map(k, Wk, bk)
        return O.mimicry_loss(q, k, pq, pk).sum()

    def fd(f, X):
        g = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            g[idx] = (f(Xp) - f(Xm)) / (2 * eps)
        return g

    for trial in range(2):
        q, k = rng.normal(size=(2, n, d)) * 0.6
        Wq, Wk = rng.normal(size=(2, d, d)) * 0.5
        bq, bk = rng.normal(size=(2, d)) * 0.3
        # one map shared by queries and keys
        g = O.mimicry_loss_grad(q, k, Wq, bq)
        np.testing.assert_allclose(g[0] + g[2], fd(lambda X: total(X, bq, X, bq, q, k), Wq),
                                   rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(g[1] + g[3], fd(lambda X: total(Wq, X, Wq, X, q, k), bq),
                                   rtol=1e-6, atol=1e-8)
        # separate query and key maps
        g = O.mimicry_loss_grad(q, k, Wq, bq, Wk, bk)
        np.testing.assert_allclose(g[0], fd(lambda X: total(X, bq, Wk, bk, q, k), Wq), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(g[1], fd(lambda X: total(Wq, X, Wk, bk, q, k), bq), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(g[2], fd(lambda X: total(Wq, bq, X, bk, q, k), Wk), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(g[3], fd(lambda X: total(Wq, bq, Wk, X, q, k), bk), rtol=1e-6, atol=1e-8)
    # batched wrapper: sum over batch of per-head gradients of the summed loss
    B, H = 2, 2
    q = rng.normal(size=(B, H, 4, d)) * 0.6
    k = rng.normal(size=(B, H, 4, d)) * 0.6
    W = rng.normal(size=(H, d, d)) * 0.5
    b = rng.normal(size=(H, d)) * 0.3
    dW, db, _, _ = O.loss_grad_causal(q, k, W, b)

    def batch_total(Wx, bx):
        return O.loss_causal("hedgehog", q, k, Wx, bx)[1].sum()

    for h in range(H):
        for idx in [(0, 1), (2, 0)]:
            Wp, Wm = W.copy(), W.copy()
            Wp[(h,) + idx] += eps
            Wm[(h,) + idx] -= eps
            f = (batch_total(Wp, b) - batch_total(Wm, b)) / (2 * eps)
            assert abs(f - dW[(h,) + idx]) <= 1e-6 * max(1.0, abs(f))
        bp, bm = b.copy(), b.copy()
        bp[h, 1] += eps
        bm[h, 1] -= eps
        f = (batch_total(W, bp) - batch_total(W, bm)) / (2 * eps)
        assert abs(f - db[h, 1]) <= 1e-6 * max(1.0, abs(f))


def check_softmax_feature_map(O, golden):
    """Choice 4 (Eq. 5): softmax over the d learned directions, bias omitted."""
    rng = np.random.default_rng(21)
    n, d = 5, 4
    x = rng.normal(size=(n, d))
    W = rng.normal(size=(d, d)) * 0.8
    b = rng.normal(size=d)
    phi = O.feature_map("hedgehog_softmax", x, W, b)
    assert phi.shape == (n, 2 * d)
    # Eq. 5 written out feature by feature, for both signs of the directions
    for i in range(n):
        for sign, off in ((1.0, 0), (-1.0, d)):
            dots = [sign * sum(W[kk, l] * x[i, kk] for kk in range(d)) for l in range(d)]
            den = sum(math.exp(t) for t in dots)
            for l in range(d):
                assert abs(phi[i, off + l] - math.exp(dots[l]) / den) <= 1e-14
    # each half is a distribution over the directions; the bias is not used
    np.testing.assert_allclose(phi[:, :d].sum(-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(phi[:, d:].sum(-1), 1.0, rtol=1e-14)
    np.testing.assert_array_equal(phi, O.feature_map("hedgehog_softmax", x, W, 0 * b))
    # adding the same projection to every direction changes nothing
    u = rng.normal(size=d)
    np.testing.assert_allclose(O.hedgehog_softmax_feature_map(x, W + u[:, None]), phi, rtol=1e-12)
    # x = 0: uniform over the directions
    np.testing.assert_allclose(O.hedgehog_softmax_feature_map(np.zeros((2, d)), W), 1.0 / d, rtol=1e-15)


def check_softmax_map_loss_grad(O, golden):
    """Gradient through the Choice 4 (Eq. 5) map against central differences.

    Also an invariant of the map itself: adding one vector u to every column
    of W leaves phi unchanged, so the loss is flat along W + u 1^T and every
    row of dW sums to zero; the negation block alone (phi_- only) is checked
    by flipping the sign of W, which swaps the two halves and keeps the loss.
    """
    rng = np.random.default_rng(29)
    n, d, eps = 6, 3, 1e-6
    kind = "hedgehog_softmax"

    def total(Wq, Wk, q, k):
        pq = O.hedgehog_softmax_feature_map(q, Wq)
        pk = O.hedgehog_softmax_feature_map(k, Wk)
        return O.mimicry_loss(q, k, pq, pk).sum()

    def fd(f, X):
        g = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            g[idx] = (f(Xp) - f(Xm)) / (2 * eps)
        return g

    for trial in range(2):
        q, k = rng.normal(size=(2, n, d)) * 0.8
        Wq, Wk = rng.normal(size=(2, d, d)) * 0.9
        g = O.mimicry_loss_grad(q, k, Wq, None, kind=kind)
        assert g[1] is None and g[3] is None
        shared = g[0] + g[2]
        np.testing.assert_allclose(shared, fd(lambda X: total(X, X, q, k), Wq), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(shared.sum(axis=1), 0.0, atol=1e-12)
        # phi(x; -W) = [phi_-; phi_+]: a_ij and the loss are unchanged, dW flips sign
        gm = O.mimicry_loss_grad(q, k, -Wq, None, kind=kind)
        np.testing.assert_allclose(gm[0] + gm[2], -shared, rtol=1e-10, atol=1e-13)
        g = O.mimicry_loss_grad(q, k, Wq, None, Wk, None, kind=kind)
        np.testing.assert_allclose(g[0], fd(lambda X: total(X, Wk, q, k), Wq), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(g[2], fd(lambda X: total(Wq, X, q, k), Wk), rtol=1e-6, atol=1e-8)
    # batched wrapper: sum over the batch of per-head gradients of the summed loss
    B, H = 2, 2
    q = rng.normal(size=(B, H, 4, d)) * 0.8
    k = rng.normal(size=(B, H, 4, d)) * 0.8
    W = rng.normal(size=(H, d, d)) * 0.9
    dW, db, dWk, dbk = O.loss_grad_causal(q, k, W, None, kind=kind)
    assert db is None and dWk is None and dbk is None

    def batch_total(Wx):
        return O.loss_causal(kind, q, k, Wx, None)[1].sum()

    for h in range(H):
        for idx in [(0, 1), (2, 0)]:
            Wp, Wm = W.copy(), W.copy()
            Wp[(h,) + idx] += eps
            Wm[(h,) + idx] -= eps
            f = (batch_total(Wp) - batch_total(Wm)) / (2 * eps)
            assert abs(f - dW[(h,) + idx]) <= 1e-6 * max(1.0, abs(f))
    Wk2 = rng.normal(size=(H, d, d)) * 0.9
    sq, _, sk, _ = O.loss_grad_causal(q, k, W, None, Wk2, None, kind=kind)
    rq, rk = np.zeros_like(sq), np.zeros_like(sk)
    for bi in range(B):
        for h in range(H):
            g = O.mimicry_loss_grad(q[bi, h], k[bi, h], W[h], None, Wk2[h], None, kind=kind)
            rq[h] += g[0]
            rk[h] += g[2]
    np.testing.assert_allclose(sq, rq, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(sk, rk, rtol=1e-13, atol=1e-15)


def check_entropies_and_kl(O, golden):
    """H(a_i) of the spikiness section, KL = CE - H(p) (Gibbs), known extremes."""
    n = 7
    # uniform rows: log i; one-hot rows: 0
    U = np.tril(np.ones((n, n))) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(O.attention_entropy(U), np.log(np.arange(1, n + 1)), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(O.attention_entropy(np.eye(n)), 0.0, atol=1e-15)
    rng = np.random.default_rng(5)
    d = 3
    q, k = rng.normal(size=(2, n, d))
    # weights equal to the target: phi(k_j) = e_j, phi(q_i)_j = exp(q_i . k_j / sqrt d)
    pk = np.eye(n)
    pq = np.exp(q @ k.T / math.sqrt(d))
    st = O.mimicry_stats(q, k, pq, pk)
    p = O.softmax_target(q, k)
    Hp = -np.sum(np.where(p > 0, p * np.log(np.where(p > 0, p, 1.0)), 0.0), axis=-1)
    np.testing.assert_allclose(st[:, 1], 0.0, atol=1e-13)
    np.testing.assert_allclose(st[:, 0], Hp, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(st[:, 2], Hp, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(st[:, 3], Hp, rtol=1e-12, atol=1e-14)
    # a generic map: KL written directly as sum p log(p / w), and non-negative
    W = rng.normal(size=(d, d)) * 0.6
    bb = rng.normal(size=d) * 0.2
    pq, pk = O.feature_map("hedgehog", q, W, bb), O.feature_map("hedgehog", k, W, bb)
    st = O.mimicry_stats(q, k, pq, pk)
    a = np.tril(pq @ pk.T)
    w = a / a.sum(-1, keepdims=True)
    kl = np.array([sum(p[i, j] * math.log(p[i, j] / w[i, j]) for j in range(i + 1)) for i in range(n)])
    np.testing.assert_allclose(st[:, 1], kl, rtol=1e-10, atol=1e-13)
    assert np.all(st[:, 1] >= -1e-13)
    np.testing.assert_allclose(st[:, 0], O.mimicry_loss(q, k, pq, pk), rtol=1e-13)
    # W = 0, b = 0: uniform linear-attention weights, H(w) = log i
    p0 = O.feature_map("hedgehog", q, np.zeros((d, d)), np.zeros(d))
    st0 = O.mimicry_stats(q, k, p0, p0)
    np.testing.assert_allclose(st0[:, 3], np.log(np.arange(1, n + 1)), rtol=1e-13, atol=1e-15)
    # batched wrapper agrees per head
    B, H = 2, 2
    qb = rng.normal(size=(B, H, 5, d))
    kb = rng.normal(size=(B, H, 5, d))
    Wb = rng.normal(size=(H, d, d)) * 0.5
    bbb = rng.normal(size=(H, d)) * 0.2
    sb = O.stats_causal("hedgehog_softmax", qb, kb, Wb, bbb)
    for bi in range(B):
        for h in range(H):
            ph_q = O.hedgehog_softmax_feature_map(qb[bi, h], Wb[h])
            ph_k = O.hedgehog_softmax_feature_map(kb[bi, h], Wb[h])
            np.testing.assert_allclose(sb[bi, h], O.mimicry_stats(qb[bi, h], kb[bi, h], ph_q, ph_k),
                                       rtol=1e-14)


PINS = [check_hand_worked, check_taylor_closed_form, check_hedgehog_cosh,
        check_identity_and_zero_maps, check_orientation, check_weight_rows,
        check_constant_values_and_first_row, check_uniform_cases,
        check_quadratic_vs_recurrent, check_softmax_target, check_loss_properties,
        check_loss_grad_finite_differences, check_softmax_feature_map, check_entropies_and_kl,
        check_softmax_map_loss_grad]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, golden):
    pin(ORACLE, golden)


# ---------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# ---------------------------------------------------------------------------

MUTANTS = {
    "negated_half_keeps_bias": ("np.exp(-h)]", "np.exp(-(x @ W) + b)]"),
    "taylor_without_sqrt2": ("outer / math.sqrt(2.0)", "outer"),
    "taylor_constant_dropped": ("[one, x, outer", "[0 * one, x, outer"),
    "W_transposed": ("h = x @ W + b", "h = x @ W.T + b"),
    "bias_dropped": ("h = x @ W + b", "h = x @ W"),
    "softmax_scale_1_over_d": ("(q @ k.T) / math.sqrt(d)", "(q @ k.T) / d"),
    "diagonal_excluded": ("a = np.tril(a)", "a = np.tril(a, -1) + np.diag(np.diag(a)) * 0 + 1e-300"),
    "quadratic_excludes_diagonal": ("a = np.tril(_f64(phi_q) @ _f64(phi_k).T)",
                                    "a = np.tril(_f64(phi_q) @ _f64(phi_k).T, -1) + 1e-300"),
    "readout_before_update": ("    S = _f64(S) + np.outer(phi_k_t, v_t)\n    z = _f64(z) + phi_k_t\n    y = (phi_q_t @ S) / (phi_q_t @ z)",
                              "    y = (phi_q_t @ (_f64(S) + 1e-300)) / (phi_q_t @ (_f64(z) + 1e-300))\n    S = _f64(S) + np.outer(phi_k_t, v_t)\n    z = _f64(z) + phi_k_t"),
    "loss_unnormalised_prediction": ("np.log(w[i, : i + 1])", "np.log(np.tril(_f64(phi_q) @ _f64(phi_k).T)[i, : i + 1])"),
    "loss_log2": ("out[i] = -np.sum(p[i, : i + 1] * np.log(w[i, : i + 1]))",
                  "out[i] = -np.sum(p[i, : i + 1] * np.log2(w[i, : i + 1]))"),
    "loss_sign_flipped": ("out[i] = -np.sum(p[i, : i + 1]", "out[i] = np.sum(p[i, : i + 1]"),
    "softmax_no_max_subtraction": ("    s = s - s.max(axis=-1, keepdims=True)\n", "    s = s * 1.0\n"),
    "grad_without_partition_term": ("1.0 / A[:, None] - p / np.where", "0.0 / A[:, None] - p / np.where"),
    "grad_negative_half_sign": ("dhq = dpq[:, :d] * pq[:, :d] - dpq[:, d:]", "dhq = dpq[:, :d] * pq[:, :d] + dpq[:, d:]"),
    "grad_no_key_side": ("k.T @ dhk, dhk.sum(axis=0)\n", "0 * (k.T @ dhk), 0 * dhk.sum(axis=0)\n"),
    "grad_W_transposed": ("return q.T @ dhq, dhq.sum(axis=0)", "return (q.T @ dhq).T, dhq.sum(axis=0)"),
    "grad_acausal": ("g = np.where(mask, 1.0 / A", "g = np.where(True, 1.0 / A"),
    "softmax_map_over_rows": ("pos = pos / pos.sum(axis=-1, keepdims=True)",
                              "pos = pos / pos.sum(axis=0, keepdims=True)"),
    "softmax_map_shared_normaliser": ("neg = neg / neg.sum(axis=-1, keepdims=True)",
                                      "neg = neg / pos.sum(axis=-1, keepdims=True)"),
    "softmax_map_negation_dropped": ("    neg = np.exp(-h)\n", "    neg = np.exp(h)\n"),
    "softmax_map_raw_dispatch": ("return hedgehog_softmax_feature_map(x, W)\n",
                                 "return hedgehog_feature_map(x, W, b)\n"),
    "softmax_grad_uncentred": ("return s * (y - (y * s).sum(axis=-1, keepdims=True))", "return s * y"),
    "softmax_grad_negative_half_added": ("dhq = _softmax_vjp(dpq[:, :d], pq[:, :d]) - _softmax_vjp",
                                         "dhq = _softmax_vjp(dpq[:, :d], pq[:, :d]) + _softmax_vjp"),
    "softmax_grad_key_side_query_features": ("dhk = _softmax_vjp(dpk[:, :d], pk[:, :d])",
                                             "dhk = _softmax_vjp(dpk[:, :d], pq[:, :d])"),
    "softmax_grad_centred_over_rows": ("(y * s).sum(axis=-1, keepdims=True)", "(y * s).sum(axis=0, keepdims=True)"),
    "entropy_log2": ("out[i] = -np.sum(nz * np.log(nz))", "out[i] = -np.sum(nz * np.log2(nz))"),
    "kl_sign_flipped": ("np.stack([ce, ce - hp, hp, hw]", "np.stack([ce, hp - ce, hp, hw]"),
    "model_entropy_of_target": ("hw = attention_entropy(w)", "hw = attention_entropy(p)"),
}


def _mutant(old, new):
    path = os.path.join(ROOT, "oracle", "hedgehog_oracle.py")
    src = open(path).read()
    assert old in src, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    with np.errstate(all="ignore"):
        exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, golden):
    mod = _mutant(*MUTANTS[name])
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod, golden)
        except (AssertionError, FloatingPointError, ValueError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"

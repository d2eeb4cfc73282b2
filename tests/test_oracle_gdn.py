"""Pins for the GDN tree-verification oracle (oracle/gdn.py), independent of it.

- The chunked form of the same recurrence, written from its algebra: with
  u_t = beta_t (v_t - alpha_t S_parent^T k_t) and g_t the product of alpha along
  the path, S_t = g_t S_0 + sum over ancestors-or-self i of (g_t / g_i) k_i u_i^T,
  so U solves the masked triangular system (I + X) U = beta * (V - g * K S_0)
  with X_ti = beta_t (g_t / g_i) k_t . k_i on strict ancestors, and
  O = g * (Q S_0) + (Y masked to ancestors-or-self) U with Y_ti = (g_t / g_i) q_t . k_i.
  The system is solved with a library triangular solve; the brute-force path
  recurrence must agree to rounding.
- Closed forms: beta = 0 only decays S_0; with alpha = beta = 1 and a unit key
  the delta rule stores v exactly (S_t^T k_t = v_t); a star tree is one step
  from S_0 per node.
- The deferred commit equals the recurrence along the accepted path, equals
  g_last S_0 + sum (g_last / g_p) k_p u_p^T over the path, and an empty accept
  keeps S_0.
"""
import numpy as np
import pytest
from scipy.linalg import solve_triangular

from oracle import gdn
import workloads


def anc_masks(parent):
    N = len(parent)
    anc = np.zeros(N, np.uint64)
    for t in range(N):
        m = 1 << t
        p = parent[t]
        if p >= 0:
            m |= int(anc[p])
        anc[t] = np.uint64(m)
    return anc


def inputs(rng, B, N, Hk, Hv, dk, dv, trees, unit_keys=True):
    parent = np.stack([trees(rng) for _ in range(B)])
    anc = np.stack([anc_masks(p) for p in parent])
    q = rng.standard_normal((B, N, Hk, dk))
    k = rng.standard_normal((B, N, Hk, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((B, N, Hv, dv))
    alpha = rng.uniform(0.6, 1.0, (B, N, Hv))
    beta = rng.uniform(0.05, 1.0, (B, N, Hv))
    state = 0.5 * rng.standard_normal((B, Hv, dk, dv))
    return dict(parent=parent, anc=anc, q=q, k=k, v=v, alpha=alpha, beta=beta, state=state)


def chunked(x):
    """The masked triangular-solve form (independent of the per-path loop)."""
    B, N, Hk, dk = x["q"].shape
    Hv, dv = x["v"].shape[2:]
    G = Hv // Hk
    out = np.zeros((B, N, Hv, dv))
    U = np.zeros((B, N, Hv, dv))
    for b in range(B):
        A = np.array([[(int(x["anc"][b, t]) >> i) & 1 for i in range(N)] for t in range(N)], float)
        As = A - np.eye(N)
        for h in range(Hv):
            K, Q = x["k"][b, :, h // G], x["q"][b, :, h // G]
            a, be = x["alpha"][b, :, h], x["beta"][b, :, h]
            lg = np.log(a)
            cum = A @ lg                          # log g_t: sum of log alpha over ancestors-or-self
            gam = np.exp(cum[:, None] - cum[None, :])  # g_t / g_i
            S0 = x["state"][b, h]
            X = be[:, None] * gam * (K @ K.T) * As
            Y = gam * (Q @ K.T) * A
            g = np.exp(cum)
            rhs = be[:, None] * (x["v"][b, :, h] - g[:, None] * (K @ S0))
            Uh = solve_triangular(np.eye(N) + X, rhs, lower=True)
            U[b, :, h] = Uh
            out[b, :, h] = g[:, None] * (Q @ S0) + Y @ Uh
    return out, U


TREES = {
    "random": lambda N: (lambda rng: workloads.tree_random(rng, N, 6)),
    "chain": lambda N: (lambda rng: workloads.tree_chain(N)),
    "star": lambda N: (lambda rng: workloads.tree_star(N)),
}


@pytest.mark.parametrize("tree", list(TREES))
@pytest.mark.parametrize("seed", range(3))
def test_recurrence_equals_chunked_solve(tree, seed):
    rng = np.random.default_rng(seed)
    N = 11
    x = inputs(rng, 2, N, 2, 4, 8, 6, TREES[tree](N))
    ref = gdn.tree_verify(x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["anc"])
    out, U = chunked(x)
    np.testing.assert_allclose(ref["out"], out, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(ref["u"], U, rtol=1e-10, atol=1e-10)


def test_beta_zero_only_decays():
    rng = np.random.default_rng(3)
    N = 9
    x = inputs(rng, 2, N, 1, 2, 8, 8, TREES["random"](N))
    x["beta"][:] = 0.0
    r = gdn.tree_verify(x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["anc"])
    for b in range(2):
        for h in range(2):
            for t in range(N):
                g = np.prod([x["alpha"][b, j, h] for j in gdn.path_of(x["anc"][b, t], t)])
                np.testing.assert_allclose(r["g"][b, t, h], g, rtol=1e-14)
                np.testing.assert_allclose(r["out"][b, t, h], g * x["state"][b, h].T @ x["q"][b, t, 0],
                                           rtol=1e-12, atol=1e-12)
    assert np.all(r["u"] == 0)


def test_delta_rule_stores_v_at_unit_key():
    """alpha = beta = 1 and |k_t| = 1: S_t^T k_t = v_t at every node."""
    rng = np.random.default_rng(4)
    N = 10
    x = inputs(rng, 2, N, 2, 2, 8, 5, TREES["random"](N))
    x["alpha"][:] = 1.0
    x["beta"][:] = 1.0
    r = gdn.tree_verify(x["state"], x["k"], x["k"], x["v"], x["alpha"], x["beta"], x["anc"])
    np.testing.assert_allclose(r["out"], x["v"], rtol=1e-12, atol=1e-12)


def test_star_tree_is_one_step_per_node():
    rng = np.random.default_rng(5)
    N = 7
    x = inputs(rng, 1, N, 1, 3, 6, 4, TREES["star"](N))
    r = gdn.tree_verify(x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["anc"])
    for h in range(3):
        for t in range(N):
            k, q, v = x["k"][0, t, 0], x["q"][0, t, 0], x["v"][0, t, h]
            a, be = x["alpha"][0, t, h], x["beta"][0, t, h]
            S0 = x["state"][0, h]
            # S_1^T q = a S0^T q - a be (k.q) S0^T k + be (k.q) v
            expect = a * S0.T @ q - a * be * (k @ q) * (S0.T @ k) + be * (k @ q) * v
            np.testing.assert_allclose(r["out"][0, t, h], expect, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_commit_is_the_path_state(seed):
    rng = np.random.default_rng(10 + seed)
    N, B, Hv = 12, 3, 2
    x = inputs(rng, B, N, 1, Hv, 6, 5, TREES["random"](N))
    r = gdn.tree_verify(x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["anc"])
    # accepted path: a random node's ancestors-or-self; sequence 2 accepts nothing
    acc = np.zeros((B, N), np.int32)
    n_acc = np.zeros(B, np.int32)
    for b in range(2):
        leaf = int(rng.integers(0, N))
        p = gdn.path_of(x["anc"][b, leaf], leaf)
        acc[b, :len(p)] = p
        n_acc[b] = len(p)
    new = gdn.commit(x["state"], x["k"], x["v"], x["alpha"], x["beta"], acc, n_acc)
    assert np.array_equal(new[2], x["state"][2])
    for b in range(2):
        last = acc[b, n_acc[b] - 1]
        for h in range(Hv):
            # the committed state reproduces the node's verify output ...
            np.testing.assert_allclose(new[b, h].T @ x["q"][b, last, 0], r["out"][b, last, h],
                                       rtol=1e-11, atol=1e-11)
            # ... and equals the deferred form g_last S_0 + sum (g_last/g_p) k_p u_p^T
            gl = r["g"][b, last, h]
            S = gl * x["state"][b, h]
            for p in acc[b, :n_acc[b]]:
                S = S + (gl / r["g"][b, p, h]) * np.outer(x["k"][b, p, 0], r["u"][b, p, h])
            np.testing.assert_allclose(new[b, h], S, rtol=1e-11, atol=1e-11)

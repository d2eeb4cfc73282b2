"""CPU oracle for rollback-free tree verification of a Gated DeltaNet layer
(test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this module; the product library never loads it and it imports nothing
from the product package.

Source: "Technische Samenvatting: Trees from Marginals (DFlash-TfM)",
"3. Rollback-vrije Boom-verificatie voor GDN": a GDN layer updates its state
by S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T; verifying
a draft tree must give every node the output of the state reached along its
own root-to-node path, without updating the committed state; the state is
committed once the accepted branch is known.

``tree_verify`` is that definition written out: for every node it runs the
recurrence along the node's path from the committed state S_0 (fp64) and
reads the output o_t = S_t^T q_t.  It also returns, per node, the quantities
the deferred commit needs:
    u_t = beta_t (v_t - alpha_t S_parent^T k_t)   (so S_t = alpha_t S_parent + k_t u_t^T)
    g_t = product of alpha along the path (root .. t).
``commit`` runs the recurrence along the accepted path (an empty accept keeps
S_0).

Readings (where the page is silent): S is d_k x d_v and the output is
o_t = S_t^T q_t with no extra scale (q arrives scaled); alpha and beta are
per node and per value head; value head h reads query/key head
h // (Hv / Hk); the path of a node is its ancestors-or-self in the order given
by the ancestor bitmask (parents precede children), root first.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def path_of(anc_row: int, t: int):
    """Ancestors-or-self of node t, root first (bit a of anc_row set <=> a is one)."""
    return [a for a in range(t + 1) if (int(anc_row) >> a) & 1]


def tree_verify(state, q, k, v, alpha, beta, anc):
    """state fp [B, Hv, dk, dv] (S_0, as d_k x d_v matrices); q, k [B, N, Hk, dk];
    v [B, N, Hv, dv]; alpha, beta [B, N, Hv]; anc uint64 [B, N].
    Returns dict of out [B, N, Hv, dv], u [B, N, Hv, dv], g [B, N, Hv] (fp64)."""
    state = np.asarray(state, np.float64)
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    B, N, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    G = Hv // Hk
    out = np.zeros((B, N, Hv, dv))
    u = np.zeros((B, N, Hv, dv))
    g = np.zeros((B, N, Hv))
    eye = np.eye(dk)
    for b in range(B):
        for h in range(Hv):
            hk = h // G
            for t in range(N):
                S = state[b, h].copy()
                gt = 1.0
                for j in path_of(anc[b, t], t):
                    kj = k[b, j, hk]
                    if j == t:  # the pseudo-value of t, from its parent's state
                        u[b, t, h] = beta[b, j, h] * (v[b, j, h] - alpha[b, j, h] * (S.T @ kj))
                    S = alpha[b, j, h] * (eye - beta[b, j, h] * np.outer(kj, kj)) @ S \
                        + beta[b, j, h] * np.outer(kj, v[b, j, h])
                    gt *= alpha[b, j, h]
                out[b, t, h] = S.T @ q[b, t, hk]
                g[b, t, h] = gt
    return dict(out=out, u=u, g=g)


def commit(state, k, v, alpha, beta, acc_nodes, n_acc):
    """The state after the accepted path: the recurrence along acc_nodes[b, :n_acc[b]]
    from S_0 (fp64).  Returns [B, Hv, dk, dv]."""
    state = np.asarray(state, np.float64)
    k, v = np.asarray(k, np.float64), np.asarray(v, np.float64)
    alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    B, Hv, dk, dv = state.shape
    Hk = k.shape[2]
    G = Hv // Hk
    new = state.copy()
    eye = np.eye(dk)
    for b in range(B):
        for h in range(Hv):
            S = state[b, h].copy()
            for j in acc_nodes[b, :n_acc[b]]:
                kj = k[b, j, h // G]
                S = alpha[b, j, h] * (eye - beta[b, j, h] * np.outer(kj, kj)) @ S \
                    + beta[b, j, h] * np.outer(kj, v[b, j, h])
            new[b, h] = S
    return new

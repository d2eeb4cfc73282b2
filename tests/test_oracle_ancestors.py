"""Pins for the oracle's ancestor mask and position ids (CPU only).

The mask rule comes from "Tree spec-decode -> vLLM serve integration spec",
"2. Verify" (node -> node block: 0 iff ancestor-or-self, else -inf; position
ids ctx_len-1+depth).  The oracle's pointer chase is checked against an
independent transitive closure of the parent relation, over every tree with
N <= 6 nodes, and against the tree printed on the DDTree page.
"""
import itertools
import os

import numpy as np
import pytest

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ddtree_printed_tree.txt")


def closure_mask(parent):
    """Ancestor-or-self relation by boolean matrix powers (reachability)."""
    N = len(parent)
    A = np.zeros((N, N), bool)
    for t, p in enumerate(parent):
        if p >= 0:
            A[t, p] = True
    R = np.eye(N, dtype=bool)
    step = np.eye(N, dtype=bool)
    for _ in range(N):
        step = (step.astype(np.int64) @ A.astype(np.int64)) > 0
        R |= step
    return R


def all_trees(N):
    """Every parent array with parent[t] in [-1, t-1]: N! labelled trees."""
    return [np.array(p, np.int32) for p in itertools.product(*[range(-1, t) for t in range(N)])]


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6])
def test_exhaustive_small_trees(oracle_mod, N):
    trees = all_trees(N)
    assert len(trees) == int(np.prod(np.arange(1, N + 1)))
    parent = np.stack(trees)
    depth = np.stack([workloads.depths_of(p) for p in trees])
    ctx = np.arange(len(trees), dtype=np.int32) % 37
    mask, pos, status = oracle_mod.ancestors(parent, depth, ctx)
    assert (status == 0).all()
    for b, p in enumerate(trees):
        R = closure_mask(p)
        assert np.array_equal(mask[b].astype(bool), R), p
        # popcount of the row equals the depth; bit t always set
        assert np.array_equal(mask[b].sum(1), depth[b])
        assert np.array_equal(pos[b], ctx[b] - 1 + depth[b])


def test_chain_is_causal_and_star_is_identity(oracle_mod):
    N = 32
    mask, _, st = oracle_mod.ancestors(workloads.tree_chain(N)[None], np.arange(1, N + 1)[None],
                                       np.array([10]))
    assert st[0] == 0
    assert np.array_equal(mask[0], np.tril(np.ones((N, N), np.uint8)))
    mask, _, st = oracle_mod.ancestors(workloads.tree_star(N)[None], np.ones((1, N)),
                                       np.array([10]))
    assert st[0] == 0
    assert np.array_equal(mask[0], np.eye(N, dtype=np.uint8))


def test_random_trees_up_to_64(oracle_mod):
    rng = np.random.Generator(np.random.PCG64(7))
    for N in (7, 17, 32, 33, 64):
        par = np.stack([workloads.tree_random(rng, N, 12) for _ in range(8)])
        dep = np.stack([workloads.depths_of(p) for p in par])
        mask, pos, st = oracle_mod.ancestors(par, dep, np.full(8, 100))
        assert (st == 0).all()
        for b in range(8):
            assert np.array_equal(mask[b].astype(bool), closure_mask(par[b]))


def read_golden():
    g = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            g[k] = [int(x) for x in v]
    return g


def test_ddtree_printed_tree(oracle_mod):
    g = read_golden()
    N = g["nodes"][0]
    parent = np.array(g["parents"], np.int32)
    depth = np.array(g["depths"], np.int32)
    assert len(parent) == len(depth) == N == 32
    ctx = 100  # mask width 132 = 100 context columns + 32 node columns
    mask, pos, st = oracle_mod.ancestors(parent[None], depth[None], np.array([ctx]))
    assert st[0] == 0, "the printed parents and depths are mutually consistent"
    m = mask[0]
    roots = parent < 0
    assert roots.sum() == 10 and (depth[roots] == 1).all()
    assert np.array_equal(m[roots], np.eye(N, dtype=np.uint8)[roots])
    for t in np.nonzero(~roots)[0]:
        assert m[t].sum() == 2 and m[t, t] == 1 and m[t, parent[t]] == 1
    bias = oracle_mod.dense_bias(m, ctx)
    assert (1, 1) + bias.shape == tuple(g["mask_shape"])
    assert (bias[:, :ctx] == 0).all()
    assert np.array_equal(np.isfinite(bias[:, ctx:]), m.astype(bool))
    assert np.array_equal(pos[0], ctx - 1 + depth)


@pytest.mark.parametrize("bad", ["parent_ge_t", "parent_lt_m1", "depth"])
def test_malformed_trees_flagged(oracle_mod, bad):
    par = workloads.tree_random(np.random.Generator(np.random.PCG64(3)), 12, 5)
    dep = workloads.depths_of(par)
    par2 = par.copy()
    dep2 = dep.copy()
    if bad == "parent_ge_t":
        par2[4] = 4
    elif bad == "parent_lt_m1":
        par2[6] = -2
    else:
        dep2[9] += 1
    mask, pos, st = oracle_mod.ancestors(np.stack([par, par2]), np.stack([dep, dep2]),
                                         np.array([5, 5]))
    assert st[0] == 0 and st[1] == 2

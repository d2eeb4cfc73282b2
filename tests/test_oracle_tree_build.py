"""Pins for the draft-tree oracle (oracle/tree_build.py), independent of it.

- topk: an explicit selection loop (repeatedly take the largest remaining value,
  lowest index first), the already-pinned argmax oracle for k = 1, bf16 bit
  patterns with known values, and planted ties / NaN / +-0 / -inf.
- build_tree (w = 1): brute force over every node of the K-ary tree of depth L:
  the tree is the set of the `budget` best-scoring nodes, popped in
  non-increasing score order.
- build_tree (any w): structural invariants every tree of this construction has
  (prefix-closed child ranks, child counts non-increasing with sibling rank),
  hand-derived examples, and the round count ceil(budget / w) of "Trees from
  Marginals", "2. Boomconstructie".
- The DDTree page's printed tree ("From Linear to Tree-Walk", "The Successful
  Test": 32 nodes, top_k = 10, horizon 5) is an output of this construction:
  per-depth log-probabilities are solved for (a linear feasibility problem)
  such that the oracle prints exactly the page's parent and depth lists.
"""
import itertools
import os

import numpy as np
import pytest

from oracle import tree_build as tb

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ddtree_printed_tree.txt")


# ------------------------------------------------------------------ topk

def select_loop(row, k):
    """Selection by repeated scans: largest remaining value, lowest index first."""
    vals = [(-np.inf if np.isnan(v) else float(v)) for v in row]
    taken = set()
    out_v, out_i = [], []
    for _ in range(k):
        best_i = None
        for i, v in enumerate(vals):
            if i in taken:
                continue
            if best_i is None or v > vals[best_i]:
                best_i = i
        taken.add(best_i)
        out_i.append(best_i)
        out_v.append(vals[best_i])
    return out_v, out_i


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_selection_loop(seed):
    rng = np.random.default_rng(seed)
    rows, V = 5, 97
    x = rng.integers(-4, 5, size=(rows, V)).astype(np.float32)  # many ties
    x[0, 3] = np.nan
    x[1, :] = -np.inf
    x[1, 50] = np.nan
    x[2, ::2] = -0.0
    x[2, 1::2] = 0.0
    for k in (1, 4, 10, V):
        vals, idx = tb.topk(x, k, "f32")
        for r in range(rows):
            ev, ei = select_loop(x[r], k)
            assert list(idx[r]) == ei
            assert np.array_equal(vals[r], np.array(ev, np.float32))


def test_topk_k1_is_the_argmax_oracle(oracle_mod):
    rng = np.random.default_rng(7)
    x = rng.integers(-3, 4, size=(40, 333)).astype(np.float32)
    x[5, 10] = np.nan
    _, idx = tb.topk(x, 1, "f32")
    assert np.array_equal(idx[:, 0], oracle_mod.argmax(x, "f32"))
    bits = (rng.integers(0, 1 << 16, size=(40, 333))).astype(np.uint16)
    _, idxb = tb.topk(bits, 1, "bf16")
    assert np.array_equal(idxb[:, 0], oracle_mod.argmax(bits, "bf16"))


def test_topk_bf16_bit_patterns():
    # 0x3F80 = 1.0, 0x4000 = 2.0, 0xC000 = -2.0, 0x7FC0 = NaN, 0xFF80 = -inf, 0x8000 = -0
    row = np.array([[0x3F80, 0x4000, 0xC000, 0x7FC0, 0xFF80, 0x8000, 0x4000]], np.uint16)
    vals, idx = tb.topk(row, 7, "bf16")
    assert list(idx[0]) == [1, 6, 0, 5, 2, 3, 4]
    assert list(vals[0]) == [2.0, 2.0, 1.0, 0.0, -2.0, -np.inf, -np.inf]


# ------------------------------------------------------------------ build_tree

def marginals(rng, L, K):
    """Per-depth sorted log-probabilities of random marginals and random token ids."""
    logits = rng.standard_normal((L, 64)).astype(np.float64)
    lp = logits - np.log(np.exp(logits).sum(1, keepdims=True))
    vals = -np.sort(-lp, axis=1)[:, :K].astype(np.float32)
    toks = rng.permutation(1000)[:L * K].reshape(L, K).astype(np.int32)
    return vals, toks


def all_nodes(vals):
    """Every node of the K-ary tree of depth L as (rank path, fp32 score)."""
    L, K = vals.shape
    out = []
    for d in range(1, L + 1):
        for path in itertools.product(range(K), repeat=d):
            s = vals[0, path[0]]
            for j in range(1, d):
                s = np.float32(s + vals[j, path[j]])
            out.append((path, np.float32(s)))
    return out


def rank_paths(tree, toks):
    L, K = toks.shape
    rank = [{int(toks[d, r]): r for r in range(K)} for d in range(L)]
    paths = []
    for t in range(tree["n"]):
        d = tree["depth"][t]
        r = rank[d - 1][int(tree["tokens"][t])]
        p = tree["parent"][t]
        paths.append((r,) if p < 0 else paths[p] + (r,))
    return paths


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("L,K,budget", [(3, 3, 10), (4, 2, 17), (2, 5, 12), (3, 4, 40)])
def test_w1_is_the_best_budget_nodes(seed, L, K, budget):
    rng = np.random.default_rng(seed)
    vals, toks = marginals(rng, L, K)
    tree = tb.build_tree_one(vals, toks, budget, w=1)
    nodes = all_nodes(vals)
    scores = sorted((s for _, s in nodes), reverse=True)
    n = min(budget, len(nodes))
    assert tree["n"] == n
    # popped in non-increasing score order, and the scores are the n best
    assert all(tree["score"][i] >= tree["score"][i + 1] for i in range(n - 1))
    assert np.array_equal(tree["score"], np.array(scores[:n], np.float32))
    if n < len(nodes) and scores[n - 1] > scores[n]:
        best = {path for path, s in nodes if s >= scores[n - 1]}
        assert set(rank_paths(tree, toks)) == best
    # each node's stored score is the fp32 path sum
    by_path = dict(nodes)
    for path, s in zip(rank_paths(tree, toks), tree["score"]):
        assert by_path[path] == s


def check_structure(tree, toks, K):
    n = tree["n"]
    par, dep = tree["parent"], tree["depth"]
    paths = rank_paths(tree, toks)
    children = {}
    for t in range(n):
        assert par[t] < t
        assert dep[t] == (1 if par[t] < 0 else dep[par[t]] + 1)
        children.setdefault(int(par[t]), []).append(paths[t][-1])
    for p, ranks in children.items():
        assert ranks == sorted(ranks) and ranks == list(range(len(ranks)))  # rank prefix
    # child counts never grow with sibling rank (one marginal per depth)
    for p in list(children) + [-1]:
        sib = [t for t in range(n) if par[t] == p]
        counts = [len(children.get(t, [])) for t in sib]
        assert counts == sorted(counts, reverse=True)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("w", [1, 2, 3, 8])
def test_structure_and_rounds_any_w(seed, w):
    rng = np.random.default_rng(100 + seed)
    L, K, budget = 5, 4, 29
    vals, toks = marginals(rng, L, K)
    tree = tb.build_tree_one(vals, toks, budget, w=w)
    assert tree["n"] == budget
    # ceil(budget / w) rounds whenever every round finds w candidates, which
    # holds from the first round on when w <= K; a narrower first round adds some
    if w <= K:
        assert tree["rounds"] == -(-budget // w)
    else:
        assert tree["rounds"] >= -(-budget // w)
    check_structure(tree, toks, K)


def test_hand_examples():
    # K=2, L=2.  Depth 1: tokens 10, 11 with log-probs -1, -5; depth 2: tokens 20, 21
    # with -0.5, -0.6.  Budget 3.
    vals = np.array([[-1.0, -5.0], [-0.5, -0.6]], np.float32)
    toks = np.array([[10, 11], [20, 21]], np.int32)
    # w = 1: pop root 10 (-1); its children -1.5 and -1.6 beat root 11 (-5).
    t1 = tb.build_tree_one(vals, toks, 3, w=1)
    assert list(t1["tokens"]) == [10, 20, 21] and list(t1["parent"]) == [-1, 0, 0]
    assert list(t1["score"]) == [np.float32(-1.0), np.float32(-1.5), np.float32(-1.6)]
    # w = 2: the first expansion round pops both roots (the only candidates); the
    # second takes the one remaining slot, child 20 of root 10 (-1.5).
    t2 = tb.build_tree_one(vals, toks, 3, w=2)
    assert list(t2["tokens"]) == [10, 11, 20] and list(t2["parent"]) == [-1, -1, 0]
    assert t2["rounds"] == 2
    # the tree is smaller than the budget when the K-ary tree runs out: 2 + 4 nodes
    t3 = tb.build_tree_one(vals, toks, 10, w=1)
    assert t3["n"] == 6 and t3["rounds"] == 6


def read_golden():
    g = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        g[k] = [int(x) for x in v]
    return g


def test_ddtree_printed_tree_is_an_output():
    """Solve for depth-1 / depth-2 log-probs a_i, b_j (top_k = 10) whose best-first
    tree of 32 nodes is exactly the printed one; deeper draft positions get
    log-probs too low to enter.  Feasible with a clear margin => the printed
    tree is an output of this construction under the per-depth-marginal
    reading."""
    from scipy.optimize import linprog
    g = read_golden()
    parents, depths = g["parents"], g["depths"]
    N, K = 32, 10
    # rank of each node among its parent's children, in node order
    seen = {}
    rank = []
    for t in range(N):
        p = parents[t]
        rank.append(seen.get(p, 0))
        seen[p] = rank[-1] + 1
    # score of node t = a[rank(root)] (+ b[rank(child)]); variables x = [a0..a9, b0..b9, delta]
    def coeff(t):
        c = np.zeros(2 * K + 1)
        if depths[t] == 1:
            c[rank[t]] = 1
        else:
            c[rank[parents[t]]] = 1
            c[K + rank[t]] = 1
        return c
    A, b = [], []
    def ge(c1, c2):  # score1 - score2 >= delta  ->  -(c1 - c2) + delta <= 0
        row = -(c1 - c2)
        row[-1] = 1
        A.append(row)
        b.append(0.0)
    for t in range(N - 1):
        ge(coeff(t), coeff(t + 1))
    # candidates never popped (next child of every node, next root) score below the last node
    last = coeff(N - 1)
    for p, cnt in seen.items():
        if p == -1:
            continue  # all 10 roots are in the tree (top_k = 10)
        if depths[p] == 1 and cnt < K:
            c = np.zeros(2 * K + 1)
            c[rank[p]] = 1
            c[K + cnt] = 1
            ge(last, c)
    for t in range(N):
        if depths[t] == 1 and t not in seen:  # a root without children: its first child
            c = np.zeros(2 * K + 1)
            c[rank[t]] = 1
            c[K] = 1
            ge(last, c)
    for i in range(K - 1):  # each depth's top-k list is sorted
        for base in (0, K):
            c1 = np.zeros(2 * K + 1); c1[base + i] = 1
            c2 = np.zeros(2 * K + 1); c2[base + i + 1] = 1
            ge(c1, c2)
    res = linprog(c=np.r_[np.zeros(2 * K), -1.0], A_ub=np.array(A), b_ub=np.array(b),
                  bounds=[(-20, -1)] * (2 * K) + [(0, 1)], method="highs")
    assert res.status == 0
    delta = res.x[-1]
    assert delta > 1e-2
    a, bb = res.x[:K], res.x[K:2 * K]
    L = 5
    vals = np.full((L, K), -1000.0, np.float32)
    vals[0], vals[1] = a, bb
    vals[2:] = -1000.0 - np.arange(K)  # deeper positions: far below every chosen node
    toks = np.arange(L * K, dtype=np.int32).reshape(L, K)
    tree = tb.build_tree_one(vals, toks, N, w=1)
    assert list(tree["parent"]) == parents
    assert list(tree["depth"]) == depths
    check_structure(tree, toks, K)

"""CPU oracle for draft-tree construction (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this module; the product library never loads it and it imports nothing
from the product package.

Two functions, each the plain definition of what the GPU path computes:

``topk``
    The K largest entries of every row with their indices, in decreasing
    order; equal values keep the lower index first; a NaN counts as -inf.
    Written as a stable sort of the negated row (a library sort is one step).
    Source: "Tree spec-decode -> vLLM serve integration spec", "1. Proposer:
    emit top-K, not top-1" (top-W candidates per spine position) and "From
    Linear to Tree-Walk: Validating DDTree's Core Algorithm in vLLM", "The
    Thinking Process" (top_k limits the branching factor).

``build_tree``
    Best-first draft-tree construction over per-depth marginals.  Source: the
    DDTree page, "The Failed First Attempt" and "The Thinking Process": the
    top-k tokens of the first draft position are the roots; the node with the
    highest cumulative log-probability is popped from a priority queue, added
    to the tree, and its candidates are pushed back; budget of nodes and a
    maximum depth.  The batched variant of "Technische Samenvatting: Trees from
    Marginals (DFlash-TfM)", "2. Boomconstructie", pops the top w candidates
    at once and expands them together, so a tree of B nodes takes ceil(B/w)
    rounds.

    Readings (where the pages leave a step open):
      - the draft distribution is one marginal per depth (the DDTree test draws
        one logit row per draft position), given here as log-probabilities, so
        a node at depth d has the depth-(d+1) top-K tokens as its candidate
        children, and a node's score is the fp32 sum of the log-probabilities
        along its path, added in depth order;
      - the candidate heap holds every child of every expanded node (all top-K
        roots at the start); ties in score go to the candidate pushed first
        (Python heapq on (-score, push counter));
      - in the batched variant the children of a round's w nodes are pushed
        after the round, in pop order, each node's children in rank order;
      - node index = the order in which nodes are popped, so parent[t] < t;
        parent -1 = a root (a child of the last accepted token), depth 1.
    Scores are fp32 on purpose: the GPU takes the same ordering decisions in
    fp32, so the two must add the same fp32 values in the same order.
"""
from __future__ import annotations

import heapq

import numpy as np


def widen(x, dtype: str):
    """Row values as float32: 'f32' as is, 'bf16' given as uint16 bit patterns."""
    if dtype == "f32":
        return np.asarray(x, np.float32)
    if dtype == "bf16":
        bits = np.asarray(x, np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32)
    raise ValueError(dtype)


def topk(x, k: int, dtype: str = "f32"):
    """Per row: (values float32 [rows, k], indices int32 [rows, k])."""
    v = widen(x, dtype)
    v = np.where(np.isnan(v), np.float32(-np.inf), v)
    rows, V = v.shape
    if not 1 <= k <= V:
        raise ValueError("need 1 <= k <= V")
    order = np.argsort(-v, axis=1, kind="stable")[:, :k]
    vals = np.take_along_axis(v, order, axis=1)
    return vals.astype(np.float32), order.astype(np.int32)


def build_tree_one(lp_vals, lp_idx, budget: int, w: int = 1):
    """One sequence.  lp_vals float32 [L, K] (each row sorted, decreasing),
    lp_idx int32 [L, K] token ids.  Returns dict of tokens, parent, depth,
    score (length n), n and the number of rounds."""
    lp_vals = np.asarray(lp_vals, np.float32)
    L, K = lp_vals.shape
    heap = []
    counter = 0
    # a candidate: (-score, counter, depth, rank, parent node index)
    for r in range(K):
        heapq.heappush(heap, (-lp_vals[0, r], counter, 1, r, -1))
        counter += 1
    tokens, parent, depth, score = [], [], [], []
    rounds = 0
    while len(tokens) < budget and heap:
        rounds += 1
        take = min(w, budget - len(tokens))
        popped = []
        while len(popped) < take and heap:
            neg, _, d, r, p = heapq.heappop(heap)
            t = len(tokens)
            tokens.append(int(lp_idx[d - 1, r]))
            parent.append(p)
            depth.append(d)
            score.append(np.float32(-neg))
            popped.append(t)
        for t in popped:  # expand the round's nodes together, in pop order
            d = depth[t]
            if d >= L:
                continue
            for r in range(K):
                s = np.float32(score[t] + lp_vals[d, r])  # one fp32 add
                heapq.heappush(heap, (-s, counter, d + 1, r, t))
                counter += 1
    return dict(tokens=np.array(tokens, np.int32), parent=np.array(parent, np.int32),
                depth=np.array(depth, np.int32), score=np.array(score, np.float32),
                n=len(tokens), rounds=rounds)


def build_tree(lp_vals, lp_idx, budget: int, w: int = 1):
    """Batched: lp_vals float32 [B, L, K], lp_idx int32 [B, L, K].  Outputs are
    [B, budget]; slots past a sequence's node count hold token -1, parent -1,
    depth 1 and score -inf (they never match a target token)."""
    lp_vals = np.asarray(lp_vals, np.float32)
    B = lp_vals.shape[0]
    out = dict(tokens=np.full((B, budget), -1, np.int32),
               parent=np.full((B, budget), -1, np.int32),
               depth=np.ones((B, budget), np.int32),
               score=np.full((B, budget), -np.inf, np.float32),
               n_nodes=np.zeros(B, np.int32), rounds=np.zeros(B, np.int32))
    for b in range(B):
        one = build_tree_one(lp_vals[b], lp_idx[b], budget, w)
        n = one["n"]
        for k in ("tokens", "parent", "depth", "score"):
            out[k][b, :n] = one[k]
        out["n_nodes"][b] = n
        out["rounds"][b] = one["rounds"]
    return out

"""Seeded synthetic inputs for the tree-verify step.

This module builds inputs only: draft trees (host, numpy PCG64), bulk tensors
(``torch.Generator`` on the requested device), block tables and planted logits.
It holds none of the verify step's arithmetic (no masks, attention, argmax,
walk or commit) and serves both the CUDA path and the CPU oracle, which receive
the same bytes.

Workloads (B = batch, N = tree nodes, Hq/Hkv/D = heads and head dim, V = vocab;
paged KV block of 16 tokens; Q/K/V drawn N(0,1) in fp32 then cast to bf16):

  tiny          B=1,  ctx 64,            4/2/64,   N=8 root+spine+siblings, V=1024 fp32 logits
  leaf_sibling  B=1,  ctx 4096,          16/8/256, N=16 (4 depths x 4 candidates), V=262144 bf16 sd 2
  best_first    B=8,  ctx U[1024,8192],  32/8/128, N=32 heap-built (Dirichlet(0.3) top-4), V=151936
  window        B=16, ctx 32768,         32/8/128, N=32 random (depth <= 10), V=151936, window (512,0)
  stress        B=64, ctx 16384,         32/8/128, N=32 random (depth <= 8), shuffled block tables, V=151936

Each workload's default seed is ``1000 + index``.
"""
from __future__ import annotations

import dataclasses
import heapq
import math
from typing import Optional

import numpy as np
import torch

BLOCK = 16          # paged-KV block size (tokens)
PLANT = 64.0        # planted logit, in units of the logits' standard deviation
MASK64 = (1 << 64) - 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    ctx: object            # int, or (lo, hi) for per-sequence uniform lengths
    Hq: int
    Hkv: int
    D: int
    N: int
    tree: str              # tiny | leaf_sibling | best_first | random
    max_depth: int
    V: int
    logits_dtype: str      # f32 | bf16
    logits_sd: float
    window_left: int = -1  # -1 = global attention
    shuffle_blocks: bool = False
    spare_blocks: int = 0  # extra blocks per sequence beyond ctx + max_depth

    @property
    def seed(self) -> int:
        return 1000 + self.index


WORKLOADS = {
    "tiny": Workload("tiny", 0, 1, 64, 4, 2, 64, 8, "tiny", 5, 1024, "f32", 1.0),
    "leaf_sibling": Workload("leaf_sibling", 1, 1, 4096, 16, 8, 256, 16, "leaf_sibling", 4,
                             262144, "bf16", 2.0),
    "best_first": Workload("best_first", 2, 8, (1024, 8192), 32, 8, 128, 32, "best_first", 8,
                           151936, "bf16", 1.0),
    "window": Workload("window", 3, 16, 32768, 32, 8, 128, 32, "random", 10, 151936, "bf16",
                       1.0, window_left=512),
    "stress": Workload("stress", 4, 64, 16384, 32, 8, 128, 32, "random", 8, 151936, "bf16",
                       1.0, shuffle_blocks=True),
}
ORDER = ["tiny", "leaf_sibling", "best_first", "window", "stress"]


def get(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[ORDER[name_or_index]]
    return WORKLOADS[name_or_index]


# --------------------------------------------------------------------------- trees

def tree_tiny():
    """Root + spine of depth 4 + one sibling at each of the first three spine depths.

    Order [root, s1, x1, s2, x2, s3, x3, s4]; the root is the depth-1 node that
    carries the root prediction (the ``[last_accepted ++ spine]`` layout).
    """
    parent = np.array([-1, 0, 0, 1, 1, 3, 3, 5], np.int32)
    return parent


def tree_leaf_sibling(k_spec: int, w: int):
    """k_spec depths x w candidates, spine-first per depth.

    Every depth-d candidate is a child of the depth-(d-1) spine node (the first
    node of its group); depth-1 candidates hang off the last accepted token.
    """
    parent = []
    for d in range(k_spec):
        p = -1 if d == 0 else (d - 1) * w
        parent += [p] * w
    return np.array(parent, np.int32)


def tree_random(rng: np.random.Generator, n: int, max_depth: int):
    """parent[t] uniform in [-1, t-1], redrawn until the node's depth <= max_depth."""
    parent = np.zeros(n, np.int32)
    depth = np.zeros(n, np.int32)
    for t in range(n):
        while True:
            p = int(rng.integers(-1, t)) if t > 0 else -1
            d = 1 if p < 0 else int(depth[p]) + 1
            if d <= max_depth:
                break
        parent[t], depth[t] = p, d
    return parent


def tree_chain(n: int):
    return np.arange(-1, n - 1, dtype=np.int32)


def tree_star(n: int):
    return np.full(n, -1, np.int32)


def tree_best_first(rng: np.random.Generator, budget: int, max_depth: int, V: int,
                    top: int = 4, alpha: float = 0.3):
    """Best-first (heap) expansion on cumulative draft log-probability.

    Each expanded position draws ``top`` distinct candidate tokens with
    probabilities ~ Dirichlet(alpha), sorted high to low.  The heap holds
    (-cumulative log-prob, insertion counter); popping a candidate appends it as
    a node and pushes its own candidates while its depth < max_depth.

    Returns parent, tokens and, per node and for the root, the highest-probability
    draft candidate (used to plant the target argmax).
    """
    def draft():
        toks = rng.choice(V, size=top, replace=False).astype(np.int64)
        p = rng.dirichlet(np.full(top, alpha))
        order = np.argsort(-p, kind="stable")
        return toks[order], np.maximum(p[order], 1e-300)

    heap = []
    counter = 0
    root_toks, root_p = draft()
    for tok, p in zip(root_toks, root_p):
        heapq.heappush(heap, (-math.log(p), counter, -1, 1, int(tok)))
        counter += 1
    parent, tokens, best_child = [], [], []
    while heap and len(parent) < budget:
        neg_lp, _, par, d, tok = heapq.heappop(heap)
        idx = len(parent)
        parent.append(par)
        tokens.append(tok)
        ct, cp = draft()
        best_child.append(int(ct[0]))
        if d < max_depth:
            for tok2, p2 in zip(ct, cp):
                heapq.heappush(heap, (neg_lp - math.log(p2), counter, idx, d + 1, int(tok2)))
                counter += 1
    return (np.array(parent, np.int32), np.array(tokens, np.int32),
            np.array(best_child, np.int32), int(root_toks[0]))


def depths_of(parent):
    parent = np.asarray(parent)
    depth = np.zeros(parent.shape, np.int32)
    for t, p in enumerate(parent):
        depth[t] = 1 if p < 0 else depth[p] + 1
    return depth


# ------------------------------------------------------------------- hash target

def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & MASK64
    return x ^ (x >> 31)


class HashTarget:
    """A deterministic stand-in for a target model: next token = H(prefix).

    The prefix is summarised by a 64-bit state; appending a token mixes it in.
    """

    def __init__(self, V: int):
        self.V = V

    @staticmethod
    def extend(state: int, token: int) -> int:
        return _splitmix64(state ^ ((token + 1) * 0xD6E8FEB86659FD93 & MASK64))

    def next_token(self, state: int) -> int:
        return _splitmix64(state) % self.V

    def greedy(self, state: int, steps: int):
        """Plain greedy decoding of ``steps`` tokens from ``state``."""
        out = []
        for _ in range(steps):
            g = self.next_token(state)
            out.append(g)
            state = self.extend(state, g)
        return out


def hash_plant(rng: np.random.Generator, parent, V: int, p_correct: float, prefix_state: int,
               family: str = "random"):
    """Tokens for a tree under the hash target, plus each node's target argmax.

    family: 'random' (a node carries the greedy-correct token with probability
    p_correct, else a random one), 'all_wrong' (no node is correct), 'all_right'
    (every node correct), 'adversarial' (siblings get decoy tokens; the correct
    child, if any, is the highest-index sibling; some decoys duplicate the correct
    token at a lower index).

    Returns tokens[N], argmax[N] (= H(path to t)), root_pred (= H(prefix)).
    """
    ht = HashTarget(V)
    parent = np.asarray(parent)
    N = len(parent)
    state = np.zeros(N, dtype=object)
    tokens = np.zeros(N, np.int32)
    kids = {}
    for t in range(N):
        kids.setdefault(int(parent[t]), []).append(t)
    for t in range(N):
        p = int(parent[t])
        pst = prefix_state if p < 0 else state[p]
        good = ht.next_token(pst)
        if family == "all_right":
            tok = good
        elif family == "all_wrong":
            tok = int(rng.integers(0, V))
            while tok == good:
                tok = int(rng.integers(0, V))
        elif family == "adversarial":
            sib = kids[p]
            last = sib[-1] == t
            if last:
                tok = good if rng.random() < p_correct else int(rng.integers(0, V))
            else:
                tok = good if rng.random() < 0.25 else int(rng.integers(0, V))
        else:
            tok = good if rng.random() < p_correct else int(rng.integers(0, V))
        tokens[t] = tok
        state[t] = ht.extend(pst, tok)
    argmax = np.array([ht.next_token(s) for s in state], np.int32)
    return tokens, argmax, ht.next_token(prefix_state)


# ------------------------------------------------------------------- bulk tensors

def _randn_bf16(shape, gen, device, chunk=1 << 27):
    """N(0,1) drawn in fp32, cast to bf16, generated in chunks to bound memory."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, device=device,
                               dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def _ctx_lengths(w: Workload, rng):
    if isinstance(w.ctx, tuple):
        lo, hi = w.ctx
        return rng.integers(lo, hi + 1, size=w.B).astype(np.int32)
    return np.full(w.B, w.ctx, np.int32)


def block_tables(rng, ctx, extra_tokens: int, spare: int, shuffle: bool):
    """Per-sequence block lists covering ctx + extra_tokens positions (+ spare blocks).

    Unused slots hold -1.  With ``shuffle`` the physical block ids are a random
    permutation of the whole pool, else sequences own consecutive ranges.
    """
    B = len(ctx)
    need = [-(-int(c + extra_tokens) // BLOCK) + spare for c in ctx]
    max_blocks = max(need) if need else 1
    total = int(sum(need))
    ids = rng.permutation(total).astype(np.int32) if shuffle else np.arange(total, dtype=np.int32)
    table = np.full((B, max_blocks), -1, np.int32)
    o = 0
    for b in range(B):
        table[b, :need[b]] = ids[o:o + need[b]]
        o += need[b]
    return table, total


def make(workload, device="cpu", seed: Optional[int] = None, *, B: Optional[int] = None,
         ctx=None, N: Optional[int] = None, tree: Optional[str] = None,
         plant: Optional[str] = None, p_correct: float = 0.5, window_left=None,
         shuffle_blocks=None, V: Optional[int] = None):
    """Build one batch of verify-step inputs.

    ``workload`` is a name or index from ``WORKLOADS``; keyword overrides give
    smaller or structurally different variants (tests).  ``plant``:
      None          the workload's own rule (tiny: tokens[0] = root_pred;
                    leaf_sibling: spine token is the argmax with p=0.7 per depth;
                    best_first: the node's top draft child with p=0.6; random
                    trees: nothing planted),
      'hash'        tokens and argmax rows from the hash target
                    (``hash_plant(..., family='random')``),
      'hash:<fam>'  the same with another family,
      'path'        one random root-to-leaf path made greedy-correct (ours: it
                    makes random-logit workloads accept at full depth).
    Returns a dict of tensors plus shape metadata.
    """
    w = get(workload)
    seed = w.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    B = w.B if B is None else B
    N = w.N if N is None else N
    V = w.V if V is None else V
    tree = w.tree if tree is None else tree
    wl = w.window_left if window_left is None else window_left
    shuffle = w.shuffle_blocks if shuffle_blocks is None else shuffle_blocks
    if ctx is None:
        ctx_len = _ctx_lengths(dataclasses.replace(w, B=B), rng)
    elif isinstance(ctx, tuple):
        ctx_len = rng.integers(ctx[0], ctx[1] + 1, size=B).astype(np.int32)
    else:
        ctx_len = np.full(B, int(ctx), np.int32)

    parent = np.zeros((B, N), np.int32)
    tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
    root_pred = rng.integers(0, V, size=B).astype(np.int32)
    plant_rows = {}            # (b, t) -> planted argmax token
    best_child = None
    for b in range(B):
        if tree == "tiny":
            par = tree_tiny()[:N] if N <= 8 else tree_random(rng, N, w.max_depth)
        elif tree == "leaf_sibling":
            par = tree_leaf_sibling(w.max_depth, max(1, N // w.max_depth))[:N]
        elif tree == "best_first":
            par, tok, bc, root_best = tree_best_first(rng, N, w.max_depth, V)
            if len(par) < N:
                raise ValueError("best-first heap ran dry before the budget")
            tokens[b] = tok
            if plant is None:
                for t in range(N):
                    if rng.random() < 0.6:
                        plant_rows[(b, t)] = int(bc[t])
                if rng.random() < 0.6:
                    root_pred[b] = root_best
        elif tree == "chain":
            par = tree_chain(N)
        elif tree == "star":
            par = tree_star(N)
        else:
            par = tree_random(rng, N, w.max_depth)
        parent[b] = par
        if plant is None and tree == "tiny" and N > 0:
            tokens[b, 0] = root_pred[b]
        if plant is None and tree == "leaf_sibling":
            Wd = max(1, N // w.max_depth)
            for d in range(w.max_depth):
                if d * Wd >= N or rng.random() >= 0.7:
                    continue
                spine_tok = int(tokens[b, d * Wd])
                if d == 0:
                    root_pred[b] = spine_tok
                else:
                    plant_rows[(b, (d - 1) * Wd)] = spine_tok
        if plant is not None and plant.startswith("hash"):
            fam = plant.split(":", 1)[1] if ":" in plant else "random"
            prefix_state = int(rng.integers(0, 1 << 63))
            tok, am, rp = hash_plant(rng, par, V, p_correct, prefix_state, fam)
            tokens[b], root_pred[b] = tok, rp
            for t in range(N):
                plant_rows[(b, t)] = int(am[t])
        if plant == "path" and N > 0:
            # one random root-to-leaf path made greedy-correct
            leaf = int(rng.integers(0, N))
            path = []
            t = leaf
            while t >= 0:
                path.append(t)
                t = int(par[t])
            path.reverse()
            root_pred[b] = tokens[b, path[0]]
            for a, c in zip(path[:-1], path[1:]):
                plant_rows[(b, a)] = int(tokens[b, c])
    depth = np.stack([depths_of(parent[b]) for b in range(B)]) if B else np.zeros((0, N), np.int32)
    max_depth = int(depth.max()) if depth.size else 0
    table, num_blocks = block_tables(rng, ctx_len, max(max_depth, 1), w.spare_blocks, shuffle)

    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    q = _randn_bf16((B, N, w.Hq, w.D), gen, dev)
    k_tree = _randn_bf16((B, N, w.Hkv, w.D), gen, dev)
    v_tree = _randn_bf16((B, N, w.Hkv, w.D), gen, dev)
    k_cache = _randn_bf16((num_blocks, w.Hkv, BLOCK, w.D), gen, dev)
    v_cache = _randn_bf16((num_blocks, w.Hkv, BLOCK, w.D), gen, dev)
    ldt = torch.float32 if w.logits_dtype == "f32" else torch.bfloat16
    logits = torch.empty((B, N, V), dtype=ldt, device=dev)
    flat = logits.view(-1)
    chunk = 1 << 27
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        flat[s:e] = (torch.randn(e - s, generator=gen, device=dev, dtype=torch.float32)
                     * w.logits_sd).to(ldt)
    if plant_rows:
        keys = sorted(plant_rows)
        bi = torch.tensor([k[0] for k in keys], dtype=torch.long, device=dev)
        ti = torch.tensor([k[1] for k in keys], dtype=torch.long, device=dev)
        vi = torch.tensor([plant_rows[k] for k in keys], dtype=torch.long, device=dev)
        logits[bi, ti, vi] = PLANT * w.logits_sd

    it = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    return dict(
        workload=w.name, B=B, N=N, Hq=w.Hq, Hkv=w.Hkv, D=w.D, V=V, block_size=BLOCK,
        window_left=int(wl), num_blocks=num_blocks, max_blocks=table.shape[1],
        logits_dtype=w.logits_dtype,
        tokens=it(tokens), parent=it(parent), depth=it(depth), ctx_len=it(ctx_len),
        root_pred=it(root_pred), block_table=it(table),
        q=q, k_tree=k_tree, v_tree=v_tree, k_cache=k_cache, v_cache=v_cache, logits=logits,
    )


def to_numpy(inp):
    """Host copies of every tensor; bf16 tensors become their uint16 bit patterns."""
    out = {}
    for k, v in inp.items():
        if isinstance(v, torch.Tensor):
            v = v.detach().cpu()
            if v.dtype == torch.bfloat16:
                v = v.view(torch.int16).numpy().view(np.uint16)
            else:
                v = v.numpy()
        out[k] = v
    return out


def kv_bytes(inp) -> int:
    """Context K+V bytes the attention must read (per-row window union)."""
    ctx = inp["ctx_len"].detach().cpu().numpy().astype(np.int64)
    wl = inp["window_left"]
    if wl >= 0:
        # rows sit at positions ctx .. ctx-1+maxdepth; the union of their windows
        # starts at ctx - wl (the shallowest row)
        vis = np.minimum(ctx, wl)
    else:
        vis = ctx
    return int(vis.sum()) * inp["Hkv"] * inp["D"] * 2 * 2


# --------------------------------------------------------------------------- draft side

@dataclasses.dataclass(frozen=True)
class DraftWorkload:
    """Draft-tree construction inputs: per-position draft log-probabilities."""
    name: str
    seed: int
    B: int        # sequences
    L: int        # draft positions (maximum tree depth)
    V: int        # vocabulary
    K: int        # candidates per position (top_k)
    budget: int   # tree nodes
    w: int = 1    # nodes popped per round


DRAFT_WORKLOADS = {
    # DDTree construction (top_k 10, 32-node budget) at the stress batch, depth <= 8
    "tree_build": DraftWorkload("tree_build", 2000, 64, 8, 151936, 10, 32, 1),
    # batched top-w rounds of the same shape
    "tree_build_w4": DraftWorkload("tree_build_w4", 2001, 64, 8, 151936, 10, 32, 4),
    # leaf-sibling proposer: top-4 per spine position over a 262144-token vocab
    "top_w": DraftWorkload("top_w", 2002, 1, 4, 262144, 4, 16, 1),
}


def make_draft(name, device="cpu", seed: Optional[int] = None, *, B: Optional[int] = None,
               L: Optional[int] = None, V: Optional[int] = None, quantum: float = 0.0,
               dtype=torch.float32):
    """Draft log-probabilities [B, L, V]: log-softmax of N(0, 1) logits drawn on
    ``device`` (the drafter's output; the tree construction starts from it).
    ``quantum`` > 0 rounds the logits to multiples of it first, which makes
    exactly tied log-probabilities (tests of the tie rules)."""
    w = DRAFT_WORKLOADS[name]
    seed = w.seed if seed is None else seed
    B = w.B if B is None else B
    L = w.L if L is None else L
    V = w.V if V is None else V
    gen = torch.Generator(device=device).manual_seed(seed)
    logits = torch.randn(B, L, V, generator=gen, device=device, dtype=torch.float32)
    if quantum > 0:
        logits = torch.round(logits / quantum) * quantum
    return torch.log_softmax(logits, dim=-1).to(dtype)


def make_layers(inp, num_layers: int, seed: int):
    """Per-layer tensors of an L-layer model sharing ``inp``'s tree, block
    table and logits: layer 0 is ``inp``'s own q / k_tree / v_tree / caches,
    layers 1.. are fresh N(0, 1) bf16 tensors of the same shapes (seeded)."""
    dev = inp["q"].device
    layers = [dict(q=inp["q"], k_tree=inp["k_tree"], v_tree=inp["v_tree"],
                   k_cache=inp["k_cache"], v_cache=inp["v_cache"])]
    for l in range(1, num_layers):
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed + 7777 * l)
        layers.append({k: _randn_bf16(tuple(inp[k].shape), gen, dev)
                       for k in ("q", "k_tree", "v_tree", "k_cache", "v_cache")})
    return layers


# --------------------------------------------------------------------------- GDN layers

@dataclasses.dataclass(frozen=True)
class GdnWorkload:
    """Tree verification through one Gated DeltaNet layer."""
    name: str
    seed: int
    B: int
    N: int
    max_depth: int
    Hk: int       # query / key heads
    Hv: int       # value heads (state heads)
    dk: int
    dv: int


GDN_WORKLOADS = {
    # the stress batch and trees through a GDN layer of 16 key / 32 value heads, 128 x 128 state
    "gdn_stress": GdnWorkload("gdn_stress", 3000, 64, 32, 8, 16, 32, 128, 128),
    "gdn_small": GdnWorkload("gdn_small", 3001, 3, 12, 5, 2, 4, 32, 64),
}


def make_gdn(name, device="cpu", seed: Optional[int] = None, *, B=None, N=None, tree=None,
             Hk=None, Hv=None, dk=None, dv=None):
    """Seeded inputs of one GDN tree verification: tree (parent, depth),
    L2-normalised q / k (bf16, as GDN layers normalise them), v ~ N(0, 1) bf16,
    decay alpha ~ U(0.8, 1), write strength beta = sigmoid(N(0, 1)), committed
    state S_0 ~ N(0, 0.3^2) fp32 stored transposed [B, Hv, dv, dk]."""
    w = GDN_WORKLOADS[name]
    seed = w.seed if seed is None else seed
    B = w.B if B is None else B
    N = w.N if N is None else N
    Hk = w.Hk if Hk is None else Hk
    Hv = w.Hv if Hv is None else Hv
    dk = w.dk if dk is None else dk
    dv = w.dv if dv is None else dv
    rng = np.random.Generator(np.random.PCG64(seed))
    parent = np.zeros((B, N), np.int32)
    for b in range(B):
        if tree == "chain":
            parent[b] = tree_chain(N)
        elif tree == "star":
            parent[b] = tree_star(N)
        else:
            parent[b] = tree_random(rng, N, w.max_depth)
    depth = np.stack([depths_of(parent[b]) for b in range(B)])
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    q = torch.randn(B, N, Hk, dk, generator=gen, device=dev)
    k = torch.randn(B, N, Hk, dk, generator=gen, device=dev)
    q = (q / q.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    v = torch.randn(B, N, Hv, dv, generator=gen, device=dev).to(torch.bfloat16)
    alpha = 0.8 + 0.2 * torch.rand(B, N, Hv, generator=gen, device=dev)
    beta = torch.sigmoid(torch.randn(B, N, Hv, generator=gen, device=dev))
    state = 0.3 * torch.randn(B, Hv, dv, dk, generator=gen, device=dev)
    it = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    return dict(B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, parent=it(parent), depth=it(depth),
                q=q, k=k, v=v, alpha=alpha.float(), beta=beta.float(), state=state.float())

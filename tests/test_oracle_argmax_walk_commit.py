"""Pins for the oracle's argmax, greedy tree walk and KV commit (CPU only).

Walk rule: "Tree spec-decode -> vLLM serve integration spec", "What's proven"
and "3. Rejection sampler": from the root follow the child whose token equals
the target argmax of its parent, then emit the bonus argmax.  The page's claim
that the accepted sequence equals plain greedy decoding for ANY tree is the pin:
a hash-defined target gives a greedy decode computed without any tree.
"""
import zlib

import numpy as np
import pytest

import workloads
from workloads import HashTarget

from test_oracle_ancestors import read_golden


# ------------------------------------------------------------------- argmax

def np_first_argmax(x):
    x = np.where(np.isnan(x), -np.inf, x)
    return np.argmax(x, axis=1)


@pytest.mark.parametrize("V", [1, 7, 1000, 4099])
def test_argmax_random_f32(oracle_mod, V):
    rng = np.random.Generator(np.random.PCG64(V))
    x = rng.standard_normal((13, V)).astype(np.float32)
    assert np.array_equal(oracle_mod.argmax(x, "f32"), np_first_argmax(x))


def to_bf16_bits(x):
    u = np.asarray(x, np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16)   # truncation: exact for values that fit bf16


def test_argmax_bf16_ties_lowest_index(oracle_mod):
    rng = np.random.Generator(np.random.PCG64(1))
    x = np.round(rng.standard_normal((20, 3001)) * 4) / 4   # coarse grid -> many ties
    x = x.astype(np.float32)
    bits = to_bf16_bits(x)
    got = oracle_mod.argmax(bits, "bf16")
    assert np.array_equal(got, np_first_argmax(x))
    # planted ties at several indices: the lowest wins
    y = np.zeros((4, 5000), np.float32)
    for r, idx in enumerate([[4999, 3, 17], [2, 1], [0, 4999], [2500, 2501, 1024]]):
        y[r, idx] = 9.0
    assert list(oracle_mod.argmax(to_bf16_bits(y), "bf16")) == [3, 1, 0, 1024]


def test_argmax_signed_zero_and_nan(oracle_mod):
    x = np.array([[-1.0, -0.0, 0.0, -2.0],
                  [np.nan, 1.0, 2.0, np.nan],
                  [-np.inf, -np.inf, -np.inf, -np.inf],
                  [np.nan, np.nan, np.nan, np.nan],
                  [0.0, -0.0, 0.0, -0.0]], np.float32)
    assert list(oracle_mod.argmax(x, "f32")) == [1, 2, 0, 0, 0]
    assert list(oracle_mod.argmax(to_bf16_bits(x), "bf16")) == [1, 2, 0, 0, 0]


# ------------------------------------------------------------------- walk

def brute_max_accept(parent, tokens, prefix_state, V):
    """Longest root path whose every token is greedy-correct, by enumerating nodes."""
    ht = HashTarget(V)
    best = 0
    for t in range(len(parent)):
        path = []
        a = t
        while a >= 0:
            path.append(a)
            a = int(parent[a])
        path.reverse()
        st = prefix_state
        ok = True
        for a in path:
            if tokens[a] != ht.next_token(st):
                ok = False
                break
            st = ht.extend(st, int(tokens[a]))
        if ok:
            best = max(best, len(path))
    return best


def unique_sibling_tokens(parent, tokens):
    seen = set()
    for p, t in zip(parent, tokens):
        if (int(p), int(t)) in seen:
            return False
        seen.add((int(p), int(t)))
    return True


FAMILIES = ["random", "adversarial", "all_wrong", "all_right"]


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("shape", ["random", "chain", "star", "leaf_sibling", "best_first"])
def test_greedy_identity_and_maximality(oracle_mod, family, shape):
    rng = np.random.Generator(np.random.PCG64(zlib.crc32(f"{family}/{shape}".encode())))
    V = 50  # small vocabulary: duplicate-token siblings happen often
    for trial in range(30):
        N = int(rng.integers(1, 33))
        if shape == "random":
            par = workloads.tree_random(rng, N, 8)
        elif shape == "chain":
            par = workloads.tree_chain(N)
        elif shape == "star":
            par = workloads.tree_star(N)
        elif shape == "leaf_sibling":
            par = workloads.tree_leaf_sibling(4, 4)
            N = 16
        else:
            par = workloads.tree_best_first(rng, N, 8, V)[0]
        prefix = int(rng.integers(0, 1 << 62))
        tokens, am, root_pred = workloads.hash_plant(rng, par, V, 0.6, prefix, family)
        ot, ne, an, na = oracle_mod.walk(tokens[None], par[None], am[None],
                                         np.array([root_pred]))
        n = int(ne[0])
        greedy = HashTarget(V).greedy(prefix, n)
        assert list(ot[0, :n]) == greedy, (family, shape, trial)
        assert n == int(na[0]) + 1
        # maximality holds when siblings carry distinct tokens (the page's "unique
        # child"); with duplicate-token siblings the lowest index is followed, which
        # keeps greedy identity but may stop short of a deeper duplicate's subtree
        best = brute_max_accept(par, tokens, prefix, V)
        if unique_sibling_tokens(par, tokens):
            assert int(na[0]) == best
        else:
            assert int(na[0]) <= best
        assert (ot[0, n:] == -1).all() and (an[0, int(na[0]):] == -1).all()
        # accepted nodes form a root path with matching tokens
        path = an[0, :int(na[0])]
        for i, c in enumerate(path):
            assert par[c] == (-1 if i == 0 else path[i - 1])
            assert tokens[c] == ot[0, i]
        if family == "all_wrong":
            assert n == 1 and ot[0, 0] == root_pred
        if family == "all_right" and shape == "chain":
            assert n == N + 1


def test_duplicate_siblings_take_lowest_index(oracle_mod):
    par = np.array([-1, -1, -1, 0, 2], np.int32)
    tok = np.array([5, 7, 5, 9, 9], np.int32)
    am = np.array([9, 0, 9, 1, 2], np.int32)
    ot, ne, an, na = oracle_mod.walk(tok[None], par[None], am[None], np.array([5]))
    assert list(an[0, :na[0]]) == [0, 3] and list(ot[0, :ne[0]]) == [5, 9, 1]


def test_bad_status_emits_root_prediction_only(oracle_mod):
    par = workloads.tree_chain(4)
    tok = np.array([3, 4, 5, 6], np.int32)
    am = np.array([4, 5, 6, 7], np.int32)
    ot, ne, an, na = oracle_mod.walk(np.stack([tok, tok]), np.stack([par, par]),
                                     np.stack([am, am]), np.array([3, 3]),
                                     status=np.array([0, 2]))
    assert list(ot[0, :ne[0]]) == [3, 4, 5, 6, 7]
    assert ne[1] == 1 and ot[1, 0] == 3 and na[1] == 0


def test_cyclic_parents_terminate(oracle_mod):
    par = np.array([-1, 2, 1, 0], np.int32)   # nodes 1 and 2 point at each other
    tok = np.array([1, 1, 1, 1], np.int32)
    am = np.array([1, 1, 1, 1], np.int32)
    ot, ne, an, na = oracle_mod.walk(tok[None], par[None], am[None], np.array([1]))
    assert 1 <= ne[0] <= 5


def test_ddtree_printed_output_is_reachable(oracle_mod):
    """Consistency with the DDTree page's printed run (structure only).

    The page prints an accepted list of two tokens, both 701, for its tree; its
    logits are not printed, so the values cannot be reproduced.  Under this library's
    reading (root prediction = 701 matches node 0, whose own argmax 701 matches
    none of its children) the walk emits exactly that list: one accepted node
    plus the bonus token.
    """
    g = read_golden()
    par = np.array(g["parents"], np.int32)
    tok = np.full(32, 1, np.int32)
    tok[:10] = g["tokens_first10"]
    am = np.zeros(32, np.int32)
    am[0] = 701
    ot, ne, an, na = oracle_mod.walk(tok[None], par[None], am[None], np.array([701]))
    assert list(ot[0, :ne[0]]) == g["accepted"]


# ------------------------------------------------------------------- commit

def gather_sequence(cache, table, b, length):
    j = np.arange(length)
    return cache[table[b, j // 16], :, j % 16, :]


@pytest.mark.parametrize("shuffle", [False, True])
def test_commit_every_accept_length(oracle_mod, shuffle):
    inp = workloads.to_numpy(workloads.make("tiny", "cpu", 9, B=6, ctx=(17, 70), N=12,
                                            tree="chain", shuffle_blocks=shuffle, V=64))
    B, N = inp["tokens"].shape
    rng = np.random.Generator(np.random.PCG64(2))
    for trial in range(3):
        n_acc = np.array([min(b + trial * 2, N) for b in range(B)], np.int32)  # 0..N
        acc = np.full((B, N), -1, np.int32)
        for b in range(B):
            acc[b, :n_acc[b]] = np.arange(n_acc[b])   # a chain accepts a prefix
        kc, vc, ctx_out, st = oracle_mod.commit(inp["k_tree"], inp["v_tree"], acc, n_acc,
                                                inp["ctx_len"], inp["block_table"],
                                                inp["k_cache"], inp["v_cache"])
        assert (st == 0).all()
        assert np.array_equal(ctx_out, inp["ctx_len"] + n_acc)
        changed = np.zeros(kc.shape[:1] + kc.shape[2:3], bool)   # [block, row]
        for b in range(B):
            ctx = int(inp["ctx_len"][b])
            for cache_new, cache_old, tree in ((kc, inp["k_cache"], inp["k_tree"]),
                                               (vc, inp["v_cache"], inp["v_tree"])):
                seq = gather_sequence(cache_new, inp["block_table"], b, ctx_out[b])
                old = gather_sequence(cache_old, inp["block_table"], b, ctx)
                assert np.array_equal(seq[:ctx], old)
                assert np.array_equal(seq[ctx:], tree[b, acc[b, :n_acc[b]]])
            j = np.arange(ctx, ctx_out[b])
            changed[inp["block_table"][b, j // 16], j % 16] = True
        # every other (block, row) is bitwise untouched
        keep = ~changed
        assert np.array_equal(kc.transpose(0, 2, 1, 3)[keep],
                              inp["k_cache"].transpose(0, 2, 1, 3)[keep])
        assert np.array_equal(vc.transpose(0, 2, 1, 3)[keep],
                              inp["v_cache"].transpose(0, 2, 1, 3)[keep])


def test_commit_bad_block_commits_nothing(oracle_mod):
    inp = workloads.to_numpy(workloads.make("tiny", "cpu", 4, B=3, ctx=(31, 31), N=4,
                                            tree="chain", V=64))
    n_acc = np.array([4, 4, 4], np.int32)
    acc = np.tile(np.arange(4, dtype=np.int32), (3, 1))
    bt = inp["block_table"].copy()
    bt[1, 2] = inp["k_cache"].shape[0]      # out of range block id at position 32
    bt[2, 2:] = -1                          # missing slot
    kc, vc, ctx_out, st = oracle_mod.commit(inp["k_tree"], inp["v_tree"], acc, n_acc,
                                            inp["ctx_len"], bt, inp["k_cache"], inp["v_cache"])
    assert list(st) == [0, 3, 3]
    assert list(ctx_out) == [35, 31, 31]
    # sequences 1 and 2 left everything alone
    for b in (1, 2):
        blocks = [x for x in bt[b] if 0 <= x < inp["k_cache"].shape[0]]
        assert np.array_equal(kc[blocks], inp["k_cache"][blocks])


def test_generators_give_valid_trees(oracle_mod):
    for name in ("tiny", "leaf_sibling", "best_first"):
        w = workloads.get(name)
        inp = workloads.make(name, "cpu", B=min(w.B, 3), ctx=100, V=1000)
        _, _, st = oracle_mod.ancestors(inp["parent"].numpy(), inp["depth"].numpy(),
                                        inp["ctx_len"].numpy())
        assert (st == 0).all()
        assert int(inp["depth"].max()) <= w.max_depth

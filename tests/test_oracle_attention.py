"""Pins for the oracle's fp64 tree attention (CPU only).

"Tree spec-decode -> vLLM serve integration spec", "2. Verify": every node
attends the whole paged context plus its ancestors and itself, composed with a
sliding window.  The oracle's loops are checked against float64
``torch.nn.functional.scaled_dot_product_attention`` (a library routine) given a
dense boolean mask built here from key positions and a transitive closure,
plus the special cases that reduce to textbook attention: a chain tree is causal
attention over context ++ chain, a star tree is N independent decodes.
"""
import numpy as np
import pytest
import torch

import workloads
from test_oracle_ancestors import closure_mask


def bf(a):
    """uint16 bf16 bit patterns -> float64 tensor (exact)."""
    return torch.from_numpy((a.astype(np.uint32) << 16).view(np.float32).astype(np.float64))


def dense_keys(inp, b):
    """Context keys/values of sequence b gathered densely through the block table."""
    ctx = int(inp["ctx_len"][b])
    j = np.arange(ctx)
    blk = inp["block_table"][b, j // 16]
    K = inp["k_cache"][blk, :, j % 16, :]          # [ctx, Hkv, D]
    Vv = inp["v_cache"][blk, :, j % 16, :]
    return K, Vv


def sdpa_reference(inp, window_left=-1):
    """Library SDPA per sequence with an explicit [N, ctx+N] boolean mask."""
    B, N, Hq, D = inp["q"].shape
    Hkv = inp["k_tree"].shape[2]
    G = Hq // Hkv
    out = np.zeros((B, N, Hq, D))
    for b in range(B):
        ctx = int(inp["ctx_len"][b])
        K, Vv = dense_keys(inp, b)
        Kall = np.concatenate([K, inp["k_tree"][b]], 0)          # [S, Hkv, D]
        Vall = np.concatenate([Vv, inp["v_tree"][b]], 0)
        depth = workloads.depths_of(inp["parent"][b])
        qpos = ctx - 1 + depth
        kpos = np.concatenate([np.arange(ctx), qpos])
        allowed = np.concatenate([np.ones((N, ctx), bool), closure_mask(inp["parent"][b])], 1)
        if window_left >= 0:
            allowed &= kpos[None, :] >= (qpos[:, None] - window_left)
        Q = bf(inp["q"][b]).permute(1, 0, 2)                        # [Hq, N, D]
        Kt = bf(Kall).permute(1, 0, 2).repeat_interleave(G, 0)      # [Hq, S, D]
        Vt = bf(Vall).permute(1, 0, 2).repeat_interleave(G, 0)
        o = torch.nn.functional.scaled_dot_product_attention(
            Q, Kt, Vt, attn_mask=torch.from_numpy(allowed))
        out[b] = o.permute(1, 0, 2).numpy()
    return out


def run_oracle(oracle_mod, inp, window_left=-1, row_sel=None):
    mask, pos, st = oracle_mod.ancestors(inp["parent"], inp["depth"], inp["ctx_len"])
    assert (st == 0).all()
    return oracle_mod.attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"],
                                inp["v_cache"], inp["block_table"], inp["ctx_len"], mask, pos,
                                window_left=window_left, row_sel=row_sel)


def small(tree, seed=5, B=2, ctx=(37, 75), N=9, window_left=-1, shuffle=True):
    return workloads.to_numpy(workloads.make("tiny", "cpu", seed, B=B, ctx=ctx, N=N, tree=tree,
                                             window_left=window_left, shuffle_blocks=shuffle,
                                             V=64))


@pytest.mark.parametrize("tree", ["random", "chain", "star", "tiny"])
def test_against_library_sdpa(oracle_mod, tree):
    inp = small(tree, N=8 if tree == "tiny" else 11)
    ref = sdpa_reference(inp)
    got = run_oracle(oracle_mod, inp)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_chain_is_causal_over_context_plus_chain(oracle_mod):
    """A chain tree is plain causal attention over the concatenated sequence."""
    inp = small("chain", B=1, ctx=(50, 50), N=7)
    ctx, N = 50, 7
    K, Vv = dense_keys(inp, 0)
    Kall = bf(np.concatenate([K, inp["k_tree"][0]], 0)).permute(1, 0, 2)
    Vall = bf(np.concatenate([Vv, inp["v_tree"][0]], 0)).permute(1, 0, 2)
    Hq, Hkv = inp["q"].shape[2], Kall.shape[0]
    G = Hq // Hkv
    Q = torch.zeros(Hq, ctx + N, Kall.shape[2], dtype=torch.float64)
    Q[:, ctx:] = bf(inp["q"][0]).permute(1, 0, 2)   # only the last N rows are checked
    o = torch.nn.functional.scaled_dot_product_attention(
        Q, Kall.repeat_interleave(G, 0), Vall.repeat_interleave(G, 0), is_causal=True)
    ref = o[:, ctx:].permute(1, 0, 2).numpy()
    got = run_oracle(oracle_mod, inp)[0]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_star_is_independent_decodes(oracle_mod):
    inp = small("star", B=1, ctx=(40, 40), N=6)
    K, Vv = dense_keys(inp, 0)
    Hq, Hkv = inp["q"].shape[2], K.shape[1]
    got = run_oracle(oracle_mod, inp)[0]
    for t in range(6):
        Kt = bf(np.concatenate([K, inp["k_tree"][0, t:t + 1]], 0)).permute(1, 0, 2)
        Vt = bf(np.concatenate([Vv, inp["v_tree"][0, t:t + 1]], 0)).permute(1, 0, 2)
        q = bf(inp["q"][0, t])[:, None, :]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, Kt.repeat_interleave(Hq // Hkv, 0), Vt.repeat_interleave(Hq // Hkv, 0))
        np.testing.assert_allclose(got[t], o[:, 0].numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("wl", [0, 1, 3, 20, 45])
def test_window_against_library_sdpa(oracle_mod, wl):
    inp = small("random", B=2, ctx=(30, 61), N=12, window_left=wl)
    ref = sdpa_reference(inp, window_left=wl)
    got = run_oracle(oracle_mod, inp, window_left=wl)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_wide_window_equals_global(oracle_mod):
    inp = small("random", ctx=(30, 61), N=10)
    span = int(inp["ctx_len"].max()) + 10
    a = run_oracle(oracle_mod, inp, window_left=span)
    g = run_oracle(oracle_mod, inp, window_left=-1)
    assert np.array_equal(a, g)


def test_block_permutation_invariance(oracle_mod):
    inp = small("random", shuffle=False)
    a = run_oracle(oracle_mod, inp)
    rng = np.random.Generator(np.random.PCG64(11))
    perm = rng.permutation(inp["k_cache"].shape[0])
    inv = np.argsort(perm)
    inp2 = dict(inp)
    inp2["k_cache"] = inp["k_cache"][perm]
    inp2["v_cache"] = inp["v_cache"][perm]
    bt = inp["block_table"].copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    inp2["block_table"] = bt
    b = run_oracle(oracle_mod, inp2)
    assert np.array_equal(a, b)


def test_row_selection(oracle_mod):
    inp = small("random")
    full = run_oracle(oracle_mod, inp)
    B, Hq = inp["q"].shape[0], inp["q"].shape[2]
    sel = np.zeros((B, Hq), bool)
    sel[1, 2] = True
    part = run_oracle(oracle_mod, inp, row_sel=sel)
    assert np.array_equal(part[1, :, 2], full[1, :, 2])
    assert np.isnan(part[0]).all()


def test_single_node_is_plain_decode(oracle_mod):
    inp = small("star", B=1, ctx=(33, 33), N=1)
    ref = sdpa_reference(inp)
    np.testing.assert_allclose(run_oracle(oracle_mod, inp), ref, rtol=1e-12, atol=1e-12)


def test_mutation_swapped_kv_is_caught(oracle_mod):
    """A plausible bug (K and V swapped) is far outside the pinned tolerance."""
    inp = small("random")
    ref = sdpa_reference(inp)
    inp2 = dict(inp)
    inp2["k_cache"], inp2["v_cache"] = inp["v_cache"], inp["k_cache"]
    got = run_oracle(oracle_mod, inp2)
    assert np.abs(got - ref).max() > 1e-3

"""Shared glue for the GPU parity tests: run the CUDA path, run the oracle on the
same bytes (or on a sampled subset of sequences / heads), compare."""
import numpy as np
import torch

import oracle
import workloads

ATOL, RTOL = 2e-2, 1e-2   # |gpu - ref| <= ATOL + RTOL * |ref|  (bf16 in, fp32 accumulate)


def step_for(inp, num_splits=0):
    import tree_speculative_decoding_build_gb300 as tv
    return tv.VerifyStep(inp["B"], inp["N"], inp["Hq"], inp["Hkv"], inp["D"], inp["V"],
                         inp["max_blocks"], window_left=inp["window_left"],
                         logits_dtype=inp["logits_dtype"], num_splits=num_splits,
                         device=inp["q"].device)


def bf16_to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def subset_numpy(inp, seqs):
    """Host copy of sequences ``seqs`` with only the cache blocks they reference.

    Block ids are remapped to the compacted cache; -1 slots stay -1.
    """
    seqs = torch.as_tensor(seqs, dtype=torch.long, device=inp["q"].device)
    bt = inp["block_table"].index_select(0, seqs)
    used = torch.unique(bt[bt >= 0])
    remap = torch.full((inp["num_blocks"],), -1, dtype=torch.int32, device=bt.device)
    remap[used] = torch.arange(used.numel(), dtype=torch.int32, device=bt.device)
    bt2 = torch.where(bt >= 0, remap[bt.clamp(min=0).long()], bt)
    sub = dict(inp)
    for k in ("tokens", "parent", "depth", "ctx_len", "root_pred", "q", "k_tree", "v_tree",
              "logits"):
        sub[k] = inp[k].index_select(0, seqs)
    sub["block_table"] = bt2
    sub["k_cache"] = inp["k_cache"].index_select(0, used)
    sub["v_cache"] = inp["v_cache"].index_select(0, used)
    sub["B"] = len(seqs)
    sub["num_blocks"] = int(used.numel())
    return workloads.to_numpy(sub)


def oracle_attention(npi, head_sel=None):
    mask, pos, st = oracle.ancestors(npi["parent"], npi["depth"], npi["ctx_len"])
    row_sel = None
    if head_sel is not None:
        B, Hq = npi["q"].shape[0], npi["q"].shape[2]
        row_sel = np.zeros((B, Hq), bool)
        row_sel[:, head_sel] = True
    return oracle.attention(npi["q"], npi["k_tree"], npi["v_tree"], npi["k_cache"],
                            npi["v_cache"], npi["block_table"], npi["ctx_len"], mask, pos,
                            window_left=npi["window_left"], row_sel=row_sel)


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max err {err.max():.3e}")


def run_attention(tv, inp, num_splits=0, window_left=None, kernel=0):
    B, N = inp["B"], inp["N"]
    wl = inp["window_left"] if window_left is None else window_left
    anc = torch.empty((B, N), dtype=torch.int64, device="cuda")
    pos = torch.empty((B, N), dtype=torch.int32, device="cuda")
    st = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(inp["q"])
    tv.tv_build_ancestors(inp["parent"], inp["depth"], inp["ctx_len"], anc, pos, st)
    tv.tv_tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"], inp["v_cache"],
                         inp["block_table"], inp["ctx_len"], pos, anc, out, st, window_left=wl,
                         num_splits=num_splits, kernel=kernel)
    torch.cuda.synchronize()
    return out, st

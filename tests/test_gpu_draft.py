"""GPU parity of the draft side (tv_topk, tv_build_tree) against the oracle.

Both are integer / selection work: indices, tokens, parents and depths must match
bit for bit; the top-k values are copies of input values and the tree scores are
float32 sums both sides add in the same order, so those match bit for bit too.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import tree_build as tb

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_decoding_build_gb300 as m
    return m


def host(x, dtype):
    if dtype == "bf16":
        return x.cpu().view(torch.int16).numpy().view(np.uint16)
    return x.cpu().numpy()


def run_topk(tv, x, k):
    rows = x.shape[0]
    vals = torch.empty(rows, k, dtype=torch.float32, device="cuda")
    idx = torch.empty(rows, k, dtype=torch.int32, device="cuda")
    tv.tv_topk(x, k, vals, idx)
    return vals.cpu().numpy(), idx.cpu().numpy()


# ------------------------------------------------------------------ topk

# (16, 262144), (64, 65536), (999, 3000) and (40000, 64) take the streaming
# plan (rows cut between warp ranges, many rows per load batch); the others the
# chunk plan.  (4, 262144, 4) is the top-W proposer's shape (64 chunks a row);
# (2, 262144, 16) folds 1024 candidates per row in the merge.
@pytest.mark.parametrize("rows,V,k", [(1, 1, 1), (3, 7, 7), (8, 1024, 4), (16, 262144, 4),
                                      (5, 100003, 16), (300, 4099, 10), (1, 40000, 16),
                                      (64, 65536, 10), (999, 3000, 10), (40000, 64, 16),
                                      (4, 262144, 4), (2, 262144, 16)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topk_matches_oracle(tv, rows, V, k, dtype):
    g = torch.Generator(device="cuda").manual_seed(rows * 31 + V + k)
    x = torch.randn(rows, V, generator=g, device="cuda")
    if V > 64:
        x[:, ::53] = 2.75                  # exact ties, across chunk boundaries
        x[0, V // 2] = 9.0
        x[0, V // 3] = 9.0
        x[rows - 1, V - 1] = 11.0
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    vals, idx = run_topk(tv, x, k)
    ev, ei = tb.topk(host(x, dtype), k, dtype)
    assert np.array_equal(idx, ei)
    assert np.array_equal(vals, ev)


@pytest.mark.parametrize("rows", [8, 40])       # chunk plan, streaming plan
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_topk_special_rows(tv, dtype, rows):
    V, k = 70000, 16
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn(rows, V, generator=g, device="cuda").to(dtype)
    inf, nan = float("inf"), float("nan")
    x[0] = -inf                            # fewer than k finite values: real indices 0..15
    x[1] = nan
    x[2] = -inf
    x[2, 100:105] = 1.0                    # 5 finite, then the lowest -inf indices
    x[3] = 0.0
    x[3, ::2] = -0.0                       # +0 == -0: indices 0..15 in order
    x[4, 5] = nan
    x[4, 6] = inf
    x[5, :] = 1.0                          # all tied
    dt = "bf16" if dtype == torch.bfloat16 else "f32"
    vals, idx = run_topk(tv, x, k)
    ev, ei = tb.topk(host(x, dt), k, dt)
    assert list(idx[0]) == list(range(16))
    assert list(idx[2][:5]) == [100, 101, 102, 103, 104] and list(idx[2][5:]) == list(range(11))
    assert idx[4][0] == 6
    assert np.array_equal(idx, ei)
    assert np.array_equal(vals, ev)


def test_topk_strided_rows_and_k1_is_argmax(tv):
    g = torch.Generator(device="cuda").manual_seed(9)
    base = torch.randn(37, 50011, generator=g, device="cuda").to(torch.bfloat16)
    x = base[:, :49999]                    # row stride 50011: rows not 16-byte aligned
    vals, idx = run_topk(tv, x, 5)
    ev, ei = tb.topk(host(x.contiguous(), "bf16"), 5, "bf16")
    assert np.array_equal(idx, ei) and np.array_equal(vals, ev)
    am = torch.empty(37, dtype=torch.int32, device="cuda")
    tv.tv_argmax(x, am)
    _, i1 = run_topk(tv, x, 1)
    assert np.array_equal(i1[:, 0], am.cpu().numpy())


def test_topk_full_size_sampled(tv):
    """The tree-build workload's 512 rows x 151936 (fp32); every 16th row checked."""
    lp = workloads.make_draft("tree_build", "cuda")
    B, L, V = lp.shape
    x = lp.view(B * L, V)
    vals, idx = run_topk(tv, x, 10)
    sel = np.arange(0, B * L, 16)
    ev, ei = tb.topk(x[torch.as_tensor(sel, device="cuda")].cpu().numpy(), 10, "f32")
    assert np.array_equal(idx[sel], ei) and np.array_equal(vals[sel], ev)


# ------------------------------------------------------------------ build_tree

def candidates(B, L, V, K, seed, quantum=0.0):
    lp = workloads.make_draft("tree_build", "cpu", seed=seed, B=B, L=L, V=V, quantum=quantum)
    vals, idx = tb.topk(lp.reshape(B * L, V).numpy(), K, "f32")
    return vals.reshape(B, L, K), idx.reshape(B, L, K)


def run_tree(tv, vals, idx, budget, w):
    B = vals.shape[0]
    dev = "cuda"
    cv = torch.as_tensor(vals, device=dev)
    ci = torch.as_tensor(idx, device=dev)
    out = {k: torch.empty(B, budget, dtype=torch.int32, device=dev) for k in ("tokens", "parent", "depth")}
    out["score"] = torch.empty(B, budget, dtype=torch.float32, device=dev)
    out["n_nodes"] = torch.empty(B, dtype=torch.int32, device=dev)
    tv.tv_build_tree(cv, ci, budget, w, out["tokens"], out["parent"], out["depth"], out["score"],
                     out["n_nodes"])
    return {k: v.cpu().numpy() for k, v in out.items()}


def assert_tree_equal(got, exp):
    for k in ("tokens", "parent", "depth", "n_nodes"):
        assert np.array_equal(got[k], exp[k]), k
    assert np.array_equal(got["score"], exp["score"])  # bit-identical fp32 sums (and -inf pads)


@pytest.mark.parametrize("L,K,budget,w", [(5, 10, 32, 1), (8, 10, 32, 1), (8, 10, 32, 4),
                                          (8, 4, 64, 3), (3, 2, 64, 1), (1, 16, 16, 1),
                                          (6, 1, 6, 1), (4, 8, 64, 64), (8, 10, 64, 7)])
def test_build_tree_matches_oracle(tv, L, K, budget, w):
    B = 24
    vals, idx = candidates(B, L, 3000, K, seed=L * 100 + K * 10 + w)
    got = run_tree(tv, vals, idx, budget, w)
    exp = tb.build_tree(vals, idx, budget, w)
    assert_tree_equal(got, exp)


@pytest.mark.parametrize("budget", [32, 64])
@pytest.mark.parametrize("w", [1, 2, 5])
def test_build_tree_ties_follow_push_order(tv, w, budget):
    """Logits on a 0.5 grid: many exactly tied log-probabilities and scores."""
    B, L, K = 32, 6, 12
    vals, idx = candidates(B, L, 200, K, seed=77 + w, quantum=0.5)
    assert any(len(set(r.tolist())) < K for r in vals.reshape(-1, K))  # ties exist
    got = run_tree(tv, vals, idx, budget, w)
    exp = tb.build_tree(vals, idx, budget, w)
    assert_tree_equal(got, exp)


@pytest.mark.parametrize("budget", [32, 64])
@pytest.mark.parametrize("w", [1, 3])
def test_build_tree_ties_and_signed_zeros(tv, budget, w):
    """Candidate values on a 0.5 grid around zero, zeros stored as -0 or +0 at
    random: many exact ties, scores that sum to +0 or -0.  The two zeros
    compare equal, so the push counter decides between them; the scores keep
    their sign bits."""
    rng = np.random.default_rng(400 + budget + w)
    B, L, K = 40, 5, 6
    vals = (rng.integers(-4, 5, (B, L, K)) * 0.5).astype(np.float32)
    vals = -np.sort(-vals, axis=-1)
    neg = rng.random((B, L, K)) < 0.5
    vals = np.where((vals == 0) & neg, np.float32(-0.0), vals).astype(np.float32)
    assert (np.signbit(vals) & (vals == 0)).any() and (~np.signbit(vals) & (vals == 0)).any()
    idx = np.arange(B * L * K, dtype=np.int32).reshape(B, L, K)
    got = run_tree(tv, vals, idx, budget, w)
    exp = tb.build_tree(vals, idx, budget, w)
    assert_tree_equal(got, exp)
    assert np.array_equal(got["score"].view(np.int32), exp["score"].view(np.int32))


def test_build_tree_minus_inf_candidates(tv):
    B, L, K = 4, 3, 5
    vals, idx = candidates(B, L, 50, K, seed=5)
    vals[0, 1, 2:] = -np.inf
    vals[1, 0, 1:] = -np.inf
    got = run_tree(tv, vals, idx, 40, 1)
    exp = tb.build_tree(vals, idx, 40, 1)
    assert_tree_equal(got, exp)


def test_draft_tree_full_size_and_verify_layout(tv):
    """The tree-build workload end to end on the GPU (top-k + construction),
    against the oracle on the GPU's candidate lists and on its own top-k for a
    sample of sequences; the trees pass tv_build_ancestors' checks."""
    w = workloads.DRAFT_WORKLOADS["tree_build"]
    lp = workloads.make_draft("tree_build", "cuda")
    dt = tv.DraftTree(w.B, w.L, w.V, w.K, w.budget, w.w)
    o = dt(lp)
    torch.cuda.synchronize()
    cv, ci = o.cand_lp.cpu().numpy(), o.cand_idx.cpu().numpy()
    exp = tb.build_tree(cv, ci, w.budget, w.w)
    got = {k: getattr(o, k).cpu().numpy() for k in ("tokens", "parent", "depth", "score", "n_nodes")}
    assert_tree_equal(got, exp)
    for b in (0, 17, 63):
        ev, ei = tb.topk(lp[b].cpu().numpy(), w.K, "f32")
        assert np.array_equal(ci[b], ei) and np.array_equal(cv[b], ev)
    B, N = w.B, w.budget
    anc = torch.empty(B, N, dtype=torch.int64, device="cuda")
    pos = torch.empty(B, N, dtype=torch.int32, device="cuda")
    st = torch.empty(B, dtype=torch.int32, device="cuda")
    ctx = torch.full((B,), 1000, dtype=torch.int32, device="cuda")
    tv.tv_build_ancestors(o.parent, o.depth, ctx, anc, pos, st)
    assert int(st.abs().sum()) == 0
    assert torch.equal(pos, ctx[:, None] - 1 + o.depth)

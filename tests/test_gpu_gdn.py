"""GPU parity of GDN tree verification and its deferred commit against the
fp64 oracle (oracle/gdn.py).

Tolerance: the kernels work in fp32 from bf16 q / k / v and an fp32 state.
Every output is a d_k-term dot product (Q S_0) plus at most depth terms of the
triangular solve, each of size O(1) for unit-norm q / k and the input scales,
so fp32 rounding stays near 1e-6; the bound checked is
|gpu - ref| <= 1e-4 + 1e-4 |ref| (states: the same on each entry).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import gdn as ogdn

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-4


@pytest.fixture(scope="module")
def tv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_decoding_build_gb300 as m
    return m


def to_dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def oracle_inputs(x):
    """Host fp64 copies in the oracle's layout (S, not S^T) and its ancestor bitmask."""
    f = lambda t: t.detach().cpu().double().numpy()
    mask, _, st = oracle.ancestors(x["parent"].cpu().numpy(), x["depth"].cpu().numpy(),
                                   np.full(x["B"], 10, np.int32))
    assert np.all(st == 0)
    anc = (mask.astype(np.uint64) << np.arange(mask.shape[2], dtype=np.uint64)).sum(-1)
    return dict(state=np.swapaxes(f(x["state"]), -1, -2), q=f(x["q"]), k=f(x["k"]), v=f(x["v"]),
                alpha=f(x["alpha"]), beta=f(x["beta"]), anc=anc)


def run_verify(tv, x, kernel=0):
    B, N, Hv, dv = x["B"], x["N"], x["Hv"], x["dv"]
    anc = torch.empty(B, N, dtype=torch.int64, device="cuda")
    pos = torch.empty(B, N, dtype=torch.int32, device="cuda")
    st = torch.empty(B, dtype=torch.int32, device="cuda")
    tv.tv_build_ancestors(x["parent"], x["depth"], torch.full((B,), 10, dtype=torch.int32,
                                                                device="cuda"), anc, pos, st)
    out = torch.full((B, N, Hv, dv), float("nan"), device="cuda")
    u = torch.full((B, N, Hv, dv), float("nan"), device="cuda")
    g = torch.full((B, N, Hv), float("nan"), device="cuda")
    tv.tv_gdn_tree_verify(x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], anc, out, u,
                          g, st, kernel=kernel)
    torch.cuda.synchronize()
    return out, u, g, st


def close(got, ref):
    got = got.detach().cpu().double().numpy()
    err = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    assert np.isfinite(got).all()
    assert err.max() <= 0, f"max excess {err.max():.3e}"


CASES = [  # kernel 0 picks the pipeline (N <= 32), else the tensor cores (d_k 64 / 128), else CUDA cores
    dict(),                                                       # gdn_small: dk 32, dv 64
    dict(B=2, N=32, Hk=4, Hv=8, dk=128, dv=128),                  # the stress head shape
    dict(B=2, N=64, Hk=1, Hv=2, dk=96, dv=64, tree="chain"),      # depth 64
    dict(B=2, N=64, Hk=2, Hv=4, dk=64, dv=128, tree="chain"),     # depth 64, 2N = 128 rows
    dict(B=2, N=40, Hk=2, Hv=2, dk=128, dv=64, tree="star"),      # depth 1 everywhere
    dict(B=3, N=45, Hk=1, Hv=3, dk=128, dv=64),                   # K and Q rows across TMEM quadrants
    dict(B=1, N=1, Hk=1, Hv=1, dk=32, dv=64),                     # a single node
    dict(B=1, N=1, Hk=1, Hv=1, dk=64, dv=64),
    dict(B=3, N=20, Hk=2, Hv=4, dk=64, dv=64),                    # pipeline: ragged N, d 64 x 64
    dict(B=2, N=32, Hk=1, Hv=2, dk=128, dv=64, tree="chain"),     # pipeline: depth 32
    dict(B=5, N=7, Hk=2, Hv=2, dk=128, dv=128, tree="star"),      # pipeline: depth 1, N < 8
    dict(B=40, N=8, Hk=2, Hv=8, dk=64, dv=64),                    # pipeline: 320 items, > 1 per CTA
]


def supported(kw, kernel):
    x = dict(workloads.GDN_WORKLOADS["gdn_small"].__dict__, **kw)
    tc = x["dk"] in (64, 128)
    return kernel in (0, 1) or (kernel == 2 and tc) or (kernel == 3 and tc and x["N"] <= 32)


@pytest.mark.parametrize("kernel", [0, 1, 2, 3])
@pytest.mark.parametrize("kw", CASES)
def test_verify_matches_oracle(tv, kw, kernel):
    if not supported(kw, kernel):
        pytest.skip("shape outside this kernel")
    x = to_dev(workloads.make_gdn("gdn_small", "cpu", **kw))
    out, u, g, _ = run_verify(tv, x, kernel)
    o = oracle_inputs(x)
    ref = ogdn.tree_verify(o["state"], o["q"], o["k"], o["v"], o["alpha"], o["beta"], o["anc"])
    close(out, ref["out"])
    close(u, ref["u"])
    close(g, ref["g"])


@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_verify_full_size_sampled(tv, kernel):
    """The gdn_stress workload (64 sequences x 32 value heads, 128 x 128 state):
    every output computed, four (sequence, head) pairs checked in full."""
    x = to_dev(workloads.make_gdn("gdn_stress", "cpu"))
    out, u, g, _ = run_verify(tv, x, kernel)
    for b, h in ((0, 0), (17, 5), (40, 31), (63, 16)):
        hk = h // (x["Hv"] // x["Hk"])
        sub = dict(x, B=1, Hk=1, Hv=1, parent=x["parent"][b:b + 1], depth=x["depth"][b:b + 1],
                   q=x["q"][b:b + 1, :, hk:hk + 1], k=x["k"][b:b + 1, :, hk:hk + 1],
                   v=x["v"][b:b + 1, :, h:h + 1], alpha=x["alpha"][b:b + 1, :, h:h + 1],
                   beta=x["beta"][b:b + 1, :, h:h + 1], state=x["state"][b:b + 1, h:h + 1])
        o = oracle_inputs(sub)
        ref = ogdn.tree_verify(o["state"], o["q"], o["k"], o["v"], o["alpha"], o["beta"], o["anc"])
        close(out[b:b + 1, :, h:h + 1], ref["out"])
        close(u[b:b + 1, :, h:h + 1], ref["u"])


@pytest.mark.parametrize("kernel,kw", [(0, dict()), (2, dict(dk=128, dv=128)),
                                       (3, dict(dk=128, dv=128))])
def test_bad_tree_is_skipped(tv, kernel, kw):
    x = to_dev(workloads.make_gdn("gdn_small", "cpu", **kw))
    x["parent"][1, 5] = 7           # parent after the child: tv_build_ancestors flags it
    out, u, g, st = run_verify(tv, x, kernel)
    assert st.cpu().tolist() == [0, st.cpu().tolist()[1], 0] and st.cpu().tolist()[1] != 0
    assert torch.isnan(out[1]).all() and torch.isnan(u[1]).all() and torch.isnan(g[1]).all()
    assert torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all()
    assert torch.isfinite(g[0]).all() and torch.isfinite(g[2]).all()


# d_k 32, 64 and 128 take the commit's shared-column loop (a thread's pieces in
# the same columns), d_k 96 the general one
@pytest.mark.parametrize("kw", [dict(), dict(B=3, N=32, Hk=4, Hv=8, dk=128, dv=128),
                                dict(B=4, N=20, Hk=2, Hv=4, dk=64, dv=128),
                                dict(B=3, N=24, Hk=1, Hv=2, dk=96, dv=64)])
def test_commit_matches_oracle(tv, kw):
    x = to_dev(workloads.make_gdn("gdn_small", "cpu", **kw))
    out, u, g, st = run_verify(tv, x)
    B, N = x["B"], x["N"]
    o = oracle_inputs(x)
    rng = np.random.default_rng(1)
    acc = np.zeros((B, N), np.int32)
    n_acc = np.zeros(B, np.int32)
    for b in range(B - 1):          # the last sequence accepts nothing
        leaf = int(rng.integers(0, N))
        p = ogdn.path_of(o["anc"][b, leaf], leaf)
        acc[b, :len(p)] = p
        n_acc[b] = len(p)
    new = torch.empty_like(x["state"])
    tv.tv_gdn_commit(x["state"], x["k"], u, x["alpha"], torch.as_tensor(acc, device="cuda"),
                     torch.as_tensor(n_acc, device="cuda"), new, st)
    torch.cuda.synchronize()
    ref = ogdn.commit(o["state"], o["k"], o["v"], o["alpha"], o["beta"], acc, n_acc)
    close(new, np.swapaxes(ref, -1, -2))
    assert torch.equal(new[B - 1], x["state"][B - 1])  # empty accept copies S_0 bit for bit


@pytest.mark.parametrize("kernel", [2, 3])
def test_tensor_and_cuda_cores_agree(tv, kernel):
    """A tensor-core kernel and the CUDA-core one on the same full-size inputs:
    every output within the tolerance of each other (each is within it of the
    fp64 oracle); g, the same product of the same alphas in the same order, equal."""
    x = to_dev(workloads.make_gdn("gdn_stress", "cpu", B=16))
    o1, u1, g1, _ = run_verify(tv, x, 1)
    o2, u2, g2, _ = run_verify(tv, x, kernel)
    close(o2, o1.double().cpu().numpy())
    close(u2, u1.double().cpu().numpy())
    assert torch.equal(g1, g2)

"""The bounded-wait expiry path of the three tensor-core kernels, on the GPU,
in the form that faults and hangs nothing: a test hook (include/tv_debug.h)
initialises one barrier of CTA 0 to expect one arrival more than its producer
makes.  The copy lands but the phase never completes, so the consumer's
bounded wait (2 s) runs out.  Each kernel must then return on its own, with
TV_ERR_CUDA in the status word of the sequence it was working on, having let
its copies land and freed its tensor memory: a normal launch in the same
process afterwards (which allocates the same tensor memory on every SM)
matches the oracle.

Collected after the other GPU tests (file name), before the no-allocation
entry point's test."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close, bf16_to_f64, oracle_attention
from oracle import gdn as ogdn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_decoding_build_gb300 as m
    yield m
    m.tv_debug_withhold_arrival(-1)


def expire(tv, fn):
    """Run fn() with the hook armed for CTA 0; returns (fn's result, seconds)."""
    tv.tv_debug_withhold_arrival(0)
    try:
        t0 = time.time()
        r = fn()
        torch.cuda.synchronize()
        return r, time.time() - t0
    finally:
        tv.tv_debug_withhold_arrival(-1)


def attention(tv, inp, max_ctas):
    B, N = inp["B"], inp["N"]
    anc = torch.empty((B, N), dtype=torch.int64, device="cuda")
    pos = torch.empty((B, N), dtype=torch.int32, device="cuda")
    st = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(inp["q"])
    tv.tv_build_ancestors(inp["parent"], inp["depth"], inp["ctx_len"], anc, pos, st)
    tv.tv_tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"], inp["v_cache"],
                         inp["block_table"], inp["ctx_len"], pos, anc, out, st,
                         window_left=inp["window_left"], kernel=2, max_ctas=max_ctas)
    return out, st


# head dim 128: the persistent kernel on 4 CTAs, so that CTA 0 has tiles (on
# every SM its range would be empty); head dim 256: one CTA per (sequence, KV
# head, split), CTA 0 being split 0 of sequence 0, KV head 0
@pytest.mark.parametrize("name,kw,ctas", [
    ("best_first", dict(B=2, ctx=(300, 900), V=1000), 4),
    ("leaf_sibling", dict(B=2, ctx=(200, 400), V=1000), 0),
])
def test_attention_wait_expiry(tv, name, kw, ctas):
    inp = workloads.make(name, "cuda", 7, **kw)
    (out, st), secs = expire(tv, lambda: attention(tv, inp, ctas))
    st = st.cpu().numpy()
    assert (st == tv.TV_ERR_CUDA).any(), st
    assert set(st.tolist()) <= {0, tv.TV_ERR_CUDA}, st
    assert secs < 30.0, secs
    # the same launch again, hook disarmed: the tensor memory is free again
    out, st = attention(tv, inp, ctas)
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()
    assert_close(bf16_to_f64(out), oracle_attention(workloads.to_numpy(inp)), f"{name} after expiry")


def test_gdn_pipeline_wait_expiry(tv):
    x = workloads.make_gdn("gdn_small", "cpu", B=3, N=20, Hk=2, Hv=4, dk=128, dv=64)
    x = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    B, N, Hv, dv = x["B"], x["N"], x["Hv"], x["dv"]

    def verify():
        anc = torch.empty(B, N, dtype=torch.int64, device="cuda")
        pos = torch.empty(B, N, dtype=torch.int32, device="cuda")
        st = torch.empty(B, dtype=torch.int32, device="cuda")
        tv.tv_build_ancestors(x["parent"], x["depth"], torch.full((B,), 10, dtype=torch.int32,
                                                                    device="cuda"), anc, pos, st)
        out = torch.empty(B, N, Hv, dv, device="cuda")
        u = torch.empty_like(out)
        g = torch.empty(B, N, Hv, device="cuda")
        tv.tv_gdn_tree_verify(x["state"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], anc, out,
                              u, g, st, kernel=3)
        return out, st

    (out, st), secs = expire(tv, verify)
    st = st.cpu().numpy()
    assert (st == tv.TV_ERR_CUDA).any(), st
    assert secs < 30.0, secs
    out, st = verify()
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()
    f = lambda t: t.detach().cpu().double().numpy()
    mask, _, _ = oracle.ancestors(x["parent"].cpu().numpy(), x["depth"].cpu().numpy(),
                                  np.full(B, 10, np.int32))
    anc = (mask.astype(np.uint64) << np.arange(mask.shape[2], dtype=np.uint64)).sum(-1)
    ref = ogdn.tree_verify(np.swapaxes(f(x["state"]), -1, -2), f(x["q"]), f(x["k"]), f(x["v"]),
                           f(x["alpha"]), f(x["beta"]), anc)
    got = f(out)
    assert np.all(np.abs(got - ref["out"]) <= 1e-4 + 1e-4 * np.abs(ref["out"]))

"""The whole multi-layer step (tv_verify_step) and its CUDA-graph form
(tv_verify_graph_*): per layer the same results as the single-layer calls and
the oracle; graph replays equal eager runs bit for bit, are idempotent, and
pick up buffers refilled in place between replays."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_decoding_build_gb300 as m
    return m


CASES = [  # (workload, overrides): D=64 CUDA-core path, D=128 tensor-core path, a window
    ("tiny", dict(plant="hash")),
    ("best_first", dict(B=3, plant="path")),
    ("stress", dict(B=4, ctx=640, plant="path", V=4096)),
    ("window", dict(B=2, ctx=1500, plant="path", V=4096)),
]


def snapshot(ms):
    o = ms.out
    d = {k: getattr(o, k).clone() for k in ("anc", "pos", "status", "argmax", "out_tokens",
                                              "n_emit", "acc_nodes", "n_acc", "ctx_len_out")}
    d["attn"] = [a.clone() for a in ms.attn]
    d["caches"] = [(ly["k_cache"].clone(), ly["v_cache"].clone()) for ly in ms.layers]
    return d


def assert_same(a, b):
    for k in a:
        if k in ("attn", "caches"):
            continue
        assert torch.equal(a[k], b[k]), k
    for x, y in zip(a["attn"], b["attn"]):
        assert torch.equal(x, y)
    for (k1, v1), (k2, v2) in zip(a["caches"], b["caches"]):
        assert torch.equal(k1, k2) and torch.equal(v1, v2)


def fresh(name, kw, L):
    inp = workloads.make(name, "cuda", **kw)
    layers = workloads.make_layers(inp, L, seed=workloads.get(name).seed)
    return inp, layers


@pytest.mark.parametrize("name,kw", CASES)
def test_step_matches_per_layer_calls_and_oracle(tv, name, kw):
    L = 3
    inp, layers = fresh(name, kw, L)
    caches0 = [(ly["k_cache"].clone(), ly["v_cache"].clone()) for ly in layers]
    ms = tv.ModelStep(inp, layers)
    ms.run()
    torch.cuda.synchronize()
    assert int(ms.out.status.abs().sum()) == 0
    for l in range(L):
        # per layer: the single-layer step on that layer's tensors (caches restored)
        li = dict(inp, q=layers[l]["q"], k_tree=layers[l]["k_tree"], v_tree=layers[l]["v_tree"],
                  k_cache=caches0[l][0].clone(), v_cache=caches0[l][1].clone())
        vs = tv.VerifyStep(inp["B"], inp["N"], inp["Hq"], inp["Hkv"], inp["D"], inp["V"],
                           inp["max_blocks"], window_left=inp["window_left"],
                           logits_dtype=inp["logits_dtype"])
        o = vs(li)
        torch.cuda.synchronize()
        assert torch.equal(o.attn, ms.attn[l])
        assert torch.equal(li["k_cache"], ms.layers[l]["k_cache"])
        assert torch.equal(li["v_cache"], ms.layers[l]["v_cache"])
        for k in ("out_tokens", "n_emit", "n_acc", "ctx_len_out"):
            assert torch.equal(getattr(o, k), getattr(ms.out, k)), k
    # layer 1 against the oracle (attention rows, walk, commit)
    li = dict(inp, q=layers[1]["q"], k_tree=layers[1]["k_tree"], v_tree=layers[1]["v_tree"],
              k_cache=caches0[1][0], v_cache=caches0[1][1])
    ref = oracle.verify_step(workloads.to_numpy(li))
    got = ms.attn[1].float().cpu().numpy()
    assert_close(got, ref["attn"])
    assert np.array_equal(ms.out.out_tokens.cpu().numpy(), ref["out_tokens"])
    assert np.array_equal(ms.out.n_acc.cpu().numpy(), ref["n_acc"])
    kc = ms.layers[1]["k_cache"].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(kc, ref["k_cache"])


@pytest.mark.parametrize("name,kw", CASES)
def test_graph_replay_equals_eager_and_is_idempotent(tv, name, kw):
    L = 3
    inp, layers = fresh(name, kw, L)
    saved = [(ly["k_cache"].clone(), ly["v_cache"].clone()) for ly in layers]
    ms = tv.ModelStep(inp, layers)
    ms.run()
    torch.cuda.synchronize()
    eager = snapshot(ms)
    # restore the caches, capture, replay twice
    for ly, (k, v) in zip(ms.layers, saved):
        ly["k_cache"].copy_(k)
        ly["v_cache"].copy_(v)
    ms.capture()
    n_attn = 1 + (1 if ms.ws_attn.numel() > 1 else 0)
    n_arg = 1 + (1 if ms.ws_arg.numel() > 1 else 0)
    assert ms.launches == 1 + L * n_attn + n_arg + 1 + L
    ms.replay()
    torch.cuda.synchronize()
    assert_same(snapshot(ms), eager)
    ms.replay()
    torch.cuda.synchronize()
    assert_same(snapshot(ms), eager)
    ms.close()


def test_graph_sees_buffers_refilled_between_replays(tv):
    """Refill the tree, logits and layer inputs in place (as a model would)
    between replays: each replay equals an eager step on the new contents."""
    L = 2
    kw = dict(B=4, ctx=640, plant="path", V=4096)   # fixed context: same buffer shapes
    inp, layers = fresh("stress", kw, L)
    ms = tv.ModelStep(inp, layers)
    ms.capture()
    for it in range(3):
        nxt, nlayers = fresh("stress", dict(kw, seed=4242 + it), L)
        assert nxt["max_blocks"] == inp["max_blocks"]
        assert nxt["k_cache"].shape == inp["k_cache"].shape
        for k in ("tokens", "parent", "depth", "ctx_len", "root_pred", "block_table", "logits"):
            inp[k].copy_(nxt[k])
        for ly, nl in zip(ms.layers, nlayers):
            for k in ("q", "k_tree", "v_tree", "k_cache", "v_cache"):
                ly[k].copy_(nl[k])
        ms.replay()
        torch.cuda.synchronize()
        got = snapshot(ms)
        for ly, nl in zip(ms.layers, nlayers):  # the same step, eagerly, on the new contents
            ly["k_cache"].copy_(nl["k_cache"])
            ly["v_cache"].copy_(nl["v_cache"])
        ms.run()
        torch.cuda.synchronize()
        assert_same(got, snapshot(ms))
        assert int(ms.out.n_acc.min()) >= 1  # the planted path is accepted
    ms.close()

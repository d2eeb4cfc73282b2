"""Tree speculative-decoding verify step on GB300 (sm_103a).

The step is five calls of the C library ``libtv.so`` (see ``include/tv.h``),
bound here through ctypes with the same names:

    tv_build_ancestors -> tv_tree_attention -> tv_argmax -> tv_tree_walk -> tv_commit_kv

``VerifyStep`` owns the output and scratch buffers of one batch shape and
enqueues the five calls on one CUDA stream with no host synchronisation.

``ModelStep`` (``include/tv_graph.h``) is the step of an L-layer model: every
layer's attention and commit in one unit, enqueued eagerly or captured once
into a CUDA graph and replayed, so nothing runs eagerly between replays.

``tv_gdn_tree_verify`` / ``tv_gdn_commit`` (``include/tv_gdn.h``) verify a
tree through a Gated DeltaNet layer without touching its state, then commit
the state of the accepted path.

The draft side (``include/tv_draft.h``) builds the tree the step verifies:
``tv_topk`` gives each draft position's candidate list and ``tv_build_tree``
expands them best-first into tokens / parent / depth.  ``DraftTree`` owns the
buffers of one shape and enqueues both calls.
"""
from __future__ import annotations

import dataclasses

import torch

from ._lib import (  # noqa: F401
    BLOCK_SIZE, EXPORTS, LIB_PATH, MAX_NODES, TOPK_MAX, TV_BF16, TV_ERR_ARG, TV_ERR_BLOCK,
    TV_ERR_CUDA, TV_ERR_SCRATCH_LIMIT, TV_ERR_TREE, TV_ERR_UNSUPPORTED, TV_F32, TV_OK, TvError,
    status_string, tv_argmax, tv_argmax_noalloc, tv_argmax_workspace_size, tv_build_ancestors,
    tv_build_tree, tv_commit_kv, tv_topk, tv_topk_workspace_size, tv_tree_attention,
    tv_tree_attention_workspace_size, tv_tree_walk, tv_gdn_commit, tv_gdn_tree_verify,
    tv_verify_graph_create,
    tv_verify_graph_destroy, tv_verify_graph_launch, tv_verify_graph_launches, tv_verify_step,
    tv_debug_withhold_arrival, tv_debug_check_failures, tv_debug_checks_enabled)
from ._lib import step_args as _step_args


@dataclasses.dataclass
class StepOutputs:
    anc: torch.Tensor          # int64 [B, N] ancestor-or-self bitmask
    pos: torch.Tensor          # int32 [B, N] position ids
    status: torch.Tensor       # int32 [B]
    attn: torch.Tensor         # bf16 [B, N, Hq, D]
    argmax: torch.Tensor       # int32 [B, N]
    out_tokens: torch.Tensor   # int32 [B, N+1]
    n_emit: torch.Tensor       # int32 [B]
    acc_nodes: torch.Tensor    # int32 [B, N]
    n_acc: torch.Tensor        # int32 [B]
    ctx_len_out: torch.Tensor  # int32 [B]


class VerifyStep:
    """One verify step for a fixed batch shape; buffers are allocated once.

    ``argmax_sms`` > 0 runs tv_argmax beside tv_tree_attention instead of after
    it: the argmax goes to a second stream holding ``argmax_sms`` SMs
    (tv_argmax_sm), the attention keeps the rest (max_ctas), and the walk waits
    for both.  The two HBM-bound kernels then read memory at the same time."""

    def __init__(self, B, N, Hq, Hkv, D, V, max_blocks, window_left=-1, logits_dtype="bf16",
                 num_splits=0, device="cuda", argmax_sms=0):
        dev = torch.device(device)
        self.argmax_sms = int(argmax_sms)
        if self.argmax_sms > 0:
            self.side = torch.cuda.Stream(device=dev)
            self.ev_fork = torch.cuda.Event()
            self.ev_join = torch.cuda.Event()
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            self.attn_ctas = max(1, sms - self.argmax_sms)
        i32 = torch.int32
        self.shape = dict(B=B, N=N, Hq=Hq, Hkv=Hkv, D=D, V=V, max_blocks=max_blocks)
        self.window_left = window_left
        self.num_splits = num_splits
        self.out = StepOutputs(
            anc=torch.empty((B, N), dtype=torch.int64, device=dev),
            pos=torch.empty((B, N), dtype=i32, device=dev),
            status=torch.empty((B,), dtype=i32, device=dev),
            attn=torch.empty((B, N, Hq, D), dtype=torch.bfloat16, device=dev),
            argmax=torch.empty((B, N), dtype=i32, device=dev),
            out_tokens=torch.empty((B, N + 1), dtype=i32, device=dev),
            n_emit=torch.empty((B,), dtype=i32, device=dev),
            acc_nodes=torch.empty((B, N), dtype=i32, device=dev),
            n_acc=torch.empty((B,), dtype=i32, device=dev),
            ctx_len_out=torch.empty((B,), dtype=i32, device=dev),
        )
        ws_attn = tv_tree_attention_workspace_size(B, N, Hq, Hkv, D, max_blocks, window_left,
                                                   num_splits)
        dt = TV_F32 if logits_dtype == "f32" else TV_BF16
        ws_arg = tv_argmax_workspace_size(B * N, V, dt)
        self.ws_attn = torch.empty(max(ws_attn, 1), dtype=torch.uint8, device=dev)
        self.ws_arg = torch.empty(max(ws_arg, 1), dtype=torch.uint8, device=dev)

    def __call__(self, inp, stream=None) -> StepOutputs:
        """Enqueue the whole step for ``inp`` (dict of device tensors)."""
        o = self.out
        B, N = inp["tokens"].shape
        main = stream if stream is not None else torch.cuda.current_stream()
        if self.argmax_sms > 0:  # the argmax on its own SMs, beside the attention
            self.ev_fork.record(main)
            self.side.wait_event(self.ev_fork)
            tv_argmax(inp["logits"].view(B * N, -1), o.argmax.view(B * N), self.ws_arg, self.side,
                      sm_limit=self.argmax_sms)
            self.ev_join.record(self.side)
        tv_build_ancestors(inp["parent"], inp["depth"], inp["ctx_len"], o.anc, o.pos, o.status,
                           stream)
        tv_tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"], inp["v_cache"],
                          inp["block_table"], inp["ctx_len"], o.pos, o.anc, o.attn, o.status,
                          window_left=self.window_left, num_splits=self.num_splits,
                          workspace=self.ws_attn, stream=stream,
                          max_ctas=self.attn_ctas if self.argmax_sms > 0 else 0)
        if self.argmax_sms > 0:
            main.wait_event(self.ev_join)
        else:
            tv_argmax(inp["logits"].view(B * N, -1), o.argmax.view(B * N), self.ws_arg, stream)
        tv_tree_walk(inp["tokens"], inp["parent"], o.argmax, inp["root_pred"], o.status,
                     o.out_tokens, o.n_emit, o.acc_nodes, o.n_acc, stream)
        tv_commit_kv(inp["k_tree"], inp["v_tree"], o.acc_nodes, o.n_acc, inp["ctx_len"],
                     inp["block_table"], inp["k_cache"], inp["v_cache"], o.ctx_len_out, o.status,
                     stream)
        return o


class ModelStep:
    """The verify step of an L-layer model for fixed buffers: tv_build_ancestors,
    every layer's tv_tree_attention, tv_argmax, tv_tree_walk, every layer's
    tv_commit_kv.  ``inp`` holds the tree, sequence state and logits (the dict
    of ``workloads.make``), ``layers`` one dict per layer with q / k_tree /
    v_tree / k_cache / v_cache tensors; each layer's attention output is
    allocated here (``self.attn[l]``).  ``run()`` enqueues the launches
    eagerly; ``capture()`` records them once into a CUDA graph, after which
    ``replay()`` launches the graph.  Buffers are used in place: refill them
    between replays."""

    def __init__(self, inp, layers, device="cuda"):
        dev = torch.device(device)
        B, N, Hq, Hkv, D = inp["B"], inp["N"], inp["Hq"], inp["Hkv"], inp["D"]
        V = inp["logits"].shape[-1]
        i32 = torch.int32
        self.inp = inp
        self.out = StepOutputs(
            anc=torch.empty((B, N), dtype=torch.int64, device=dev),
            pos=torch.empty((B, N), dtype=i32, device=dev),
            status=torch.empty((B,), dtype=i32, device=dev),
            attn=torch.empty((0,), dtype=torch.bfloat16, device=dev),
            argmax=torch.empty((B, N), dtype=i32, device=dev),
            out_tokens=torch.empty((B, N + 1), dtype=i32, device=dev),
            n_emit=torch.empty((B,), dtype=i32, device=dev),
            acc_nodes=torch.empty((B, N), dtype=i32, device=dev),
            n_acc=torch.empty((B,), dtype=i32, device=dev),
            ctx_len_out=torch.empty((B,), dtype=i32, device=dev))
        self.attn = [torch.empty((B, N, Hq, D), dtype=torch.bfloat16, device=dev) for _ in layers]
        self.layers = [dict(ly, out=o) for ly, o in zip(layers, self.attn)]
        ws_attn = tv_tree_attention_workspace_size(B, N, Hq, Hkv, D, inp["max_blocks"],
                                                   inp["window_left"])
        dt = TV_F32 if inp["logits"].dtype == torch.float32 else TV_BF16
        ws_arg = tv_argmax_workspace_size(B * N, V, dt)
        self.ws_attn = torch.empty(max(ws_attn, 1), dtype=torch.uint8, device=dev)
        self.ws_arg = torch.empty(max(ws_arg, 1), dtype=torch.uint8, device=dev)
        flat = dict(inp, logits=inp["logits"].reshape(B * N, V))
        self.args = _step_args(flat, self.out, self.layers, self.ws_attn, self.ws_arg)
        self.graph = None

    def run(self, stream=None):
        tv_verify_step(self.args, stream)
        return self.out

    def capture(self):
        if self.graph is None:
            self.graph = tv_verify_graph_create(self.args)
        return self

    def replay(self, stream=None):
        tv_verify_graph_launch(self.graph, stream)
        return self.out

    @property
    def launches(self):
        return tv_verify_graph_launches(self.graph) if self.graph is not None else None

    def close(self):
        if self.graph is not None:
            tv_verify_graph_destroy(self.graph)
            self.graph = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


@dataclasses.dataclass
class DraftOutputs:
    cand_lp: torch.Tensor      # float32 [B, L, K] per-depth candidate log-probs
    cand_idx: torch.Tensor     # int32 [B, L, K] their token ids
    tokens: torch.Tensor       # int32 [B, budget]
    parent: torch.Tensor       # int32 [B, budget]
    depth: torch.Tensor        # int32 [B, budget]
    score: torch.Tensor        # float32 [B, budget] cumulative log-prob
    n_nodes: torch.Tensor      # int32 [B]


class DraftTree:
    """Draft-tree construction for a fixed shape: ``tv_topk`` over the draft
    log-probabilities [B, L, V] (one row per draft position), then
    ``tv_build_tree``.  Buffers are allocated once."""

    def __init__(self, B, L, V, K, budget, w=1, dtype=torch.float32, device="cuda"):
        self.B, self.L, self.V, self.K, self.budget, self.w = B, L, V, K, budget, w
        dev = torch.device(device)
        i32, f32 = torch.int32, torch.float32
        self.out = DraftOutputs(
            cand_lp=torch.empty(B, L, K, dtype=f32, device=dev),
            cand_idx=torch.empty(B, L, K, dtype=i32, device=dev),
            tokens=torch.empty(B, budget, dtype=i32, device=dev),
            parent=torch.empty(B, budget, dtype=i32, device=dev),
            depth=torch.empty(B, budget, dtype=i32, device=dev),
            score=torch.empty(B, budget, dtype=f32, device=dev),
            n_nodes=torch.empty(B, dtype=i32, device=dev))
        dt = TV_F32 if dtype == torch.float32 else TV_BF16
        need = tv_topk_workspace_size(B * L, V, K, dt)
        self.ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)

    def __call__(self, logprobs, stream=None):
        """``logprobs`` [B, L, V] (float32 or bf16): log-probabilities of each
        draft position.  Returns the outputs (enqueued on ``stream``)."""
        o = self.out
        B, L, V = logprobs.shape
        tv_topk(logprobs.reshape(B * L, V), self.K, o.cand_lp.view(B * L, self.K),
                o.cand_idx.view(B * L, self.K), self.ws, stream)
        tv_build_tree(o.cand_lp, o.cand_idx, self.budget, self.w, o.tokens, o.parent, o.depth,
                      o.score, o.n_nodes, stream)
        return o

"""ctypes binding of libtv.so: argument marshalling only.

Each ``tv_*`` function here has the name and argument order of the C entry
point in ``include/tv.h``, ``tv_draft.h``, ``tv_graph.h`` or ``tv_gdn.h``; it checks dtypes, devices and contiguity of the
torch tensors it is given, passes their device pointers, and raises
``TvError`` on a non-zero host status.  All arithmetic runs in the library's
CUDA kernels; there is no fallback of any kind: without the compiled library
importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
# TV_LIB_PATH selects another build of the same library (the TV_DEBUG build's
# libtv_debug.so); by default the release build
LIB_PATH = os.environ.get("TV_LIB_PATH") or _build.LIB

(TV_OK, TV_ERR_ARG, TV_ERR_TREE, TV_ERR_BLOCK, TV_ERR_CUDA, TV_ERR_UNSUPPORTED,
 TV_ERR_SCRATCH_LIMIT) = range(7)
TV_F32, TV_BF16 = 0, 1
BLOCK_SIZE = 16
TOPK_MAX = 16
MAX_NODES = 64

EXPORTS = (
    "tv_status_string",
    "tv_build_ancestors",
    "tv_tree_attention_workspace_size",
    "tv_tree_attention",
    "tv_argmax_workspace_size",
    "tv_argmax",
    "tv_argmax_sm",
    "tv_argmax_noalloc",
    "tv_tree_walk",
    "tv_commit_kv",
    "tv_topk_workspace_size",
    "tv_topk",
    "tv_build_tree",
    "tv_verify_step",
    "tv_verify_graph_create",
    "tv_verify_graph_launch",
    "tv_verify_graph_launches",
    "tv_verify_graph_destroy",
    "tv_gdn_tree_verify",
    "tv_gdn_commit",
    "tv_debug_withhold_arrival",
    "tv_debug_checks_enabled",
    "tv_debug_check_failures",
)


class TvError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn}: {status_string(code)} (status {code})")


class AttnArgs(ctypes.Structure):
    """Mirror of ``tv_attn_args``."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_tree", ctypes.c_void_p), ("v_tree", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("ctx_len", ctypes.c_void_p), ("pos", ctypes.c_void_p),
        ("anc", ctypes.c_void_p),
        ("B", ctypes.c_int), ("N", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("D", ctypes.c_int), ("block_size", ctypes.c_int), ("max_blocks", ctypes.c_int),
        ("num_blocks", ctypes.c_int), ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
        ("sm_scale", ctypes.c_float), ("num_splits", ctypes.c_int), ("kernel", ctypes.c_int),
        ("max_ctas", ctypes.c_int), ("out", ctypes.c_void_p), ("status", ctypes.c_void_p),
    ]


class Layer(ctypes.Structure):
    """Mirror of ``tv_layer``."""
    _fields_ = [("q", ctypes.c_void_p), ("k_tree", ctypes.c_void_p), ("v_tree", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("out", ctypes.c_void_p)]


class StepArgs(ctypes.Structure):
    """Mirror of ``tv_step_args``."""
    _fields_ = [
        ("tokens", ctypes.c_void_p), ("parent", ctypes.c_void_p), ("depth", ctypes.c_void_p),
        ("ctx_len", ctypes.c_void_p), ("root_pred", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("B", ctypes.c_int), ("N", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("D", ctypes.c_int), ("max_blocks", ctypes.c_int), ("num_blocks", ctypes.c_int),
        ("window_left", ctypes.c_int), ("sm_scale", ctypes.c_float),
        ("num_layers", ctypes.c_int), ("layers", ctypes.POINTER(Layer)),
        ("attn_workspace", ctypes.c_void_p), ("attn_workspace_bytes", ctypes.c_size_t),
        ("logits", ctypes.c_void_p), ("logits_dtype", ctypes.c_int), ("V", ctypes.c_int64),
        ("argmax_workspace", ctypes.c_void_p), ("argmax_workspace_bytes", ctypes.c_size_t),
        ("anc", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("argmax", ctypes.c_void_p), ("out_tokens", ctypes.c_void_p), ("n_emit", ctypes.c_void_p),
        ("acc_nodes", ctypes.c_void_p), ("n_acc", ctypes.c_void_p),
        ("ctx_len_out", ctypes.c_void_p),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libtv.so is not built ({LIB_PATH}); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, L, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.tv_status_string.argtypes = [I]
    lib.tv_status_string.restype = ctypes.c_char_p
    lib.tv_build_ancestors.argtypes = [P, P, P, I, I, P, P, P, P]
    lib.tv_tree_attention_workspace_size.argtypes = [ctypes.POINTER(AttnArgs)]
    lib.tv_tree_attention_workspace_size.restype = S
    lib.tv_tree_attention.argtypes = [ctypes.POINTER(AttnArgs), P, S, P]
    lib.tv_argmax_workspace_size.argtypes = [L, L, I]
    lib.tv_argmax_workspace_size.restype = S
    lib.tv_argmax.argtypes = [P, I, L, L, L, P, P, S, P]
    lib.tv_argmax_sm.argtypes = [P, I, L, L, L, P, P, S, I, P]
    lib.tv_argmax_sm.restype = I
    lib.tv_argmax_noalloc.argtypes = [P, I, L, L, L, P, P]
    lib.tv_argmax_noalloc.restype = I
    lib.tv_tree_walk.argtypes = [P, P, P, P, P, I, I, P, P, P, P, P]
    lib.tv_commit_kv.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, P, P]
    lib.tv_topk_workspace_size.argtypes = [L, L, I, I]
    lib.tv_topk_workspace_size.restype = S
    lib.tv_topk.argtypes = [P, I, L, L, L, I, P, P, P, S, P]
    lib.tv_build_tree.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P, P]
    lib.tv_verify_step.argtypes = [ctypes.POINTER(StepArgs), P]
    lib.tv_verify_graph_create.argtypes = [ctypes.POINTER(StepArgs), ctypes.POINTER(P)]
    lib.tv_verify_graph_launch.argtypes = [P, P]
    lib.tv_verify_graph_launches.argtypes = [P]
    lib.tv_verify_graph_launches.restype = I
    lib.tv_verify_graph_destroy.argtypes = [P]
    lib.tv_verify_graph_destroy.restype = None
    lib.tv_gdn_tree_verify.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, I, P, P]
    lib.tv_gdn_commit.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P]
    lib.tv_debug_withhold_arrival.argtypes = [I]
    lib.tv_debug_withhold_arrival.restype = None
    lib.tv_debug_checks_enabled.argtypes = []
    lib.tv_debug_checks_enabled.restype = I
    lib.tv_debug_check_failures.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(I), I]
    lib.tv_debug_check_failures.restype = ctypes.c_uint
    for f in ("tv_build_ancestors", "tv_tree_attention", "tv_argmax", "tv_tree_walk",
              "tv_commit_kv", "tv_topk", "tv_build_tree", "tv_verify_step",
              "tv_verify_graph_create", "tv_verify_graph_launch", "tv_gdn_tree_verify",
              "tv_gdn_commit"):
        getattr(lib, f).restype = I
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.tv_status_string(int(code)).decode()


def _check(fn, code):
    if code != TV_OK:
        raise TvError(fn, code)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def tv_build_ancestors(parent, depth, ctx_len, anc, pos, status, stream=None):
    B, N = parent.shape
    _check("tv_build_ancestors", lib.tv_build_ancestors(
        _ptr(parent, torch.int32, "parent"), _ptr(depth, torch.int32, "depth"),
        _ptr(ctx_len, torch.int32, "ctx_len"), B, N, _ptr(anc, torch.int64, "anc"),
        _ptr(pos, torch.int32, "pos"), _ptr(status, torch.int32, "status"), _stream(stream)))


KERNEL_AUTO, KERNEL_CUDA_CORE, KERNEL_TENSOR_CORE = 0, 1, 2


def attn_args(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_len, pos, anc, out, status,
              window_left=-1, window_right=0, sm_scale=0.0, num_splits=0, kernel=0, max_ctas=0):
    bf = torch.bfloat16
    B, N, Hq, D = q.shape
    a = AttnArgs()
    a.q = _ptr(q, bf, "q")
    a.k_tree = _ptr(k_tree, bf, "k_tree")
    a.v_tree = _ptr(v_tree, bf, "v_tree")
    a.k_cache = _ptr(k_cache, bf, "k_cache")
    a.v_cache = _ptr(v_cache, bf, "v_cache")
    a.block_table = _ptr(block_table, torch.int32, "block_table")
    a.ctx_len = _ptr(ctx_len, torch.int32, "ctx_len")
    a.pos = _ptr(pos, torch.int32, "pos")
    a.anc = _ptr(anc, torch.int64, "anc")
    a.B, a.N, a.Hq, a.Hkv, a.D = B, N, Hq, k_tree.shape[2], D
    a.block_size = k_cache.shape[2]
    a.max_blocks = block_table.shape[1]
    a.num_blocks = k_cache.shape[0]
    a.window_left = int(window_left)
    a.window_right = int(window_right)
    a.sm_scale = float(sm_scale)
    a.num_splits = int(num_splits)
    a.kernel = int(kernel)
    a.max_ctas = int(max_ctas)
    a.out = _ptr(out, bf, "out")
    a.status = _ptr(status, torch.int32, "status")
    return a


def tv_tree_attention_workspace_size(B, N, Hq, Hkv, D, max_blocks, window_left=-1, num_splits=0,
                                     kernel=0):
    a = AttnArgs()
    a.kernel = kernel
    a.B, a.N, a.Hq, a.Hkv, a.D = B, N, Hq, Hkv, D
    a.block_size = BLOCK_SIZE
    a.max_blocks = max_blocks
    a.window_left = window_left
    a.window_right = 0
    a.num_splits = num_splits
    return int(lib.tv_tree_attention_workspace_size(ctypes.byref(a)))


def tv_tree_attention(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_len, pos, anc, out,
                      status, window_left=-1, window_right=0, sm_scale=0.0, num_splits=0,
                      workspace=None, stream=None, kernel=0, max_ctas=0):
    a = attn_args(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_len, pos, anc, out, status,
                  window_left, window_right, sm_scale, num_splits, kernel, max_ctas)
    need = int(lib.tv_tree_attention_workspace_size(ctypes.byref(a)))
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wp = _ptr(workspace, None, "workspace") if workspace is not None else None
    wb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("tv_tree_attention", lib.tv_tree_attention(ctypes.byref(a), wp, wb, _stream(stream)))


def tv_argmax_workspace_size(rows, V, dtype):
    return int(lib.tv_argmax_workspace_size(rows, V, dtype))


def _logits_dtype(t):
    if t.dtype == torch.bfloat16:
        return TV_BF16
    if t.dtype == torch.float32:
        return TV_F32
    raise TypeError(f"logits: unsupported dtype {t.dtype}")


def tv_argmax(logits, out_idx, workspace=None, stream=None, sm_limit=None):
    """Row argmax of a 2-D ``logits`` [rows, V] (rows may be strided).  With
    ``sm_limit`` the streaming plan uses at most that many SMs (tv_argmax_sm)."""
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits: expected a 2-D tensor with unit inner stride")
    if not logits.is_cuda:
        raise ValueError("logits: must be a CUDA tensor")
    rows, V = logits.shape
    dt = _logits_dtype(logits)
    need = tv_argmax_workspace_size(rows, V, dt)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=logits.device)
    wp = _ptr(workspace, None, "workspace") if workspace is not None else None
    wb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if sm_limit is not None:
        _check("tv_argmax_sm", lib.tv_argmax_sm(
            ctypes.c_void_p(logits.data_ptr()), dt, rows, V, logits.stride(0),
            _ptr(out_idx, torch.int32, "out_idx"), wp, wb, int(sm_limit), _stream(stream)))
        return
    _check("tv_argmax", lib.tv_argmax(ctypes.c_void_p(logits.data_ptr()), dt, rows, V,
                                      logits.stride(0), _ptr(out_idx, torch.int32, "out_idx"),
                                      wp, wb, _stream(stream)))


def tv_argmax_noalloc(logits, out_idx, stream=None):
    """``tv_argmax`` without a workspace: for callers that may not allocate
    device memory (see include/tv.h).  Calls that could overlap on the GPU
    share one scratch array and must not be issued."""
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits: expected a 2-D tensor with unit inner stride")
    if not logits.is_cuda:
        raise ValueError("logits: must be a CUDA tensor")
    rows, V = logits.shape
    _check("tv_argmax_noalloc", lib.tv_argmax_noalloc(
        ctypes.c_void_p(logits.data_ptr()), _logits_dtype(logits), rows, V, logits.stride(0),
        _ptr(out_idx, torch.int32, "out_idx"), _stream(stream)))


def tv_tree_walk(tokens, parent, argmax, root_pred, status, out_tokens, n_emit, acc_nodes, n_acc,
                 stream=None):
    B, N = tokens.shape
    i32 = torch.int32
    _check("tv_tree_walk", lib.tv_tree_walk(
        _ptr(tokens, i32, "tokens"), _ptr(parent, i32, "parent"), _ptr(argmax, i32, "argmax"),
        _ptr(root_pred, i32, "root_pred"), _ptr(status, i32, "status"), B, N,
        _ptr(out_tokens, i32, "out_tokens"), _ptr(n_emit, i32, "n_emit"),
        _ptr(acc_nodes, i32, "acc_nodes"), _ptr(n_acc, i32, "n_acc"), _stream(stream)))


def tv_commit_kv(k_tree, v_tree, acc_nodes, n_acc, ctx_len_in, block_table, k_cache, v_cache,
                 ctx_len_out, status, stream=None):
    B, N, Hkv, D = k_tree.shape
    i32, bf = torch.int32, torch.bfloat16
    _check("tv_commit_kv", lib.tv_commit_kv(
        _ptr(k_tree, bf, "k_tree"), _ptr(v_tree, bf, "v_tree"), _ptr(acc_nodes, i32, "acc_nodes"),
        _ptr(n_acc, i32, "n_acc"), _ptr(ctx_len_in, i32, "ctx_len_in"),
        _ptr(block_table, i32, "block_table"), B, N, Hkv, D, block_table.shape[1],
        k_cache.shape[0], _ptr(k_cache, bf, "k_cache"), _ptr(v_cache, bf, "v_cache"),
        _ptr(ctx_len_out, i32, "ctx_len_out"), _ptr(status, i32, "status"), _stream(stream)))


def tv_topk_workspace_size(rows, V, k, dtype):
    return int(lib.tv_topk_workspace_size(rows, V, k, dtype))


def tv_topk(x, k, out_vals, out_idx, workspace=None, stream=None):
    """The k largest entries of every row of a 2-D ``x`` [rows, V] (rows may be
    strided) with their indices, in decreasing order."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x: expected a 2-D tensor with unit inner stride")
    if not x.is_cuda:
        raise ValueError("x: must be a CUDA tensor")
    rows, V = x.shape
    dt = _logits_dtype(x)
    need = tv_topk_workspace_size(rows, V, k, dt)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wp = _ptr(workspace, None, "workspace") if workspace is not None else None
    wb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("tv_topk", lib.tv_topk(ctypes.c_void_p(x.data_ptr()), dt, rows, V, x.stride(0), int(k),
                                  _ptr(out_vals, torch.float32, "out_vals"),
                                  _ptr(out_idx, torch.int32, "out_idx"), wp, wb, _stream(stream)))


def tv_build_tree(cand_lp, cand_idx, budget, w, tokens, parent, depth, score, n_nodes,
                  stream=None):
    """Best-first draft tree of ``budget`` nodes from per-depth candidate lists
    ``cand_lp`` float32 [B, L, K] / ``cand_idx`` int32 [B, L, K]."""
    B, L, K = cand_lp.shape
    i32 = torch.int32
    _check("tv_build_tree", lib.tv_build_tree(
        _ptr(cand_lp, torch.float32, "cand_lp"), _ptr(cand_idx, i32, "cand_idx"), B, L, K,
        int(budget), int(w), _ptr(tokens, i32, "tokens"), _ptr(parent, i32, "parent"),
        _ptr(depth, i32, "depth"), _ptr(score, torch.float32, "score"),
        _ptr(n_nodes, i32, "n_nodes"), _stream(stream)))


def step_args(inp, out, layers, attn_ws, argmax_ws):
    """A ``StepArgs`` for the tensors of one batch: ``inp`` holds the tree,
    sequence state and logits (as produced by ``workloads.make``), ``out`` the
    step outputs, ``layers`` a list of dicts with q / k_tree / v_tree / k_cache
    / v_cache / out tensors.  The returned object keeps the layer array alive."""
    i32, bf16 = torch.int32, torch.bfloat16
    arr = (Layer * len(layers))()
    for j, ly in enumerate(layers):
        arr[j] = Layer(_ptr(ly["q"], bf16, "q"), _ptr(ly["k_tree"], bf16, "k_tree"),
                       _ptr(ly["v_tree"], bf16, "v_tree"), _ptr(ly["k_cache"], bf16, "k_cache"),
                       _ptr(ly["v_cache"], bf16, "v_cache"), _ptr(ly["out"], bf16, "out"))
    lg = inp["logits"]
    a = StepArgs(
        tokens=_ptr(inp["tokens"], i32, "tokens"), parent=_ptr(inp["parent"], i32, "parent"),
        depth=_ptr(inp["depth"], i32, "depth"), ctx_len=_ptr(inp["ctx_len"], i32, "ctx_len"),
        root_pred=_ptr(inp["root_pred"], i32, "root_pred"),
        block_table=_ptr(inp["block_table"], i32, "block_table"),
        B=inp["B"], N=inp["N"], Hq=inp["Hq"], Hkv=inp["Hkv"], D=inp["D"],
        max_blocks=inp["max_blocks"], num_blocks=layers[0]["k_cache"].shape[0],
        window_left=inp["window_left"], sm_scale=0.0,
        num_layers=len(layers), layers=arr,
        attn_workspace=_ptr(attn_ws, None, "attn_workspace") if attn_ws is not None else None,
        attn_workspace_bytes=attn_ws.numel() if attn_ws is not None else 0,
        logits=_ptr(lg, None, "logits"), logits_dtype=_logits_dtype(lg), V=lg.shape[-1],
        argmax_workspace=_ptr(argmax_ws, None, "argmax_workspace") if argmax_ws is not None else None,
        argmax_workspace_bytes=argmax_ws.numel() if argmax_ws is not None else 0,
        anc=_ptr(out.anc, torch.int64, "anc"), pos=_ptr(out.pos, i32, "pos"),
        status=_ptr(out.status, i32, "status"), argmax=_ptr(out.argmax, i32, "argmax"),
        out_tokens=_ptr(out.out_tokens, i32, "out_tokens"), n_emit=_ptr(out.n_emit, i32, "n_emit"),
        acc_nodes=_ptr(out.acc_nodes, i32, "acc_nodes"), n_acc=_ptr(out.n_acc, i32, "n_acc"),
        ctx_len_out=_ptr(out.ctx_len_out, i32, "ctx_len_out"))
    a._layers = arr
    return a


def tv_verify_step(args, stream=None):
    _check("tv_verify_step", lib.tv_verify_step(ctypes.byref(args), _stream(stream)))


def tv_verify_graph_create(args):
    h = ctypes.c_void_p()
    _check("tv_verify_graph_create", lib.tv_verify_graph_create(ctypes.byref(args), ctypes.byref(h)))
    return h


def tv_verify_graph_launch(graph, stream=None):
    _check("tv_verify_graph_launch", lib.tv_verify_graph_launch(graph, _stream(stream)))


def tv_verify_graph_launches(graph):
    return int(lib.tv_verify_graph_launches(graph))


def tv_verify_graph_destroy(graph):
    lib.tv_verify_graph_destroy(graph)


def tv_gdn_tree_verify(state, q, k, v, alpha, beta, anc, out, u, g, status=None, kernel=0,
                       stream=None):
    """GDN outputs of every tree node from the committed state (include/tv_gdn.h).
    state float32 [B, Hv, dv, dk] (S^T); q, k bf16 [B, N, Hk, dk]; v bf16
    [B, N, Hv, dv]; alpha, beta float32 [B, N, Hv]; anc int64 [B, N]."""
    B, N, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    f32, bf16 = torch.float32, torch.bfloat16
    _check("tv_gdn_tree_verify", lib.tv_gdn_tree_verify(
        _ptr(state, f32, "state"), _ptr(q, bf16, "q"), _ptr(k, bf16, "k"), _ptr(v, bf16, "v"),
        _ptr(alpha, f32, "alpha"), _ptr(beta, f32, "beta"), _ptr(anc, torch.int64, "anc"),
        B, N, Hk, Hv, dk, dv, _ptr(out, f32, "out"), _ptr(u, f32, "u"), _ptr(g, f32, "g"),
        int(kernel), _ptr(status, torch.int32, "status") if status is not None else None,
        _stream(stream)))


def tv_gdn_commit(state_in, k, u, alpha, acc_nodes, n_acc, state_out, status=None, stream=None):
    """The GDN state after the accepted path (include/tv_gdn.h)."""
    B, N, Hk, dk = k.shape
    Hv, dv = u.shape[2], u.shape[3]
    f32, i32 = torch.float32, torch.int32
    _check("tv_gdn_commit", lib.tv_gdn_commit(
        _ptr(state_in, f32, "state_in"), _ptr(k, torch.bfloat16, "k"), _ptr(u, f32, "u"),
        _ptr(alpha, f32, "alpha"), _ptr(acc_nodes, i32, "acc_nodes"), _ptr(n_acc, i32, "n_acc"),
        B, N, Hk, Hv, dk, dv, _ptr(state_out, f32, "state_out"),
        _ptr(status, i32, "status") if status is not None else None, _stream(stream)))


def tv_debug_withhold_arrival(cta):
    """Test hook (include/tv_debug.h): from the next launch on, the tensor-core
    kernels' CTA ``cta`` waits for a barrier arrival that never comes, so its
    bounded wait runs out; a negative ``cta`` disarms it."""
    lib.tv_debug_withhold_arrival(int(cta))


DEBUG_RECORDS = ("tree.cu", "argmax.cu", "attention.cu", "attention_tc.cu", "attention_tc256.cu",
                 "draft.cu", "gdn.cu")


def tv_debug_check_failures(clear=False):
    """Index checks of the TV_DEBUG build that failed since the last clear:
    (count, first failing source file or None, its line).  Always (0, None, 0)
    for the release build (tv_debug_checks_enabled() == 0)."""
    line = ctypes.c_uint(0)
    which = ctypes.c_int(-1)
    n = int(lib.tv_debug_check_failures(ctypes.byref(line), ctypes.byref(which), int(bool(clear))))
    if n == 0xFFFFFFFF:
        raise TvError("tv_debug_check_failures", TV_ERR_CUDA)
    return n, (DEBUG_RECORDS[which.value] if which.value >= 0 else None), int(line.value)


def tv_debug_checks_enabled():
    return bool(lib.tv_debug_checks_enabled())

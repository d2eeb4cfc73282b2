"""CPU oracle for the tree speculative-decoding verify step (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this package.  The product library never loads it, and it imports
nothing from the product package: the two share no code.

The arithmetic lives in ``tv_oracle.c`` (fp64 / integer, one plain loop nest per
step, OpenMP over independent (sequence, head) pairs).  This module compiles it
with the host C compiler on first use and wraps each function for numpy arrays.
bf16 tensors travel as their raw 16-bit patterns (``numpy.uint16``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``tv_oracle.c`` into ``oracle/_build/liboracle.so`` (host gcc)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # no OpenMP runtime
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_longlong
            lib.oracle_num_threads.restype = I
            lib.oracle_ancestors.argtypes = [I, I, P, P, P, P, P, P]
            lib.oracle_attention.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P,
                                             P, P, P, I, ctypes.c_double, P, P]
            lib.oracle_argmax.argtypes = [P, I, L, L, L, P]
            lib.oracle_walk.argtypes = [I, I, P, P, P, P, P, P, P, P, P]
            lib.oracle_commit.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P,
                                          P, P, P, P]
            for f in ("oracle_ancestors", "oracle_attention", "oracle_argmax",
                      "oracle_walk", "oracle_commit"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use (1 without OpenMP)."""
    return int(_load().oracle_num_threads())


def ancestors(parent, depth, ctx_len):
    """Ancestor-or-self mask uint8[B,N,N], positions int32[B,N], status int32[B]."""
    parent = _c(parent, np.int32)
    depth = _c(depth, np.int32)
    ctx_len = _c(ctx_len, np.int32)
    B, N = parent.shape
    mask = np.zeros((B, N, N), np.uint8)
    pos = np.zeros((B, N), np.int32)
    status = np.zeros((B,), np.int32)
    _load().oracle_ancestors(B, N, _ptr(parent), _ptr(depth), _ptr(ctx_len),
                             _ptr(mask), _ptr(pos), _ptr(status))
    return mask, pos, status


def dense_bias(mask_b, ctx_len_b):
    """The additive attention bias of one sequence, shape [N, ctx+N].

    Context columns are 0 (every node sees the whole context), node columns are
    0 for ancestor-or-self and -inf otherwise -- the layout whose shape the
    DDTree page prints for its 32-node tree over 100 context tokens.
    """
    N = mask_b.shape[0]
    bias = np.zeros((N, ctx_len_b + N), np.float64)
    bias[:, ctx_len_b:] = np.where(mask_b.astype(bool), 0.0, -np.inf)
    return bias


def attention(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_len, mask, pos,
              window_left=-1, sm_scale=None, row_sel=None):
    """fp64 tree attention; bf16 inputs given as uint16 bit patterns.

    Returns float64 [B, N, Hq, D].  ``row_sel`` (bool [B, Hq]) limits the work
    to selected (sequence, head) pairs; other rows come back as NaN.
    """
    q = _c(q, np.uint16)
    k_tree = _c(k_tree, np.uint16)
    v_tree = _c(v_tree, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    block_table = _c(block_table, np.int32)
    ctx_len = _c(ctx_len, np.int32)
    mask = _c(mask, np.uint8)
    pos = _c(pos, np.int32)
    B, N, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    BS = k_cache.shape[2]
    max_blocks = block_table.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    sel = None
    if row_sel is not None:
        sel = _c(np.asarray(row_sel, bool).reshape(B * Hq), np.uint8)
    out = np.full((B, N, Hq, D), np.nan, np.float64)
    _load().oracle_attention(B, N, Hq, Hkv, D, BS, max_blocks, _ptr(q), _ptr(k_tree),
                             _ptr(v_tree), _ptr(k_cache), _ptr(v_cache),
                             _ptr(block_table), _ptr(ctx_len), _ptr(mask), _ptr(pos),
                             int(window_left), float(sm_scale), _ptr(sel), _ptr(out))
    return out


def argmax(x, dtype: str):
    """Lowest-index argmax of each row; ``dtype`` 'f32' (float32) or 'bf16' (uint16 bits)."""
    if dtype == "f32":
        x = _c(x, np.float32)
        code = 0
    elif dtype == "bf16":
        x = _c(x, np.uint16)
        code = 1
    else:
        raise ValueError(dtype)
    rows, V = x.shape
    idx = np.zeros((rows,), np.int32)
    _load().oracle_argmax(_ptr(x), code, rows, V, V, _ptr(idx))
    return idx


def walk(tokens, parent, argmax_idx, root_pred, status=None):
    """Greedy tree walk: (out_tokens[B,N+1], n_emit[B], acc_nodes[B,N], n_acc[B])."""
    tokens = _c(tokens, np.int32)
    parent = _c(parent, np.int32)
    argmax_idx = _c(argmax_idx, np.int32)
    root_pred = _c(root_pred, np.int32)
    st = None if status is None else _c(status, np.int32)
    B, N = tokens.shape
    out_tokens = np.zeros((B, N + 1), np.int32)
    n_emit = np.zeros((B,), np.int32)
    acc_nodes = np.zeros((B, N), np.int32)
    n_acc = np.zeros((B,), np.int32)
    _load().oracle_walk(B, N, _ptr(tokens), _ptr(parent), _ptr(argmax_idx),
                        _ptr(root_pred), _ptr(st), _ptr(out_tokens), _ptr(n_emit),
                        _ptr(acc_nodes), _ptr(n_acc))
    return out_tokens, n_emit, acc_nodes, n_acc


def commit(k_tree, v_tree, acc_nodes, n_acc, ctx_len, block_table, k_cache, v_cache):
    """Commit accepted rows into copies of the caches.

    Returns (k_cache', v_cache', ctx_len_out, status); the inputs are not modified.
    """
    k_tree = _c(k_tree, np.uint16)
    v_tree = _c(v_tree, np.uint16)
    acc_nodes = _c(acc_nodes, np.int32)
    n_acc = _c(n_acc, np.int32)
    ctx_len = _c(ctx_len, np.int32)
    block_table = _c(block_table, np.int32)
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    B, N, Hkv, D = k_tree.shape
    num_blocks, _, BS, _ = kc.shape
    max_blocks = block_table.shape[1]
    ctx_out = np.zeros((B,), np.int32)
    status = np.zeros((B,), np.int32)
    _load().oracle_commit(B, N, Hkv, D, BS, max_blocks, num_blocks, _ptr(k_tree),
                          _ptr(v_tree), _ptr(acc_nodes), _ptr(n_acc), _ptr(ctx_len),
                          _ptr(block_table), _ptr(kc), _ptr(vc), _ptr(ctx_out),
                          _ptr(status))
    return kc, vc, ctx_out, status


def verify_step(inp, row_sel=None):
    """The whole step on the CPU: ancestors -> attention -> argmax -> walk -> commit.

    ``inp`` is a dict of numpy arrays (bf16 as uint16), as produced by
    ``workloads.to_numpy``.  Returns a dict of every step's outputs.
    """
    mask, pos, status = ancestors(inp["parent"], inp["depth"], inp["ctx_len"])
    out = attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"],
                    inp["v_cache"], inp["block_table"], inp["ctx_len"], mask, pos,
                    window_left=inp["window_left"], row_sel=row_sel)
    logits = inp["logits"]
    B, N = inp["tokens"].shape
    am = argmax(logits.reshape(B * N, -1), inp["logits_dtype"]).reshape(B, N)
    out_tokens, n_emit, acc_nodes, n_acc = walk(inp["tokens"], inp["parent"], am,
                                                inp["root_pred"], status)
    kc, vc, ctx_out, cstatus = commit(inp["k_tree"], inp["v_tree"], acc_nodes, n_acc,
                                      inp["ctx_len"], inp["block_table"],
                                      inp["k_cache"], inp["v_cache"])
    status = np.where(status != 0, status, cstatus).astype(np.int32)
    return dict(mask=mask, pos=pos, status=status, attn=out, argmax=am,
                out_tokens=out_tokens, n_emit=n_emit, acc_nodes=acc_nodes,
                n_acc=n_acc, k_cache=kc, v_cache=vc, ctx_len_out=ctx_out)

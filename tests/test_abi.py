"""The C ABI without a GPU: the library builds, loads, exports every function
that the headers under include/ declare, and rejects bad arguments on the host
before any launch."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path)


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(tv_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_step(lib):
    names = declared_functions()
    for f in ("tv_build_ancestors", "tv_tree_attention", "tv_argmax", "tv_tree_walk",
              "tv_commit_kv"):
        assert f in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names
    for f in names:
        assert hasattr(lib, f), f"{f} declared in include/ but not exported"


def test_binding_lists_every_export():
    import tree_speculative_decoding_build_gb300 as tv
    assert sorted(tv.EXPORTS) == declared_functions()


def test_status_strings(lib):
    lib.tv_status_string.restype = ctypes.c_char_p
    assert lib.tv_status_string(0) == b"ok"
    assert b"tree" in lib.tv_status_string(2)
    assert lib.tv_status_string(99) == b"unknown status"


def test_host_argument_checks(lib):
    P = ctypes.c_void_p
    lib.tv_build_ancestors.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P]
    assert lib.tv_build_ancestors(None, None, None, 1, 65, None, None, None, None) == 1
    assert lib.tv_build_ancestors(None, None, None, -1, 4, None, None, None, None) == 1
    assert lib.tv_build_ancestors(None, None, None, 0, 4, None, None, None, None) == 0
    lib.tv_tree_walk.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P, P]
    assert lib.tv_tree_walk(None, None, None, None, None, 2, 8, None, None, None, None, None) == 1
    lib.tv_argmax.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                              P, P, ctypes.c_size_t, P]
    assert lib.tv_argmax(None, 7, 1, 1, 1, None, None, 0, None) == 5
    assert lib.tv_argmax(None, 1, 1, 0, 1, None, None, 0, None) == 1
    assert lib.tv_argmax(None, 1, 0, 10, 10, None, None, 0, None) == 0
    lib.tv_commit_kv.argtypes = [P] * 6 + [ctypes.c_int] * 6 + [P] * 5
    assert lib.tv_commit_kv(*([None] * 6), 1, 4, 8, 12, 4, 4, *([None] * 5)) == 5   # D % 8
    assert lib.tv_commit_kv(*([None] * 6), 1, 4, 8, 128, 4, 4, *([None] * 5)) == 1


def test_attention_argument_checks(lib):
    from tree_speculative_decoding_build_gb300._lib import AttnArgs
    lib.tv_tree_attention.argtypes = [ctypes.POINTER(AttnArgs), ctypes.c_void_p, ctypes.c_size_t,
                                      ctypes.c_void_p]
    a = AttnArgs()
    a.B, a.N, a.Hq, a.Hkv, a.D, a.block_size, a.max_blocks = 1, 8, 4, 2, 64, 16, 4
    a.window_left, a.window_right = -1, 0
    assert lib.tv_tree_attention(ctypes.byref(a), None, 0, None) == 1          # NULL pointers
    a.D = 96
    assert lib.tv_tree_attention(ctypes.byref(a), None, 0, None) == 5
    a.D, a.block_size = 64, 32
    assert lib.tv_tree_attention(ctypes.byref(a), None, 0, None) == 5
    a.block_size, a.Hq = 16, 5
    assert lib.tv_tree_attention(ctypes.byref(a), None, 0, None) == 1
    a.Hq, a.N = 8, 65
    assert lib.tv_tree_attention(ctypes.byref(a), None, 0, None) == 1
    a.N, a.B = 8, 0
    assert lib.tv_tree_attention(ctypes.byref(a), None, 0, None) == 0          # nothing to do


def test_draft_host_argument_checks(lib):
    P, I, L, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.tv_topk.argtypes = [P, I, L, L, L, I, P, P, P, S, P]
    lib.tv_topk.restype = I
    assert lib.tv_topk(None, 7, 1, 8, 8, 2, None, None, None, 0, None) == 5   # dtype
    assert lib.tv_topk(None, 0, 1, 8, 8, 0, None, None, None, 0, None) == 1   # k < 1
    assert lib.tv_topk(None, 0, 1, 8, 8, 9, None, None, None, 0, None) == 1   # k > V
    assert lib.tv_topk(None, 0, 1, 64, 64, 17, None, None, None, 0, None) == 1  # k > 16
    assert lib.tv_topk(None, 0, 1, 8, 4, 2, None, None, None, 0, None) == 1   # stride < V
    assert lib.tv_topk(None, 0, 0, 8, 8, 2, None, None, None, 0, None) == 0   # no rows
    lib.tv_build_tree.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P, P]
    lib.tv_build_tree.restype = I
    args = [None] * 6
    assert lib.tv_build_tree(None, None, 2, 5, 10, 65, 1, *args) == 1  # budget > 64
    assert lib.tv_build_tree(None, None, 2, 5, 10, 32, 0, *args) == 1  # w < 1
    assert lib.tv_build_tree(None, None, 2, 0, 10, 32, 1, *args) == 1  # L < 1
    assert lib.tv_build_tree(None, None, 2, 5, 10, 32, 1, *args) == 1  # NULL pointers
    assert lib.tv_build_tree(None, None, 0, 5, 10, 32, 1, *args) == 0  # empty batch
    lib.tv_topk_workspace_size.argtypes = [L, L, I, I]
    lib.tv_topk_workspace_size.restype = S
    assert lib.tv_topk_workspace_size(1, 8, 0, 0) == 0


def test_graph_host_argument_checks(lib):
    P = ctypes.c_void_p
    lib.tv_verify_step.argtypes = [P, P]
    lib.tv_verify_step.restype = ctypes.c_int
    assert lib.tv_verify_step(None, None) == 1
    lib.tv_verify_graph_create.argtypes = [P, ctypes.POINTER(P)]
    lib.tv_verify_graph_create.restype = ctypes.c_int
    h = P()
    assert lib.tv_verify_graph_create(None, ctypes.byref(h)) == 1 and not h.value
    assert lib.tv_verify_graph_create(None, None) == 1
    lib.tv_verify_graph_launch.argtypes = [P, P]
    lib.tv_verify_graph_launch.restype = ctypes.c_int
    assert lib.tv_verify_graph_launch(None, None) == 1
    lib.tv_verify_graph_launches.argtypes = [P]
    assert lib.tv_verify_graph_launches(None) == 0
    lib.tv_verify_graph_destroy.argtypes = [P]
    lib.tv_verify_graph_destroy(None)


def test_graph_rejects_aliased_ctx_len(lib):
    """Two layers whose commits share one ctx_len array for input and output
    would commit the second layer's rows n_acc positions too far: rejected on
    the host before anything is enqueued (no GPU needed)."""
    from tree_speculative_decoding_build_gb300._lib import Layer, StepArgs
    P = ctypes.c_void_p
    lib.tv_verify_step.argtypes = [ctypes.POINTER(StepArgs), P]
    lib.tv_verify_step.restype = ctypes.c_int
    lib.tv_verify_graph_create.argtypes = [ctypes.POINTER(StepArgs), ctypes.POINTER(P)]
    lib.tv_verify_graph_create.restype = ctypes.c_int
    layers = (Layer * 2)()
    a = StepArgs(B=1, N=8, Hq=4, Hkv=2, D=64, max_blocks=4, num_blocks=4, window_left=-1,
                 num_layers=2, layers=layers)
    a.ctx_len = a.ctx_len_out = P(0x1000)
    assert lib.tv_verify_step(ctypes.byref(a), None) == 1
    h = P()
    assert lib.tv_verify_graph_create(ctypes.byref(a), ctypes.byref(h)) == 1 and not h.value


def test_gdn_host_argument_checks(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.tv_gdn_tree_verify.argtypes = [P] * 7 + [I] * 6 + [P] * 3 + [I, P, P]
    lib.tv_gdn_tree_verify.restype = I
    nul = [None] * 7

    def verify(B, N, Hk, Hv, dk, dv, kernel):
        return lib.tv_gdn_tree_verify(*nul, B, N, Hk, Hv, dk, dv, None, None, None, kernel, None,
                                      None)
    assert verify(1, 32, 1, 2, 128, 128, 4) == 1    # kernel out of range
    assert verify(1, 32, 1, 2, 128, 128, -1) == 1
    assert verify(1, 65, 1, 2, 128, 128, 0) == 1    # N > 64
    assert verify(1, 32, 2, 3, 128, 128, 0) == 1    # Hv % Hk
    assert verify(1, 32, 1, 2, 96, 96, 0) == 1      # d_v not a multiple of 64
    assert verify(1, 32, 1, 2, 96, 128, 2) == 5     # tensor cores: d_k 64 or 128
    assert verify(1, 33, 1, 2, 128, 128, 3) == 5    # pipeline: N <= 32
    assert verify(1, 32, 1, 2, 32, 64, 3) == 5      # pipeline: d_k 64 or 128
    assert verify(0, 32, 1, 2, 128, 128, 3) == 0    # empty batch
    assert verify(1, 32, 1, 2, 128, 128, 3) == 1    # NULL pointers
    lib.tv_gdn_commit.argtypes = [P] * 6 + [I] * 6 + [P, P, P]
    lib.tv_gdn_commit.restype = I
    assert lib.tv_gdn_commit(*[None] * 6, 1, 32, 1, 2, 128, 128, None, None, None) == 1
    assert lib.tv_gdn_commit(*[None] * 6, 0, 32, 1, 2, 128, 128, None, None, None) == 0

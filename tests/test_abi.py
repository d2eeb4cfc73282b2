"""The C ABI without a GPU: the library builds, loads, exports every function
that include/tv.h declares, and rejects bad arguments on the host before any
launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tv.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(tv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_step(lib):
    names = declared_functions()
    for f in ("tv_build_ancestors", "tv_tree_attention", "tv_argmax", "tv_tree_walk",
              "tv_commit_kv"):
        assert f in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names
    for f in names:
        assert hasattr(lib, f), f"{f} declared in tv.h but not exported"


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

"""tv_argmax_noalloc, the argmax entry point for callers that cannot allocate
device memory (a serving loop whose memory is owned by one pool, a plugin host
that only hands over input and output buffers, a decode loop where cudaMalloc's
possible device synchronisation is not allowed).

It must give exactly what tv_argmax gives, call after call, although every call
reuses the same fixed scratch array inside the library.  This file is named to
be collected last, so a run that stops at the first failure has already run
every other test.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

SHAPES = [
    (16, 262144, torch.bfloat16),   # few rows: split into many chunks (uses the scratch)
    (3, 100003, torch.float32),     # odd length, chunked
    (8, 1024, torch.float32),
    (2048, 151936, torch.bfloat16), # one chunk per row: no scratch needed
]


@pytest.mark.parametrize("rows,V,dtype", SHAPES)
def test_noalloc_matches_argmax_on_consecutive_calls(rows, V, dtype):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_decoding_build_gb300 as tv
    g = torch.Generator(device="cuda").manual_seed(rows + V)
    for call in range(2):
        x = torch.randn(rows, V, generator=g, device="cuda").to(dtype)
        x[:, ::131] = 2.5                       # ties: the lowest index must win
        x[call % rows, (V * (call + 1)) // 3] = 40.0
        ref = torch.empty(rows, dtype=torch.int32, device="cuda")
        got = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
        tv.tv_argmax(x, ref)
        tv.tv_argmax_noalloc(x, got)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {call}"

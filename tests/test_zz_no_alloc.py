"""tv_argmax_noalloc, the argmax entry point for callers that cannot allocate
device memory (a serving loop whose memory is owned by one pool, a plugin host
that only hands over input and output buffers, a decode loop where cudaMalloc's
possible device synchronisation is not allowed).

It must give exactly what tv_argmax and the oracle's scalar argmax give, call
after call, although every call reuses the same fixed scratch array inside the
library.  This file is named to be collected last, so a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

# (rows, V, dtype, whether the plan writes partials into the scratch array)
SHAPES = [
    (16, 262144, torch.bfloat16, True),    # few long rows: each row cut into many chunks
    (3, 100003, torch.float32, True),      # odd length: chunked, unaligned rows
    (8, 1024, torch.float32, False),       # small: one chunk per row, no partials
    (2048, 151936, torch.bfloat16, True),  # streaming plan: two partials per warp
]


@pytest.mark.parametrize("rows,V,dtype,scratch", SHAPES)
def test_noalloc_matches_argmax_and_oracle_on_consecutive_calls(rows, V, dtype, scratch,
                                                                 oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tree_speculative_decoding_build_gb300 as tv
    tdt = tv.TV_BF16 if dtype == torch.bfloat16 else tv.TV_F32
    # the plan's partial count is what tv_argmax_workspace_size reports for
    # dense aligned rows: pin which branch (scratch used or not) each shape takes
    assert (tv.tv_argmax_workspace_size(rows, V, tdt) > 0) == scratch
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
        assert torch.equal(got, ref), f"call {call}: differs from tv_argmax"
        if dtype == torch.bfloat16:
            host = x.cpu().view(torch.int16).numpy().view(np.uint16)
            want = oracle_mod.argmax(host, "bf16")
        else:
            want = oracle_mod.argmax(x.cpu().numpy(), "f32")
        assert np.array_equal(got.cpu().numpy(), want), f"call {call}: differs from the oracle"

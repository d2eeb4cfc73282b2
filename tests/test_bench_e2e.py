"""Host logic of bench.py's end-to-end loop, on the CPU with stand-in streams.

The loop double-buffers the device inputs and uploads step s+1 on copy streams
while step s runs.  With every stream and event replaced by a no-op (so each
copy completes when it is issued), these tests check what the loop issues:
every step runs on a buffer holding the whole upload (big tensors arrive in
chunks that must cover them exactly), the buffers alternate, each step's
results are read back, and the warm-up is not counted in the time.
"""
import contextlib
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _Event:
    def __init__(self, enable_timing=False):
        pass

    def record(self, stream=None):
        pass

    def elapsed_time(self, other):
        return 6.0  # ms between the two timing events


class _Stream:
    def __init__(self, device=None):
        self.waits = 0

    def wait_event(self, ev):
        self.waits += 1


@pytest.fixture
def fake_cuda(monkeypatch):
    monkeypatch.setattr(torch.cuda, "Stream", _Stream)
    monkeypatch.setattr(torch.cuda, "Event", _Event)
    monkeypatch.setattr(torch.cuda, "stream", lambda s: contextlib.nullcontext())
    monkeypatch.setattr(torch.cuda, "synchronize", lambda device=None: None)


@pytest.mark.parametrize("steps", [1, 2, 3, 8])
def test_every_step_sees_its_whole_upload(fake_cuda, steps):
    # a small tensor and one past the 64 MB chunking threshold (cut in four)
    host = {"tokens": torch.arange(37, dtype=torch.int32),
            "logits": torch.zeros(3, (64 << 20) // 2 // 3 + 11, dtype=torch.bfloat16)}
    bufs = [{k: torch.full_like(v, -1) for k, v in host.items()} for _ in range(2)]
    seen = []
    out = torch.zeros(4)
    res = torch.zeros(4)

    host["logits"].copy_(torch.randn(host["logits"].shape))

    def step(d):
        b = next(i for i, x in enumerate(bufs) if x is d)
        assert torch.equal(d["tokens"], host["tokens"])
        assert torch.equal(d["logits"], host["logits"])
        seen.append(b)
        out.fill_(len(seen))
        d["tokens"].fill_(-1)          # spent: the next use of this buffer needs a new upload
        d["logits"].fill_(-1)

    ms = bench.pipelined_e2e(step, host, bufs, [(res, out)], steps, _Stream(), "cpu")
    assert ms == pytest.approx(6.0 / steps)
    assert len(seen) == 2 + steps                   # two warm-up steps, then the timed ones
    assert seen[2:] == [s % 2 for s in range(steps)]
    assert res[0].item() == len(seen)               # the last step's results were read back


def test_passes_report_the_median_and_time_only_the_passes(monkeypatch):
    # stand-in events whose timed intervals are 9, 3 and 6 ms: the median is 6
    lengths = iter([9.0, 3.0, 6.0])

    class _TimedEvent(_Event):
        def elapsed_time(self, other):
            return next(lengths)

    monkeypatch.setattr(torch.cuda, "Stream", _Stream)
    monkeypatch.setattr(torch.cuda, "Event", _TimedEvent)
    monkeypatch.setattr(torch.cuda, "stream", lambda s: contextlib.nullcontext())
    monkeypatch.setattr(torch.cuda, "synchronize", lambda device=None: None)
    host = {"tokens": torch.arange(5, dtype=torch.int32)}
    bufs = [{k: torch.zeros_like(v) for k, v in host.items()} for _ in range(2)]
    calls = []

    def step(d):
        assert torch.equal(d["tokens"], host["tokens"])
        calls.append(1)

    steps = 3
    ms = bench.pipelined_e2e(step, host, bufs, [], steps, _Stream(), "cpu", passes=3)
    assert ms == pytest.approx(6.0 / steps)
    assert len(calls) == 2 + 3 * steps            # one warm-up, then every pass

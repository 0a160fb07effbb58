"""Host logic of the binding's cached SSD workspace (no GPU): one workspace
per (device, stream), reused while large enough, replaced when a call needs
more, and allocated with the call's stream current."""
import contextlib

import torch

import selective_state_update_gb300 as ssu


class _FakeStream:
    def __init__(self, handle, device=None):
        self.cuda_stream = handle


def test_workspace_per_device_and_stream(monkeypatch):
    allocated = []
    current = {"stream": None}

    @contextlib.contextmanager
    def fake_stream_ctx(s):
        prev, current["stream"] = current["stream"], s.cuda_stream
        yield
        current["stream"] = prev

    def fake_empty(n, dtype=None, device=None):
        allocated.append((n, device, current["stream"]))
        return torch.zeros(n, dtype=torch.uint8)

    monkeypatch.setattr(ssu, "_SSD_WORKSPACE", {})
    monkeypatch.setattr(ssu, "_stream", lambda stream: stream if isinstance(stream, int) else 7)
    monkeypatch.setattr(torch.cuda, "ExternalStream", _FakeStream)
    monkeypatch.setattr(torch.cuda, "stream", fake_stream_ctx)
    monkeypatch.setattr(torch, "empty", fake_empty)

    a = ssu._ssd_workspace("cuda:0", 1000, None)       # the current stream (handle 7)
    assert allocated == [(1000, "cuda:0", None)]     # no stream switch
    assert ssu._ssd_workspace("cuda:0", 800, None) is a  # reused while large enough
    b = ssu._ssd_workspace("cuda:0", 500, 11)           # another stream: its own, allocated on it
    assert b is not a and allocated[-1] == (500, "cuda:0", 11)
    c = ssu._ssd_workspace("cuda:0", 4000, None)        # grows
    assert c is not a and c.numel() == 4000 and allocated[-1] == (4000, "cuda:0", None)
    assert ssu._ssd_workspace("cuda:0", 400, 11) is b
    d = ssu._ssd_workspace("cuda:1", 10, None)          # another device
    assert d.numel() == 256 and allocated[-1] == (256, "cuda:1", None)
    assert len(allocated) == 4

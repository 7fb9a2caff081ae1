"""Host logic of the Python binding, on CPU: the workspace that the default
calls pass to the library (one per device and stream, zeroed on the stream
that uses it, never created inside a graph capture) and the entry point each
call reaches. The CUDA runtime pieces the binding touches (current stream,
stream context, capture status, current device and device context) and the
library are fakes
that record what they are asked; no kernel runs."""

import contextlib

import pytest

torch = pytest.importorskip("torch")

from sparse_attention_indexer_fp32_gb300 import _binding  # noqa: E402


class FakeStream:
    def __init__(self, handle, capturing=False):
        self.cuda_stream = handle
        self.capturing = capturing


class FakeLib:
    """Records the entry point and the stream/workspace of every call."""

    def __init__(self):
        self.calls = []

    def _record(self, name, args):
        self.calls.append((name, args))
        return 0

    def topk_ragged(self, *args):
        return self._record("topk_ragged", args)

    def topk_ragged_ws(self, *args):
        return self._record("topk_ragged_ws", args)

    def topk_paged(self, *args):
        return self._record("topk_paged", args)

    def topk_paged_ws(self, *args):
        return self._record("topk_paged_ws", args)


@pytest.fixture
def fake_cuda(monkeypatch):
    state = {"current": FakeStream(100), "zeroed_on": []}
    lib = FakeLib()

    @contextlib.contextmanager
    def stream_ctx(s):
        prev, state["current"] = state["current"], s
        try:
            yield
        finally:
            state["current"] = prev

    real_zeros = torch.zeros

    def zeros(*args, **kwargs):  # torch.zeros itself is patched: record only workspaces (uint8)
        if kwargs.get("dtype") is torch.uint8:
            state["zeroed_on"].append(state["current"].cuda_stream)
        kwargs.pop("device", None)
        return real_zeros(*args, **kwargs)

    monkeypatch.setattr(_binding.torch.cuda, "current_stream", lambda device=None: state["current"])
    monkeypatch.setattr(_binding.torch.cuda, "stream", stream_ctx)
    monkeypatch.setattr(_binding.torch.cuda, "is_current_stream_capturing",
                        lambda: state["current"].capturing)
    monkeypatch.setattr(_binding.torch.cuda, "device", lambda d: contextlib.nullcontext())
    monkeypatch.setattr(_binding.torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(_binding.torch, "zeros", zeros)
    monkeypatch.setattr(_binding, "load_library", lambda path=None: lib)
    monkeypatch.setattr(_binding, "workspace_bytes", lambda k=2048, max_split_rows=0: 4096)
    monkeypatch.setattr(_binding, "_prepare",
                        lambda s, l, k, out: (s.shape[0], s.shape[1],
                                              out if out is not None else real_zeros((s.shape[0], k),
                                                                                     dtype=torch.int32)))
    monkeypatch.setattr(_binding, "_workspaces", {})
    return state, lib


def _inputs(B=4, stride=64):
    return torch.zeros((B, stride)), torch.zeros(B, dtype=torch.int32)


def test_default_call_gets_one_workspace_per_stream(fake_cuda):
    state, lib = fake_cuda
    s, l = _inputs()
    _binding.topk_ragged(s, l, 8)
    _binding.topk_ragged(s, l, 8)
    side = FakeStream(200)
    _binding.topk_ragged(s, l, 8, stream=side)
    names = [c[0] for c in lib.calls]
    assert names == ["topk_ragged_ws"] * 3
    # the last argument is the stream handle; the two before it the workspace
    ws_ptrs = [c[1][-3] for c in lib.calls]
    assert ws_ptrs[0] == ws_ptrs[1] != ws_ptrs[2]
    assert [c[1][-1] for c in lib.calls] == [100, 100, 200]
    assert [c[1][-2] for c in lib.calls] == [4096] * 3
    assert set(_binding._workspaces) == {(-1, 100), (-1, 200)}


def test_workspace_is_zeroed_on_the_stream_that_uses_it(fake_cuda):
    """A call given another stream than the current one zeroes its new
    workspace on that stream (ordered before the call), not on the current
    stream."""
    state, lib = fake_cuda
    s, l = _inputs()
    _binding.topk_ragged(s, l, 8, stream=FakeStream(300))
    assert state["zeroed_on"] == [300]
    assert state["current"].cuda_stream == 100  # the current stream is restored


def test_capture_without_workspace_takes_the_unsplit_entry_point(fake_cuda):
    state, lib = fake_cuda
    s, l = _inputs()
    pt = torch.zeros((4, 1), dtype=torch.int32)
    capturing = FakeStream(400, capturing=True)
    with _binding.torch.cuda.stream(capturing):
        _binding.topk_ragged(s, l, 8)
        _binding.topk_paged(s, l, 8, pt, 64)
    assert [c[0] for c in lib.calls] == ["topk_ragged", "topk_paged"]
    assert state["zeroed_on"] == []
    assert (-1, 400) not in _binding._workspaces
    # once the capture has ended, the same stream gets its workspace
    capturing.capturing = False
    _binding.topk_ragged(s, l, 8, stream=capturing)
    assert lib.calls[-1][0] == "topk_ragged_ws"
    assert state["zeroed_on"] == [400]


def test_capture_with_existing_workspace_keeps_the_split_path(fake_cuda):
    state, lib = fake_cuda
    s, l = _inputs()
    st = FakeStream(500)
    _binding.topk_ragged(s, l, 8, stream=st)  # eager warm-up creates the workspace
    st.capturing = True
    _binding.topk_ragged(s, l, 8, stream=st)
    assert [c[0] for c in lib.calls] == ["topk_ragged_ws", "topk_ragged_ws"]
    assert lib.calls[0][1][-3] == lib.calls[1][1][-3]
    assert state["zeroed_on"] == [500]


def test_split_false_never_creates_a_workspace(fake_cuda):
    state, lib = fake_cuda
    s, l = _inputs()
    _binding.topk_ragged(s, l, 8, split=False)
    assert [c[0] for c in lib.calls] == ["topk_ragged"]
    assert _binding._workspaces == {} and state["zeroed_on"] == []

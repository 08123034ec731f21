"""The Python binding's marshalling: with no stream given, every entry
point runs on torch's current stream, which the binding reads through
torch's C-level query; checked against torch.cuda.current_stream() on the
default stream and inside a stream context, on the current device."""
import pytest
import torch

from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def test_current_stream_matches_torch():
    assert cr._current_stream() == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert cr._current_stream() == s.cuda_stream == torch.cuda.current_stream().cuda_stream
    assert cr._current_stream() == torch.cuda.current_stream().cuda_stream


def test_call_on_side_stream_is_ordered():
    """An all-reduce issued with no explicit stream inside a stream context
    runs on that stream: work queued before it on the same stream is seen."""
    n, count = 4, 1 << 20
    bufs = [torch.zeros(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for r, b in enumerate(bufs):
            b.fill_(float(r + 1))
        cr.cr_all_reduce(bufs, count, "f32", "sum", bufs, "f32")
    s.synchronize()
    for b in bufs:
        assert torch.all(b == 10.0)

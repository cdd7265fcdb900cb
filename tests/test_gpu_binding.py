"""The Python binding's stream handling on the GPU: the handle it passes to
the library is torch's current stream, on the default stream, on a side
stream, and while a CUDA graph is being captured."""
import pytest
import torch

from paged_kv_cache_29_gb300 import _binding as pa

pytestmark = pytest.mark.gpu


def _expected():
    return torch.cuda.current_stream().cuda_stream or None


def test_stream_handle_is_the_current_stream():
    assert pa._stream(None) == _expected()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert pa._stream(None) == _expected() == side.cuda_stream
    assert pa._stream(side) == side.cuda_stream
    g = torch.cuda.CUDAGraph()
    seen = []
    with torch.cuda.graph(g):
        seen.append((pa._stream(None), _expected()))
        torch.zeros(1, device="cuda").add_(1)
    assert seen[0][0] == seen[0][1]

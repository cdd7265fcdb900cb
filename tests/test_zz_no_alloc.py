"""pa_decode_noalloc (the decode call on the library's fixed device scratch)
against pa_decode with a caller-provided workspace, through the C ABI.

The file name sorts last so that the call also runs after every other test
has used the library in this process; it passes on its own as well."""
import numpy as np
import pytest
import torch

from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

from gpu_helpers import DeviceStep  # noqa: E402


def _noalloc(ds: DeviceStep, out: torch.Tensor) -> None:
    s = ds.step
    pa.pa_decode_noalloc(ds.q, ds.k_cache, ds.v_cache, ds.tables, ds.lens, s.scale, out,
                         s.max_context_len, error_word=ds.err)


@pytest.mark.parametrize("name", ["tiny", "7b_mha", "8b_gqa"])
def test_noalloc_matches_pa_decode_on_two_calls_in_a_row(name):
    step = wl.make(name)
    ds = DeviceStep(step)
    ds.append()
    ds.decode()
    ref = ds.out.clone()

    out1 = torch.full_like(ds.out, float("nan"))
    _noalloc(ds, out1)
    # The second call gets a different query, so stale scratch contents from
    # the first call would show up as a mismatch.
    ds.q.mul_(-0.5)
    ds.decode()
    ref2 = ds.out.clone()
    out2 = torch.full_like(ds.out, float("nan"))
    _noalloc(ds, out2)
    torch.cuda.synchronize()
    assert int(ds.err.item()) == 0
    # Same kernels, same partitions, same merge order: the outputs are equal
    # bit for bit, not just within the oracle tolerance.
    for got, want in ((out1, ref), (out2, ref2)):
        assert torch.isfinite(got.float()).all()
        assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else
                           got.view(torch.int32),
                           want.view(torch.int16) if want.dtype == torch.bfloat16 else
                           want.view(torch.int32))
    assert not torch.equal(ref, ref2)   # the two calls differ


def test_noalloc_rejects_a_request_larger_than_its_scratch():
    step = wl.make("tiny")
    ds = DeviceStep(step)
    huge = 1 << 24                     # rows: far past the fixed scratch
    need = pa.pa_decode_workspace_size(step.num_seqs, step.num_heads, step.head_dim, huge)
    assert need > pa.NOALLOC_SCRATCH_BYTES
    tables = torch.zeros(step.num_seqs, huge // step.block_size, dtype=torch.int32,
                         device="cuda")
    out = torch.zeros_like(ds.out)
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_decode_noalloc(ds.q, ds.k_cache, ds.v_cache, tables, ds.lens, step.scale, out,
                             huge, error_word=ds.err)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(ds.err.item()) == 0
    assert not out.any()               # nothing was enqueued

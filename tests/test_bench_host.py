"""bench.py's host-side pieces on the CPU: the packed layout of a step's
inputs (one host buffer, one copy per end-to-end step) holds every array
unchanged, 256-byte aligned, and the same layout cut from another buffer
gives the same views; which --kernel choices apply to which workload."""
import numpy as np
import pytest
import torch

import bench
from paged_kv_cache_29_gb300 import workloads as wl


def _host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@pytest.mark.parametrize("name", ["tiny", "8b_gqa_mq2"])
def test_packed_inputs_round_trip(name):
    step = wl.make(name)
    arrays = [step.q, step.k_new, step.v_new, step.slot_mapping, step.block_tables,
              step.context_lens]
    buf, views = bench.packed_buffer(arrays)
    assert buf.dtype == torch.uint8 and buf.numel() >= sum(a.nbytes for a in arrays)
    base = buf.data_ptr()
    for a, v in zip(arrays, views):
        assert (v.data_ptr() - base) % 256 == 0
        assert tuple(v.shape) == a.shape
        np.testing.assert_array_equal(_host(v), a)
    # The same layout over a copy (as the device buffer is cut) reads the same.
    _, again = bench.packed_buffer(arrays, storage=buf.clone())
    for a, v in zip(arrays, again):
        np.testing.assert_array_equal(_host(v), a)


def test_kernel_choices_per_workload():
    """--kernel applies where the workload's decode call takes a kernel
    choice; elsewhere the run stops before touching the GPU."""
    tiny, fp8 = wl.make("tiny"), wl.make("8b_gqa_fp8")
    for k in ("auto", "mma", "simt", "generic"):
        assert bench.kernel_supported(tiny, k)
    assert not bench.kernel_supported(tiny, "tc")
    assert bench.kernel_supported(fp8, "tc") and bench.kernel_supported(fp8, "mma")
    assert not bench.kernel_supported(fp8, "simt")
    for name in ("8b_gqa_int8", "8b_gqa_mq2", "8b_gqa_win1024"):
        step = wl.make(name)
        assert bench.kernel_supported(step, "auto")
        assert not any(bench.kernel_supported(step, k) for k in ("mma", "simt", "generic", "tc"))


def test_kernel_source_hash_follows_code_not_comments(tmp_path):
    """The profile guard's hash changes with the kernel code only."""
    src = tmp_path / "k.cu"
    src.write_text("// header\n__global__ void k(int* a) {\n    a[0] = 1;   /* one */\n}\n")
    h0 = bench.kernel_source_hash(str(tmp_path))
    src.write_text("// another header\n\n__global__ void k(int* a) {\n    a[0] = 1;   // one\n}\n")
    assert bench.kernel_source_hash(str(tmp_path)) == h0
    src.write_text("// header\n__global__ void k(int* a) {\n    a[0] = 2;\n}\n")
    assert bench.kernel_source_hash(str(tmp_path)) != h0

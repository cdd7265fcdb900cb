"""Failure detection on the GPU without a fault: every shared-memory barrier
wait of the tile-ring decode kernels is bounded (about 2 s). A test hook makes
CTA 0's producer announce one tile to its consumer without copying it or
completing its barrier (a flag nothing sets); the consumer's wait gives up,
the kernel flags PA_DEVERR_TIMEOUT and winds down, and the call completes by
itself. The CUDA context stays usable: the next call on the same tensors is
exact. Both issue orders are covered: in stream order (bf16) and per
consumer warp (FP8)."""
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_parity, from_torch, to_torch
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

LENS = [3000, 700, 1500, 40]    # CTA 0's first item is a full partition (32+ tiles)


def _tensors(step, fmt):
    if fmt == "fp8":
        kc = torch.from_numpy(np.ascontiguousarray(step.k_cache)).cuda()
        vc = torch.from_numpy(np.ascontiguousarray(step.v_cache)).cuda()
        q = to_torch(step.q, "bf16")
    else:
        kc, vc, q = to_torch(step.k_cache, fmt), to_torch(step.v_cache, fmt), to_torch(step.q, fmt)
    return q, kc, vc, to_torch(step.block_tables), to_torch(step.context_lens)


@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
def test_withheld_tile_times_out_and_context_stays_usable(fmt):
    step = wl.build_step(f"wait_{fmt}", LENS, 32, 8, 128, cache_dtype=fmt, seed=51)
    assert step.k_scale == 1.0 and step.v_scale == 1.0      # the hook's FP8 scales
    q, kc, vc, bt, cl = _tensors(step, fmt)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, float("nan"))
    torch.cuda.synchronize()
    t0 = time.monotonic()
    pa.pa_test_withhold_tile(q, kc, vc, bt, cl, step.scale, out, step.max_context_len, 5, err)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(err.item()) & pa.PA_DEVERR_TIMEOUT
    assert 1.0 < elapsed < 20.0, elapsed      # waited out its limit, then ended by itself

    # Same context, same tensors: a clean call is exact and flags nothing.
    err.zero_()
    out = torch.full_like(q, float("nan"))
    if fmt == "fp8":
        pa.pa_decode_fp8(q, kc, vc, bt, cl, step.scale, out, step.max_context_len, 1.0, 1.0,
                         error_word=err)
        want = oracle.decode_kv(step.q, step.k_cache, step.v_cache, step.block_tables,
                                step.context_lens, step.scale, 1.0, 1.0)
    else:
        pa.pa_decode(q, kc, vc, bt, cl, step.scale, out, step.max_context_len, error_word=err)
        want = oracle.decode(step.q, step.k_cache, step.v_cache, step.block_tables,
                             step.context_lens, step.scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = wl.as_f32(from_torch(out), "bf16").astype(np.float64)
    assert_parity(got, want, "bf16")


def test_withhold_past_the_stream_changes_nothing():
    """A tile index CTA 0 never reaches: nothing is withheld, the call is exact."""
    step = wl.build_step("wait_none", [40, 17], 8, 2, 128, cache_dtype="bf16", seed=52)
    q, kc, vc, bt, cl = _tensors(step, "bf16")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, float("nan"))
    pa.pa_test_withhold_tile(q, kc, vc, bt, cl, step.scale, out, step.max_context_len, 10_000,
                             err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.decode(step.q, step.k_cache, step.v_cache, step.block_tables,
                         step.context_lens, step.scale)
    assert_parity(wl.as_f32(from_torch(out), "bf16").astype(np.float64), want, "bf16")

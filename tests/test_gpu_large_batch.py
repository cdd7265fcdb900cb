"""Batches above the work list's 4096-sequence limit run as consecutive
launches over slices of the batch that reuse one workspace (the fused calls
also offset the new rows and slots per slice): every sequence of a 4,400-
sequence batch against the oracle, through pa_decode, pa_append_decode
and the FP8 and INT8 fused calls."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceStep, assert_parity, from_torch, oracle_reference, to_torch
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

B = 4400


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _lens(seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 48, size=B)
    lens[::97] = rng.integers(500, 1500, size=len(lens[::97]))   # some span several partitions
    lens[4096 + 7] = 1200                                         # one in the second slice
    return lens.tolist()


def test_large_batch_two_calls_and_fused():
    step = wl.build_step("large", _lens(1), 8, 2, 64, cache_dtype="bf16", seed=41)
    k_ref, v_ref, out_ref = oracle_reference(step)
    two = DeviceStep(step)
    two.append()
    two.decode("auto")
    fused = DeviceStep(step)
    pa.pa_append_decode(fused.k_new, fused.v_new, fused.slots, fused.k_cache, fused.v_cache,
                        fused.q, fused.tables, fused.lens, step.scale, fused.out,
                        step.max_context_len, workspace=fused.workspace, error_word=fused.err)
    torch.cuda.synchronize()
    assert two.error_word() == 0 and fused.error_word() == 0
    for dev in (two, fused):
        np.testing.assert_array_equal(from_torch(dev.k_cache), k_ref)
        np.testing.assert_array_equal(from_torch(dev.v_cache), v_ref)
        assert_parity(dev.result(), out_ref, "bf16")
    np.testing.assert_array_equal(from_torch(fused.out), from_torch(two.out))


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_large_batch_quantised_fused(fmt):
    step = wl.build_step(f"large_{fmt}", _lens(2), 8, 2, 128, cache_dtype=fmt, seed=42)
    k, v = step.k_cache.copy(), step.v_cache.copy()
    kc, vc = _u8(step.k_cache), _u8(step.v_cache)
    q = to_torch(step.q, "bf16")
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (to_torch(step.k_new, "bf16"), to_torch(step.v_new, "bf16"),
            to_torch(step.slot_mapping), kc, vc)
    rest = (q, to_torch(step.block_tables), to_torch(step.context_lens), step.scale, out,
            step.max_context_len)
    if fmt == "fp8":
        pa.pa_append_decode_fp8(*args, *rest, 0.75, 1.5, error_word=err)
        oracle.append_fp8(step.k_new, step.v_new, step.slot_mapping, k, v, 0.75, 1.5)
        want = oracle.decode_kv(step.q, k, v, step.block_tables, step.context_lens, step.scale,
                                0.75, 1.5)
        pairs = [(kc, k), (vc, v)]
    else:
        ks, vs = step.k_row_scales.copy(), step.v_row_scales.copy()
        ksc, vsc = _u8(ks), _u8(vs)
        pa.pa_append_decode_int8(*args, ksc, vsc, *rest, error_word=err)
        oracle.append_int8(step.k_new, step.v_new, step.slot_mapping, k, v, ks, vs)
        want = oracle.decode_int8(step.q, k, v, ks, vs, step.block_tables, step.context_lens,
                                  step.scale)
        pairs = [(kc, k), (vc, v), (ksc, ks), (vsc, vs)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for dev, ref in pairs:
        np.testing.assert_array_equal(dev.cpu().numpy().view(np.uint8),
                                      np.ascontiguousarray(ref).view(np.uint8))
    got = wl.as_f32(from_torch(out), "bf16").astype(np.float64)
    assert_parity(got, want, "bf16")

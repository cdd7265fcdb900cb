"""pa_append_decode on the GPU through the C ABI: the fused decode step (each
sequence's new K/V row written by the decode kernel's CTA that loads it)
against the oracle's append then decode, and bitwise against
pa_reshape_and_cache + pa_decode on the same inputs; slot checks."""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, DeviceStep, from_torch, max_abs, oracle_reference
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

LENS = [1, 15, 16, 17, 31, 100, 511, 512, 513, 1000, 1025, 2047, 4000]


def _poison_new_slots(step):
    """The slots the step appends to hold NaN before the step, so a row the
    kernel fails to write shows in the output."""
    k, v = step.k_cache.copy(), step.v_cache.copy()
    bs = step.block_size
    nan = np.uint16(0x7FC0) if step.cache_dtype == "bf16" else np.float32(np.nan)
    for slot in step.slot_mapping:
        if slot >= 0:
            k[slot // bs, :, slot % bs, :] = nan
            v[slot // bs, :, slot % bs, :] = nan
    return dataclasses.replace(step, k_cache=k, v_cache=v)


def _fused(step):
    dev = DeviceStep(step)
    pa.pa_append_decode(dev.k_new, dev.v_new, dev.slots, dev.k_cache, dev.v_cache, dev.q,
                        dev.tables, dev.lens, step.scale, dev.out, step.max_context_len,
                        workspace=dev.workspace, error_word=dev.err)
    torch.cuda.synchronize()
    return dev


def _two_calls(step):
    dev = DeviceStep(step)
    dev.append()
    dev.decode("auto")
    torch.cuda.synchronize()
    return dev


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [
    ("bf16", 32, 8, 128, 16),     # tensor-core tile ring
    ("bf16", 8, 8, 64, 16),
    ("bf16", 16, 2, 128, 32),
    ("f32", 8, 2, 128, 16),       # SIMT tile ring
    ("bf16", 8, 2, 64, 8),        # no tile ring: append kernel, then the plain kernel
])
def test_fused_step_equals_append_then_decode(dtype, hq, hkv, d, bs):
    step = _poison_new_slots(wl.build_step("fused", LENS, hq, hkv, d, cache_dtype=dtype,
                                           block_size=bs, seed=hq + d + bs))
    k_ref, v_ref, out_ref = oracle_reference(step)
    fused, two = _fused(step), _two_calls(step)
    assert fused.error_word() == 0 and two.error_word() == 0
    np.testing.assert_array_equal(from_torch(fused.k_cache), k_ref)
    np.testing.assert_array_equal(from_torch(fused.v_cache), v_ref)
    np.testing.assert_array_equal(from_torch(fused.out), from_torch(two.out))
    assert max_abs(fused.result(), out_ref) <= TOL[dtype]


def test_negative_slots_append_nothing():
    step = wl.build_step("fneg", LENS, 32, 8, 128, cache_dtype="bf16", seed=5)
    slots = step.slot_mapping.copy()
    slots[[0, 3, 7]] = -1
    step = dataclasses.replace(step, slot_mapping=slots)
    k_ref, v_ref, out_ref = oracle_reference(step)      # the oracle skips negative slots
    fused = _fused(step)
    assert fused.error_word() == 0
    np.testing.assert_array_equal(from_torch(fused.k_cache), k_ref)
    np.testing.assert_array_equal(from_torch(fused.v_cache), v_ref)
    assert max_abs(fused.result(), out_ref) <= TOL["bf16"]


def test_slot_of_another_row_is_flagged_and_not_written():
    lens = [40, 700, 33, 0, 1300]
    step = wl.build_step("fbad", lens, 32, 8, 128, cache_dtype="bf16", seed=6)
    bs = step.block_size
    slots = step.slot_mapping.copy()
    n = lens[1]
    wrong = int(step.block_tables[1][(n - 2) // bs]) * bs + (n - 2) % bs   # row n - 2's slot
    slots[1] = wrong
    slots[3] = 5                                          # an empty sequence with a slot
    bad = dataclasses.replace(step, slot_mapping=slots)
    fused = _fused(bad)
    assert fused.error_word() & pa.PA_DEVERR_SLOT
    k_after = from_torch(fused.k_cache)
    np.testing.assert_array_equal(k_after[wrong // bs, :, wrong % bs, :],
                                  step.k_cache[wrong // bs, :, wrong % bs, :])
    # The other sequences are exact: the oracle on the same inputs, their rows appended.
    ok = dataclasses.replace(step, slot_mapping=np.where(np.isin(np.arange(len(lens)), [1, 3]),
                                                         -1, step.slot_mapping))
    _, _, out_ref = oracle_reference(ok)
    keep = [0, 2, 4]
    assert max_abs(fused.result()[keep], out_ref[keep]) <= TOL["bf16"]

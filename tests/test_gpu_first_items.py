"""First work items of the tile-ring decode kernels (GPU only).

The producer warp finds its CTA's first work item alone (a warp scan of the
full-partition counts over the context lengths, 32 sequences at a time) and
starts loading it while the consumer warps compute the CTA's work list; the
two must agree on every CTA's first item. These cases aim at that scan:
flagged context lengths (negative, past max_context_len, shorter than the
query tokens) and empty sequences before, between and after the sequences
whose full partitions are the launch's first items, over four 32-sequence
chunks, on plain, sliding-window and multi-query decode. Valid sequences must
match the oracle; the flagged ones are reported in the error word.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceStep, assert_parity, from_torch, oracle_reference, to_torch
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

B = 100
FLAGGED = [0, 1, 2, 5, 31, 32, 33, 40, 64, 70, 97, 99]   # set to bad lengths on the device
EMPTY = [3, 34, 65]                                       # empty sequences (zero rows)


def _lens(seed, lo=1):
    lens = [int(x) for x in np.random.default_rng(seed).integers(lo, 2600, size=B)]
    for s in EMPTY:
        lens[s] = 0
    return lens


def _flag(lens_dev, mcl, short=None):
    """Flag the FLAGGED sequences on the device: negative, past mcl, or (with
    several query tokens) shorter than them."""
    for i, s in enumerate(FLAGGED):
        lens_dev[s] = [-3, mcl + 100, short if short is not None else -3][i % 3]


def _keep():
    return [s for s in range(B) if s not in FLAGGED]


@pytest.mark.parametrize("kernel", ["mma", "simt"])
def test_flagged_lengths_around_the_first_items(kernel):
    step = wl.build_step("first", _lens(11), 32, 8, 128, cache_dtype="bf16", seed=11)
    _, _, ref = oracle_reference(step)
    dev = DeviceStep(step)
    dev.append()
    _flag(dev.lens, step.max_context_len)
    dev.decode(kernel)
    torch.cuda.synchronize()
    assert dev.error_word() & pa.PA_DEVERR_CONTEXT
    keep = _keep()
    assert_parity(dev.result()[keep], ref[keep], "bf16", kernel)


def test_flagged_lengths_around_the_first_items_window():
    step = wl.build_step("first_win", _lens(12), 32, 8, 128, cache_dtype="bf16", seed=12)
    window = 700
    k, v = step.k_cache.copy(), step.v_cache.copy()
    oracle.append(step.k_new, step.v_new, step.slot_mapping, k, v)
    ref = oracle.decode_window(step.q, k, v, step.block_tables, step.context_lens, step.scale,
                               window)
    dev = DeviceStep(step)
    dev.append()
    _flag(dev.lens, step.max_context_len)
    out = torch.full_like(dev.q, float("nan"))
    pa.pa_decode_window(dev.q, dev.k_cache, dev.v_cache, dev.tables, dev.lens, step.scale,
                        window, out, step.max_context_len, error_word=dev.err)
    torch.cuda.synchronize()
    assert dev.error_word() & pa.PA_DEVERR_CONTEXT
    got = wl.as_f32(from_torch(out), "bf16").astype(np.float64)
    keep = _keep()
    assert_parity(got[keep], ref[keep], "bf16", "window")


def test_flagged_lengths_around_the_first_items_multi_query():
    step = wl.build_step("first_mq", _lens(13, lo=2), 32, 8, 128, cache_dtype="bf16", seed=13,
                         num_queries=2)
    k, v = step.k_cache.copy(), step.v_cache.copy()
    oracle.append(step.k_new, step.v_new, step.slot_mapping, k, v)
    ref = oracle.decode_multi(step.q, k, v, step.block_tables, step.context_lens, step.scale)
    q = to_torch(step.q, "bf16")
    kc, vc = to_torch(step.k_cache, "bf16"), to_torch(step.v_cache, "bf16")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(to_torch(step.k_new, "bf16"), to_torch(step.v_new, "bf16"),
                            to_torch(step.slot_mapping), kc, vc, error_word=err)
    lens = to_torch(step.context_lens)
    _flag(lens, step.max_context_len, short=1)        # 1 row < 2 query tokens
    out = torch.full_like(q, float("nan"))
    pa.pa_decode_multi(q, kc, vc, to_torch(step.block_tables), lens, step.scale, out,
                       step.max_context_len, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_CONTEXT
    got = wl.as_f32(from_torch(out), "bf16").astype(np.float64)
    keep = _keep()
    assert_parity(got[keep], ref[keep], "bf16", "multi-query")

"""Sliding-window decode on the GPU against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_parity, from_torch, to_torch
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _gpu(step, window, append=True, mcl=None, plain=False):
    cd = step.cache_dtype
    q = to_torch(step.q, cd)
    k, v = to_torch(step.k_cache, cd), to_torch(step.v_cache, cd)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if append:
        pa.pa_reshape_and_cache(to_torch(step.k_new, cd), to_torch(step.v_new, cd),
                                to_torch(step.slot_mapping), k, v, error_word=err)
    out = torch.full_like(q, float("nan"))
    args = (q, k, v, to_torch(step.block_tables), to_torch(step.context_lens), step.scale)
    m = step.max_context_len if mcl is None else mcl
    if plain:
        pa.pa_decode(*args, out, m, error_word=err)
    else:
        pa.pa_decode_window(*args, window, out, m, error_word=err)
    torch.cuda.synchronize()
    return wl.as_f32(from_torch(out), cd).astype(np.float64), int(err.item())


def _oracle(step, window, append=True):
    k, v = step.k_cache.copy(), step.v_cache.copy()
    if append:
        oracle.append(step.k_new, step.v_new, step.slot_mapping, k, v)
    return oracle.decode_window(step.q, k, v, step.block_tables, step.context_lens, step.scale,
                                window)


def test_window_workload():
    step = wl.make("8b_gqa_win1024")
    got, err = _gpu(step, step.window)
    assert err == 0
    assert_parity(got, _oracle(step, step.window), "bf16")


LENS = [1, 15, 16, 17, 100, 511, 512, 513, 1000, 1025, 2049, 5000]


@pytest.mark.parametrize("dtype,hq,hkv,d", [("bf16", 32, 8, 128), ("bf16", 8, 8, 64),
                                            ("f32", 16, 8, 128), ("f32", 8, 4, 64)])
@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 512, 513, 1000])
def test_window_ragged(dtype, hq, hkv, d, window):
    step = wl.build_step("win", LENS, hq, hkv, d, cache_dtype=dtype, seed=window + hq)
    got, err = _gpu(step, window)
    assert err == 0
    assert_parity(got, _oracle(step, window), dtype)


def test_window_past_every_sequence_equals_pa_decode_bitwise():
    step = wl.build_step("winall", LENS, 32, 8, 128, seed=5)
    got_w, _ = _gpu(step, 5000)
    got_p, _ = _gpu(step, 0, plain=True)
    np.testing.assert_array_equal(got_w, got_p)


def test_window_batch_invariance():
    big = wl.build_step("winb", [3000, 40, 700, 1100, 9], 32, 8, 128, seed=12)
    got_big, _ = _gpu(big, 600, append=False)
    for s in range(big.num_seqs):
        one = wl.DecodeStep(name="one", cache_dtype="bf16", num_heads=32, num_kv_heads=8,
                            head_dim=128, block_size=16, q=big.q[s:s + 1],
                            k_new=big.k_new[s:s + 1], v_new=big.v_new[s:s + 1],
                            slot_mapping=big.slot_mapping[s:s + 1], k_cache=big.k_cache,
                            v_cache=big.v_cache, block_tables=big.block_tables[s:s + 1],
                            context_lens=big.context_lens[s:s + 1], scale=big.scale, seed=0)
        got_one, _ = _gpu(one, 600, append=False, mcl=big.max_context_len)
        np.testing.assert_array_equal(got_one[0], got_big[s])


def test_window_bad_arguments():
    step = wl.build_step("winx", [40, 50], 32, 8, 128, seed=1)
    for w in (0, -3):
        with pytest.raises(pa.PagedAttentionError) as e:
            _gpu(step, w)
        assert e.value.status == pa.PA_ERR_INVALID_ARG
    step = wl.build_step("winx", [40, 50], 32, 8, 128, block_size=8, seed=1)   # no tile ring
    with pytest.raises(pa.PagedAttentionError) as e:
        _gpu(step, 16)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED

"""Multi-query decode (several new tokens per sequence, causal within them)
on the GPU against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_parity, from_torch, to_torch
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _q4(step):
    return step.q if step.q.ndim == 4 else step.q[:, None]       # [B][Q][Hq][D]


def _gpu(step, append=True, mcl=None):
    cd = step.cache_dtype
    q = to_torch(np.ascontiguousarray(_q4(step)), cd)
    k, v = to_torch(step.k_cache, cd), to_torch(step.v_cache, cd)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if append:
        pa.pa_reshape_and_cache(to_torch(step.k_new, cd), to_torch(step.v_new, cd),
                                to_torch(step.slot_mapping), k, v, error_word=err)
    out = torch.full_like(q, float("nan"))
    pa.pa_decode_multi(q, k, v, to_torch(step.block_tables), to_torch(step.context_lens),
                       step.scale, out, step.max_context_len if mcl is None else mcl,
                       error_word=err)
    torch.cuda.synchronize()
    return wl.as_f32(from_torch(out), cd).astype(np.float64), int(err.item())


def _oracle(step, append=True):
    k, v = step.k_cache.copy(), step.v_cache.copy()
    if append:
        oracle.append(step.k_new, step.v_new, step.slot_mapping, k, v)
    return oracle.decode_multi(_q4(step), k, v, step.block_tables, step.context_lens, step.scale)


def test_multi_query_workload():
    step = wl.make("8b_gqa_mq2")
    got, err = _gpu(step)
    assert err == 0
    assert_parity(got, _oracle(step), "bf16")


@pytest.mark.parametrize("hq,hkv,Q,d", [(8, 8, 2, 128), (8, 8, 3, 64), (16, 8, 3, 128),
                                        (32, 8, 2, 128), (16, 8, 4, 64), (8, 8, 8, 128),
                                        (64, 8, 1, 128)])
def test_multi_query_ragged(hq, hkv, Q, d):
    lens = [Q, Q + 1, 17, 511, 512, 512 + 1, 512 + Q - 1, 1030, 2048 + Q - 2, 3001]
    step = wl.build_step("mq", lens, hq, hkv, d, seed=hq * 10 + Q, num_queries=Q)
    got, err = _gpu(step)
    assert err == 0
    assert_parity(got, _oracle(step), "bf16")


def test_single_query_matches_pa_decode_bitwise():
    step = wl.build_step("mq1", [5, 600, 1500], 32, 8, 128, seed=4, num_queries=1)
    cd = step.cache_dtype
    q3 = to_torch(step.q, cd)
    k, v = to_torch(step.k_cache, cd), to_torch(step.v_cache, cd)
    tables, lens = to_torch(step.block_tables), to_torch(step.context_lens)
    out3 = torch.empty_like(q3)
    pa.pa_decode(q3, k, v, tables, lens, step.scale, out3, step.max_context_len)
    out4 = torch.empty_like(q3).unsqueeze(1)
    pa.pa_decode_multi(q3.unsqueeze(1).contiguous(), k, v, tables, lens, step.scale, out4,
                       step.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out3, out4[:, 0])


def test_multi_query_batch_invariance():
    big = wl.build_step("mqb", [700, 40, 2600, 3, 515], 32, 8, 128, seed=8, num_queries=2)
    got_big, _ = _gpu(big, append=False)
    for s in range(big.num_seqs):
        one = wl.DecodeStep(name="one", cache_dtype="bf16", num_heads=32, num_kv_heads=8,
                            head_dim=128, block_size=16, q=big.q[s:s + 1],
                            k_new=big.k_new[2 * s:2 * s + 2], v_new=big.v_new[2 * s:2 * s + 2],
                            slot_mapping=big.slot_mapping[2 * s:2 * s + 2],
                            k_cache=big.k_cache, v_cache=big.v_cache,
                            block_tables=big.block_tables[s:s + 1],
                            context_lens=big.context_lens[s:s + 1], scale=big.scale, seed=0,
                            num_queries=2)
        got_one, _ = _gpu(one, append=False, mcl=big.max_context_len)
        np.testing.assert_array_equal(got_one[0], got_big[s])


def test_multi_query_empty_and_short_sequences():
    step = wl.build_step("mqe", [0, 9, 0, 40], 16, 8, 128, seed=2, num_queries=2)
    got, err = _gpu(step)
    assert err == 0
    assert not got[0].any() and not got[2].any()
    want = _oracle(step)
    assert_parity(got[[1, 3]], want[[1, 3]], "bf16")
    # a sequence shorter than its query tokens is flagged
    step.context_lens[1] = 1
    _, err = _gpu(step, append=False)
    assert err & pa.PA_DEVERR_CONTEXT


def test_multi_query_unsupported():
    step = wl.build_step("mqu", [40, 50], 32, 8, 128, seed=1, num_queries=3)   # 4 x 3 > 8 columns
    with pytest.raises(pa.PagedAttentionError) as e:
        _gpu(step)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    step = wl.build_step("mqu", [40, 50], 8, 8, 64, cache_dtype="f32", seed=1, num_queries=2)
    with pytest.raises(pa.PagedAttentionError) as e:
        _gpu(step)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED

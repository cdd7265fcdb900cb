"""Seeded random shapes against the oracle: dtype, head grouping, head_dim,
block size, partition size and ragged lengths (with empty sequences) drawn
per case, through the two-call step and the fused step (and the FP8 and INT8
calls), so that combinations no hand-written case names are exercised too.
Every case is reproducible from its index."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceStep, assert_parity, from_torch, oracle_reference, to_torch
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

GROUPS = [(8, 2), (4, 4), (16, 2), (6, 3), (32, 4), (8, 1)]


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    dtype = ["f32", "bf16"][i % 2]
    hq, hkv = GROUPS[rng.integers(len(GROUPS))]
    d = int(rng.choice([64, 128, 96, 32]))
    bs = int(rng.choice([16, 32, 8, 64]))
    part = int(rng.choice([0, 16, 64, 512]))
    B = int(rng.integers(1, 9))
    lens = rng.integers(0, 2500, size=B)
    lens[rng.random(B) < 0.2] = 0
    lens[rng.random(B) < 0.2] = rng.integers(1, 20)
    return dtype, hq, hkv, d, bs, part, [int(x) for x in lens], int(rng.integers(1 << 30))


@pytest.mark.parametrize("i", range(28))
def test_random_shape(i):
    dtype, hq, hkv, d, bs, part, lens, seed = _draw(i)
    step = wl.build_step(f"rand{i}", lens, hq, hkv, d, cache_dtype=dtype, block_size=bs,
                         seed=seed)
    k_ref, v_ref, ref = oracle_reference(step)
    dev = DeviceStep(step, partition_size=part)
    out = dev.run("auto")
    assert dev.error_word() == 0, (i, dtype, hq, hkv, d, bs, part, lens)
    np.testing.assert_array_equal(from_torch(dev.k_cache), k_ref)
    assert_parity(out, ref, dtype, (i, dtype, hq, hkv, d, bs, part, lens))
    if part == 0:
        fused = DeviceStep(step)
        pa.pa_append_decode(fused.k_new, fused.v_new, fused.slots, fused.k_cache, fused.v_cache,
                            fused.q, fused.tables, fused.lens, step.scale, fused.out,
                            step.max_context_len, workspace=fused.workspace,
                            error_word=fused.err)
        torch.cuda.synchronize()
        assert fused.error_word() == 0
        np.testing.assert_array_equal(from_torch(fused.k_cache), k_ref)
        assert_parity(fused.result(), ref, dtype)


@pytest.mark.parametrize("i", range(12))
def test_random_shape_8bit(i):
    rng = np.random.default_rng(2000 + i)
    fmt = ["fp8", "int8"][i % 2]
    g = int(rng.choice([1, 2, 4, 8]))
    hkv = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32]))
    B = int(rng.integers(1, 9))
    lens = rng.integers(0, 5000, size=B)
    lens[rng.random(B) < 0.2] = 0
    lens = [int(x) for x in lens]
    step = wl.build_step(f"rand8_{i}", lens, g * hkv, hkv, 128, cache_dtype=fmt, block_size=bs,
                         seed=int(rng.integers(1 << 30)))
    k, v = step.k_cache.copy(), step.v_cache.copy()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kc, vc = dev(k), dev(v)
    q = to_torch(step.q, "bf16")
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (to_torch(step.k_new, "bf16"), to_torch(step.v_new, "bf16"),
            to_torch(step.slot_mapping), kc, vc)
    rest = (q, to_torch(step.block_tables), to_torch(step.context_lens), step.scale, out,
            step.max_context_len)
    if fmt == "fp8":
        pa.pa_append_decode_fp8(*args, *rest, 1.0, 1.0, error_word=err)
        oracle.append_fp8(step.k_new, step.v_new, step.slot_mapping, k, v, 1.0, 1.0)
        want = oracle.decode_kv(step.q, k, v, step.block_tables, step.context_lens, step.scale,
                                1.0, 1.0)
        pairs = [(kc, k), (vc, v)]
    else:
        ks, vs = step.k_row_scales.copy(), step.v_row_scales.copy()
        ksc, vsc = dev(ks), dev(vs)
        pa.pa_append_decode_int8(*args, ksc, vsc, *rest, error_word=err)
        oracle.append_int8(step.k_new, step.v_new, step.slot_mapping, k, v, ks, vs)
        want = oracle.decode_int8(step.q, k, v, ks, vs, step.block_tables, step.context_lens,
                                  step.scale)
        pairs = [(kc, k), (vc, v), (ksc, ks), (vsc, vs)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0, (i, fmt, g, hkv, bs, lens)
    for got, ref in pairs:
        np.testing.assert_array_equal(got.cpu().numpy().view(np.uint8),
                                      np.ascontiguousarray(ref).view(np.uint8))
    got = wl.as_f32(from_torch(out), "bf16").astype(np.float64)
    assert_parity(got, want, "bf16", (i, fmt, g, hkv, bs, lens))


@pytest.mark.parametrize("i", range(10))
def test_random_window(i):
    import test_gpu_window as tw
    rng = np.random.default_rng(3000 + i)
    dtype = ["f32", "bf16"][i % 2]
    hkv = int(rng.choice([1, 2, 4, 8]))
    hq = hkv * int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32]))
    lens = rng.integers(0, 4000, size=int(rng.integers(1, 9)))
    lens[rng.random(len(lens)) < 0.2] = 0
    window = int(rng.integers(1, 3000))
    step = wl.build_step(f"rwin{i}", [int(x) for x in lens], hq, hkv, d, cache_dtype=dtype,
                         block_size=bs, seed=int(rng.integers(1 << 30)))
    got, err = tw._gpu(step, window)
    assert err == 0, (i, dtype, hq, hkv, d, bs, window, list(lens))
    assert_parity(got, tw._oracle(step, window), dtype, (i, window))


@pytest.mark.parametrize("i", range(10))
def test_random_multi_query(i):
    import test_gpu_multi as tm
    rng = np.random.default_rng(4000 + i)
    Q = int(rng.choice([1, 2, 3, 4, 8]))
    g = int(rng.choice([g for g in (1, 2, 4, 8) if g * Q <= 8]))
    hkv = int(rng.choice([1, 2, 8]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32]))
    lens = rng.integers(Q, 4000, size=int(rng.integers(1, 9)))
    lens[rng.random(len(lens)) < 0.2] = 0
    step = wl.build_step(f"rmq{i}", [int(x) for x in lens], g * hkv, hkv, d, block_size=bs,
                         seed=int(rng.integers(1 << 30)), num_queries=Q)
    got, err = tm._gpu(step)
    assert err == 0, (i, Q, g, hkv, d, bs, list(lens))
    assert_parity(got, tm._oracle(step), "bf16", (i, Q, g))

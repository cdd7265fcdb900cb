"""pa_append_decode on the GPU through the C ABI: the fused decode step (each
sequence's new K/V row written by the decode kernel's CTA that loads it)
against the oracle's append then decode, and bitwise against
pa_reshape_and_cache + pa_decode on the same inputs; slot checks."""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import DeviceStep, assert_parity, from_torch, oracle_reference
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
    assert_parity(fused.result(), out_ref, dtype)


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
    assert_parity(fused.result(), out_ref, "bf16")


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
    assert_parity(fused.result()[keep], out_ref[keep], "bf16")


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _quant_step_tensors(step):
    from gpu_helpers import to_torch
    t = dict(q=to_torch(step.q, "bf16"), k_new=to_torch(step.k_new, "bf16"),
             v_new=to_torch(step.v_new, "bf16"), slots=to_torch(step.slot_mapping),
             tables=to_torch(step.block_tables), lens=to_torch(step.context_lens),
             k=_u8(step.k_cache), v=_u8(step.v_cache),
             err=torch.zeros(1, dtype=torch.int32, device="cuda"))
    t["out"] = torch.full_like(t["q"], float("nan"))
    if step.cache_dtype == "int8":
        t["ks"], t["vs"] = _u8(step.k_row_scales), _u8(step.v_row_scales)
    return t


def _poison_quant(step):
    """NaN codes (FP8) or NaN scales (INT8) in the slots the step appends to."""
    bs = step.block_size
    k, v = step.k_cache.copy(), step.v_cache.copy()
    extra = {}
    if step.cache_dtype == "int8":
        ks, vs = step.k_row_scales.copy(), step.v_row_scales.copy()
    for slot in step.slot_mapping:
        if slot >= 0:
            if step.cache_dtype == "fp8":
                k[slot // bs, :, slot % bs, :] = 0x7F
                v[slot // bs, :, slot % bs, :] = 0xFF
            else:
                ks[slot // bs, :, slot % bs] = np.nan
                vs[slot // bs, :, slot % bs] = np.nan
    if step.cache_dtype == "int8":
        extra = dict(k_row_scales=ks, v_row_scales=vs)
    return dataclasses.replace(step, k_cache=k, v_cache=v, **extra)


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 2)])
def test_quantised_fused_step_equals_append_then_decode(fmt, hq, hkv):
    _check_quantised_fused(fmt, _poison_quant(wl.build_step(f"q{fmt}", LENS, hq, hkv, 128,
                                                            cache_dtype=fmt, seed=hq + hkv)))


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
@pytest.mark.parametrize("bs", [32, 64])
def test_quantised_fused_step_larger_blocks(fmt, bs):
    """The new row lands in a block of several tiles (and INT8 scale rows)."""
    _check_quantised_fused(fmt, _poison_quant(wl.build_step(f"q{fmt}{bs}", LENS, 32, 8, 128,
                                                            cache_dtype=fmt, block_size=bs,
                                                            seed=bs)))


def _check_quantised_fused(fmt, step):
    import oracle
    ksc, vsc = (0.75, 1.5) if fmt == "fp8" else (1.0, 1.0)
    fused, two = _quant_step_tensors(step), _quant_step_tensors(step)
    if fmt == "fp8":
        pa.pa_append_decode_fp8(fused["k_new"], fused["v_new"], fused["slots"], fused["k"],
                                fused["v"], fused["q"], fused["tables"], fused["lens"],
                                step.scale, fused["out"], step.max_context_len, ksc, vsc,
                                error_word=fused["err"])
        pa.pa_reshape_and_cache_fp8(two["k_new"], two["v_new"], two["slots"], two["k"], two["v"],
                                    ksc, vsc, error_word=two["err"])
        pa.pa_decode_fp8(two["q"], two["k"], two["v"], two["tables"], two["lens"], step.scale,
                         two["out"], step.max_context_len, ksc, vsc, error_word=two["err"])
        k, v = step.k_cache.copy(), step.v_cache.copy()
        oracle.append_fp8(step.k_new, step.v_new, step.slot_mapping, k, v, ksc, vsc)
        want = oracle.decode_kv(step.q, k, v, step.block_tables, step.context_lens, step.scale,
                                ksc, vsc)
        refs = [("k", k), ("v", v)]
    else:
        pa.pa_append_decode_int8(fused["k_new"], fused["v_new"], fused["slots"], fused["k"],
                                 fused["v"], fused["ks"], fused["vs"], fused["q"],
                                 fused["tables"], fused["lens"], step.scale, fused["out"],
                                 step.max_context_len, error_word=fused["err"])
        pa.pa_reshape_and_cache_int8(two["k_new"], two["v_new"], two["slots"], two["k"], two["v"],
                                     two["ks"], two["vs"], error_word=two["err"])
        pa.pa_decode_int8(two["q"], two["k"], two["v"], two["ks"], two["vs"], two["tables"],
                          two["lens"], step.scale, two["out"], step.max_context_len,
                          error_word=two["err"])
        k, v = step.k_cache.copy(), step.v_cache.copy()
        ks, vs = step.k_row_scales.copy(), step.v_row_scales.copy()
        oracle.append_int8(step.k_new, step.v_new, step.slot_mapping, k, v, ks, vs)
        want = oracle.decode_int8(step.q, k, v, ks, vs, step.block_tables, step.context_lens,
                                  step.scale)
        refs = [("k", k), ("v", v), ("ks", ks), ("vs", vs)]
    torch.cuda.synchronize()
    assert int(fused["err"].item()) == 0 and int(two["err"].item()) == 0
    for name, ref in refs:
        got = fused[name].cpu().numpy()
        np.testing.assert_array_equal(got.view(np.uint8), two[name].cpu().numpy().view(np.uint8))
        np.testing.assert_array_equal(got.view(np.uint8), np.ascontiguousarray(ref).view(np.uint8))
    np.testing.assert_array_equal(from_torch(fused["out"]), from_torch(two["out"]))
    got = wl.as_f32(from_torch(fused["out"]), "bf16").astype(np.float64)
    assert_parity(got, want, "bf16")


@pytest.mark.parametrize("name", ["8b_gqa", "7b_mha", "long_skew", "prefix_shared"])
def test_fused_step_on_full_workloads(name):
    """The benchmarked workloads at full size: the pools after the fused step
    equal the oracle's append bit for bit, the output is within tolerance of
    the oracle and bitwise equal to the two-call step."""
    step = wl.make(name)
    k_ref, v_ref, out_ref = oracle_reference(step)
    fused, two = _fused(step), _two_calls(step)
    assert fused.error_word() == 0
    np.testing.assert_array_equal(from_torch(fused.k_cache), k_ref)
    np.testing.assert_array_equal(from_torch(fused.v_cache), v_ref)
    np.testing.assert_array_equal(from_torch(fused.out), from_torch(two.out))
    assert_parity(fused.result(), out_ref, step.cache_dtype)


def test_fused_steps_in_a_row_follow_the_oracle():
    """Four decode steps in a row through pa_append_decode: every step appends
    one row per sequence (crossing block boundaries) and attends to all."""
    import oracle
    from paged_kv_cache_29_gb300.block_manager import BlockManager
    rng = np.random.default_rng(11)
    hq, hkv, d, bs, nb = 32, 8, 128, 16, 160
    lens0 = [14, 15, 16, 511, 1023]
    mgr = BlockManager(nb, bs, free_order=rng.permutation(nb), prefix_caching=False)
    for s, n in enumerate(lens0):
        mgr.admit(f"s{s}", [0] * n)
    k = wl.to_cache_dtype(rng.standard_normal((nb, hkv, bs, d), dtype=np.float32), "bf16")
    v = wl.to_cache_dtype(rng.standard_normal((nb, hkv, bs, d), dtype=np.float32), "bf16")
    kd = torch.from_numpy(k.copy()).view(torch.bfloat16).cuda()
    vd = torch.from_numpy(v.copy()).view(torch.bfloat16).cuda()
    B = len(lens0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(4):
        slots = np.array([mgr.append(f"s{s}", 0).slot for s in range(B)], np.int64)
        lens = np.array([mgr.num_tokens(f"s{s}") for s in range(B)], np.int32)
        bt = np.full((B, 72), -1, np.int32)
        for s in range(B):
            t = mgr.block_table(f"s{s}")
            bt[s, :len(t)] = t
        q = wl.to_cache_dtype(rng.standard_normal((B, hq, d), dtype=np.float32), "bf16")
        kn = wl.to_cache_dtype(rng.standard_normal((B, hkv, d), dtype=np.float32), "bf16")
        vn = wl.to_cache_dtype(rng.standard_normal((B, hkv, d), dtype=np.float32), "bf16")
        oracle.append(kn, vn, slots, k, v)
        ref = oracle.decode(q, k, v, bt, lens, 1 / np.sqrt(d))
        dq = torch.from_numpy(q).view(torch.bfloat16).cuda()
        out = torch.empty_like(dq)
        pa.pa_append_decode(torch.from_numpy(kn).view(torch.bfloat16).cuda(),
                            torch.from_numpy(vn).view(torch.bfloat16).cuda(),
                            torch.from_numpy(slots).cuda(), kd, vd, dq,
                            torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda(),
                            1 / np.sqrt(d), out, int(lens.max()), error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = wl.as_f32(from_torch(out), "bf16").astype(np.float64)
        assert_parity(got, ref, "bf16")
        assert np.array_equal(from_torch(kd), k) and np.array_equal(from_torch(vd), v)


@pytest.mark.parametrize("name", ["8b_gqa_fp8", "8b_gqa_int8"])
def test_quantised_fused_step_on_full_workloads(name):
    """The benchmarked 8-bit workloads at full size: codes (and row scales)
    after the fused step equal the two-call step's bit for bit, and so does
    the output."""
    step = wl.make(name)
    fused, two = _quant_step_tensors(step), _quant_step_tensors(step)
    if step.cache_dtype == "fp8":
        pa.pa_append_decode_fp8(fused["k_new"], fused["v_new"], fused["slots"], fused["k"],
                                fused["v"], fused["q"], fused["tables"], fused["lens"],
                                step.scale, fused["out"], step.max_context_len, step.k_scale,
                                step.v_scale, error_word=fused["err"])
        pa.pa_reshape_and_cache_fp8(two["k_new"], two["v_new"], two["slots"], two["k"], two["v"],
                                    step.k_scale, step.v_scale, error_word=two["err"])
        pa.pa_decode_fp8(two["q"], two["k"], two["v"], two["tables"], two["lens"], step.scale,
                         two["out"], step.max_context_len, step.k_scale, step.v_scale,
                         error_word=two["err"])
        names = ["k", "v"]
    else:
        pa.pa_append_decode_int8(fused["k_new"], fused["v_new"], fused["slots"], fused["k"],
                                 fused["v"], fused["ks"], fused["vs"], fused["q"],
                                 fused["tables"], fused["lens"], step.scale, fused["out"],
                                 step.max_context_len, error_word=fused["err"])
        pa.pa_reshape_and_cache_int8(two["k_new"], two["v_new"], two["slots"], two["k"], two["v"],
                                     two["ks"], two["vs"], error_word=two["err"])
        pa.pa_decode_int8(two["q"], two["k"], two["v"], two["ks"], two["vs"], two["tables"],
                          two["lens"], step.scale, two["out"], step.max_context_len,
                          error_word=two["err"])
        names = ["k", "v", "ks", "vs"]
    torch.cuda.synchronize()
    assert int(fused["err"].item()) == 0 and int(two["err"].item()) == 0
    for n in names:
        assert torch.equal(fused[n].view(torch.uint8), two[n].view(torch.uint8)), n
    np.testing.assert_array_equal(from_torch(fused["out"]), from_torch(two["out"]))

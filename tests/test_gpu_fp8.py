"""FP8 (e4m3) KV cache on the GPU against the oracle, through the C ABI:
the quantising append is bit-exact (codes), decode attention over the codes
with per-tensor scales is within the bf16 output tolerance of the fp64
oracle on the same codes."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, assert_parity, from_torch, max_abs, to_torch
from parity import assert_scaled
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def _dev(step):
    return dict(q=to_torch(step.q, "bf16"), k_new=to_torch(step.k_new, "bf16"),
                v_new=to_torch(step.v_new, "bf16"), k=_u8(step.k_cache), v=_u8(step.v_cache),
                slots=to_torch(step.slot_mapping), tables=to_torch(step.block_tables),
                lens=to_torch(step.context_lens),
                err=torch.zeros(1, dtype=torch.int32, device="cuda"))


def _gpu_step(step, k_scale=1.0, v_scale=1.0, append=True, mcl=None, kernel="auto"):
    d = _dev(step)
    if append:
        pa.pa_reshape_and_cache_fp8(d["k_new"], d["v_new"], d["slots"], d["k"], d["v"],
                                    k_scale, v_scale, error_word=d["err"])
    out = torch.full_like(d["q"], float("nan"))
    pa.pa_decode_fp8(d["q"], d["k"], d["v"], d["tables"], d["lens"], step.scale, out,
                     step.max_context_len if mcl is None else mcl, k_scale, v_scale,
                     error_word=d["err"], kernel=kernel)
    torch.cuda.synchronize()
    return d, wl.as_f32(from_torch(out), "bf16").astype(np.float64)


def _oracle_step(step, k_scale=1.0, v_scale=1.0, append=True):
    k, v = step.k_cache.copy(), step.v_cache.copy()
    if append:
        oracle.append_fp8(step.k_new, step.v_new, step.slot_mapping, k, v, k_scale, v_scale)
    out = oracle.decode_kv(step.q, k, v, step.block_tables, step.context_lens, step.scale,
                           k_scale, v_scale)
    return k, v, out


# Both FP8 kernels: the tile ring with mma.sync on widened codes, and the
# tcgen05 kernel (e4m3 products on 128-row chunks, tensor-memory accumulators).
FP8_KERNELS = ["mma", "tc"]


@pytest.mark.parametrize("kernel", FP8_KERNELS)
@pytest.mark.parametrize("lens,g", [([1, 2, 15, 16, 17, 100, 127, 128, 129, 300], 8),
                                    ([5, 128, 1023, 1024, 1025, 3000], 4),
                                    ([40, 257, 700], 2), ([33, 1200], 1)])
def test_fp8_small_shapes(kernel, lens, g):
    step = wl.build_step("fp8s", lens, 8 * g, 8, 128, cache_dtype="fp8", seed=len(lens) + g)
    d, got = _gpu_step(step, kernel=kernel)
    _, _, want = _oracle_step(step)
    assert int(d["err"].item()) == 0
    assert np.isfinite(got).all()
    assert_parity(got, want, "bf16", (kernel, lens, g))


@pytest.mark.parametrize("kernel", FP8_KERNELS)
def test_fp8_workload_append_and_decode(kernel):
    step = wl.make("8b_gqa_fp8")
    d, got = _gpu_step(step, kernel=kernel)
    k, v, want = _oracle_step(step)
    assert int(d["err"].item()) == 0
    np.testing.assert_array_equal(d["k"].cpu().numpy(), k)
    np.testing.assert_array_equal(d["v"].cpu().numpy(), v)
    assert_parity(got, want, "bf16", "8b_gqa_fp8")


@pytest.mark.parametrize("new_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.37, 3.0), (0.01, 0.02)])
def test_fp8_append_codes_bit_exact(new_dtype, k_scale, v_scale):
    rng = np.random.default_rng(int(k_scale * 1000) + (new_dtype == "f32"))
    nb, hkv, bs, d, T = 40, 4, 16, 128, 97
    kn = wl.to_cache_dtype(rng.standard_normal((T, hkv, d)).astype(np.float32) *
                           10.0 ** rng.uniform(-3, 3, (T, hkv, 1)).astype(np.float32), new_dtype)
    vn = wl.to_cache_dtype(rng.standard_normal((T, hkv, d)).astype(np.float32) * 5, new_dtype)
    kc = rng.integers(0, 256, (nb, hkv, bs, d)).astype(np.uint8)
    vc = rng.integers(0, 256, (nb, hkv, bs, d)).astype(np.uint8)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[3] = -1
    slots[7] = nb * bs + 5                      # past the pool: flagged, skipped
    kd, vd = _u8(kc), _u8(vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache_fp8(to_torch(kn, new_dtype), to_torch(vn, new_dtype),
                                to_torch(slots), kd, vd, k_scale, v_scale, error_word=err)
    torch.cuda.synchronize()
    assert oracle.append_fp8(kn, vn, slots, kc, vc, k_scale, v_scale) == 1
    assert int(err.item()) == pa.PA_DEVERR_SLOT
    np.testing.assert_array_equal(kd.cpu().numpy(), kc)
    np.testing.assert_array_equal(vd.cpu().numpy(), vc)


@pytest.mark.parametrize("kernel", FP8_KERNELS)
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8)])
@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.5, 3.0), (0.01, 0.02)])
def test_fp8_ragged_groups_and_scales(kernel, hq, hkv, k_scale, v_scale):
    lens = [1, 15, 16, 17, 100, 511, 512, 513, 1500, 3000]
    step = wl.build_step("fp8r", lens, hq, hkv, 128, cache_dtype="fp8", seed=hq + hkv)
    _, got = _gpu_step(step, k_scale, v_scale, kernel=kernel)
    _, _, want = _oracle_step(step, k_scale, v_scale)
    # The output is v_scale times an attention over e4m3 values: the absolute
    # bar, stated for outputs of unit-size values, grows with v_scale above 1
    # (bf16 rounding of a 3x larger output is 3x larger); the output-scaled
    # bound needs no such change.
    err = max_abs(got, want)
    assert err <= TOL["bf16"] * max(1.0, v_scale), err
    assert_scaled(got, want, "bf16", f"fp8 {hq}/{hkv} scales {k_scale}, {v_scale}")


@pytest.mark.parametrize("kernel", FP8_KERNELS)
def test_fp8_nan_codes_past_the_end_do_not_leak(kernel):
    lens = [3, 17, 40, 600]
    step = wl.build_step("fp8nan", lens, 32, 8, 128, cache_dtype="fp8", seed=9)
    bs = step.block_size
    for s, n in enumerate(lens):                 # poison every row past each sequence's end
        t = step.block_tables[s]
        for i in range(n, -(-n // bs) * bs):
            step.k_cache[t[i // bs], :, i % bs, :] = 0x7F
            step.v_cache[t[i // bs], :, i % bs, :] = 0xFF
    _, got = _gpu_step(step, append=False, kernel=kernel)
    _, _, want = _oracle_step(step, append=False)
    assert np.isfinite(got).all()
    assert_parity(got, want, "bf16")


@pytest.mark.parametrize("kernel", FP8_KERNELS)
def test_fp8_batch_invariance(kernel):
    lens = [700, 33, 4000, 1, 515]
    big = wl.build_step("fp8b", lens, 32, 8, 128, cache_dtype="fp8", seed=3)
    _, got_big = _gpu_step(big, append=False, kernel=kernel)
    for s in (0, 2, 4):
        one = wl.DecodeStep(name="one", cache_dtype="fp8", num_heads=32, num_kv_heads=8,
                            head_dim=128, block_size=16, q=big.q[s:s + 1],
                            k_new=big.k_new[s:s + 1], v_new=big.v_new[s:s + 1],
                            slot_mapping=big.slot_mapping[s:s + 1], k_cache=big.k_cache,
                            v_cache=big.v_cache, block_tables=big.block_tables[s:s + 1],
                            context_lens=big.context_lens[s:s + 1], scale=big.scale,
                            seed=0, act_dtype="bf16")
        _, got_one = _gpu_step(one, append=False, mcl=big.max_context_len, kernel=kernel)
        np.testing.assert_array_equal(got_one[0], got_big[s])


def test_fp8_unsupported_and_bad_arguments():
    step = wl.build_step("fp8u", [20, 40], 32, 8, 64, cache_dtype="fp8", seed=1)
    with pytest.raises(pa.PagedAttentionError) as e:
        _gpu_step(step, append=False)                         # head_dim 64
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    step = wl.build_step("fp8u", [20, 40], 24, 8, 128, cache_dtype="fp8", seed=1)
    with pytest.raises(pa.PagedAttentionError) as e:
        _gpu_step(step, append=False)                         # 3 query heads per KV head
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    step = wl.build_step("fp8u", [20, 40], 32, 8, 128, cache_dtype="fp8", seed=1)
    for ks in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(pa.PagedAttentionError) as e:
            _gpu_step(step, k_scale=ks, append=False)
        assert e.value.status == pa.PA_ERR_INVALID_ARG

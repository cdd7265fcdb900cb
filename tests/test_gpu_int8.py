"""INT8 KV cache with per-row scales on the GPU against the oracle, through
the C ABI: the quantising append is bit-exact (codes and scales), decode
attention is within the bf16 output tolerance of the fp64 oracle on the
same codes and scales."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_parity, from_torch, to_torch
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _gpu_step(step, append=True, mcl=None):
    q = to_torch(step.q, "bf16")
    kc, vc = _dev(step.k_cache), _dev(step.v_cache)
    ks, vs = _dev(step.k_row_scales), _dev(step.v_row_scales)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if append:
        pa.pa_reshape_and_cache_int8(to_torch(step.k_new, "bf16"), to_torch(step.v_new, "bf16"),
                                     to_torch(step.slot_mapping), kc, vc, ks, vs,
                                     error_word=err)
    out = torch.full_like(q, float("nan"))
    pa.pa_decode_int8(q, kc, vc, ks, vs, to_torch(step.block_tables), to_torch(step.context_lens),
                      step.scale, out, step.max_context_len if mcl is None else mcl,
                      error_word=err)
    torch.cuda.synchronize()
    return (kc, vc, ks, vs), wl.as_f32(from_torch(out), "bf16").astype(np.float64), int(err.item())


def _oracle_step(step, append=True):
    kc, vc = step.k_cache.copy(), step.v_cache.copy()
    ks, vs = step.k_row_scales.copy(), step.v_row_scales.copy()
    if append:
        oracle.append_int8(step.k_new, step.v_new, step.slot_mapping, kc, vc, ks, vs)
    out = oracle.decode_int8(step.q, kc, vc, ks, vs, step.block_tables, step.context_lens,
                             step.scale)
    return (kc, vc, ks, vs), out


def test_int8_workload_append_and_decode():
    step = wl.make("8b_gqa_int8")
    dev, got, err = _gpu_step(step)
    pools, want = _oracle_step(step)
    assert err == 0
    for d, w in zip(dev, pools):
        np.testing.assert_array_equal(d.cpu().numpy(), w)
    assert_parity(got, want, "bf16")


@pytest.mark.parametrize("new_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [16, 64, 128, 256])
def test_int8_append_bit_exact(new_dtype, d):
    rng = np.random.default_rng(d + (new_dtype == "f32"))
    nb, hkv, bs, T = 30, 4, 16, 77
    x = rng.standard_normal((2, T, hkv, d)).astype(np.float32)
    x *= 10.0 ** rng.uniform(-4, 4, (2, T, hkv, 1)).astype(np.float32)
    x[:, 5, 2] = 0.0                                     # all-zero rows
    kn, vn = wl.to_cache_dtype(x[0], new_dtype), wl.to_cache_dtype(x[1], new_dtype)
    kc = rng.integers(-128, 128, (nb, hkv, bs, d)).astype(np.int8)
    vc = rng.integers(-128, 128, (nb, hkv, bs, d)).astype(np.int8)
    ks = rng.uniform(0, 1, (nb, hkv, bs)).astype(np.float32)
    vs = rng.uniform(0, 1, (nb, hkv, bs)).astype(np.float32)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[3] = -1
    slots[9] = nb * bs + 1                               # past the pool: flagged, skipped
    dev = [_dev(a) for a in (kc, vc, ks, vs)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache_int8(to_torch(kn, new_dtype), to_torch(vn, new_dtype),
                                 to_torch(slots), *dev, error_word=err)
    torch.cuda.synchronize()
    assert oracle.append_int8(kn, vn, slots, kc, vc, ks, vs) == 1
    assert int(err.item()) == pa.PA_DEVERR_SLOT
    for dv, want in zip(dev, (kc, vc, ks, vs)):
        np.testing.assert_array_equal(dv.cpu().numpy(), want)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8)])
def test_int8_ragged_groups(hq, hkv):
    lens = [1, 15, 16, 17, 100, 511, 512, 513, 1500, 3000]
    step = wl.build_step("i8r", lens, hq, hkv, 128, cache_dtype="int8", seed=hq + hkv)
    _, got, err = _gpu_step(step)
    _, want = _oracle_step(step)
    assert err == 0
    assert_parity(got, want, "bf16")


def test_int8_garbage_scales_past_the_end_do_not_leak():
    lens = [3, 17, 40, 600]
    step = wl.build_step("i8nan", lens, 32, 8, 128, cache_dtype="int8", seed=9)
    bs = step.block_size
    for s, n in enumerate(lens):                 # poison every scale past each sequence's end
        t = step.block_tables[s]
        for i in range(n, -(-n // bs) * bs):
            step.k_row_scales[t[i // bs], :, i % bs] = np.nan
            step.v_row_scales[t[i // bs], :, i % bs] = np.inf
    _, got, _ = _gpu_step(step, append=False)
    _, want = _oracle_step(step, append=False)
    assert np.isfinite(got).all()
    assert_parity(got, want, "bf16")


def test_int8_batch_invariance():
    big = wl.build_step("i8b", [700, 33, 4000, 1, 515], 32, 8, 128, cache_dtype="int8", seed=3)
    _, got_big, _ = _gpu_step(big, append=False)
    for s in (0, 2, 4):
        one = wl.DecodeStep(name="one", cache_dtype="int8", num_heads=32, num_kv_heads=8,
                            head_dim=128, block_size=16, q=big.q[s:s + 1],
                            k_new=big.k_new[s:s + 1], v_new=big.v_new[s:s + 1],
                            slot_mapping=big.slot_mapping[s:s + 1], k_cache=big.k_cache,
                            v_cache=big.v_cache, block_tables=big.block_tables[s:s + 1],
                            context_lens=big.context_lens[s:s + 1], scale=big.scale, seed=0,
                            act_dtype="bf16", k_row_scales=big.k_row_scales,
                            v_row_scales=big.v_row_scales)
        _, got_one, _ = _gpu_step(one, append=False, mcl=big.max_context_len)
        np.testing.assert_array_equal(got_one[0], got_big[s])


def test_int8_unsupported():
    step = wl.build_step("i8u", [20, 40], 32, 8, 64, cache_dtype="int8", seed=1)
    with pytest.raises(pa.PagedAttentionError) as e:
        _gpu_step(step, append=False)                         # head_dim 64
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


def test_int8_copy_on_write_copies_codes_and_scales():
    """pa_copy_blocks on the codes, then on the row scales viewed as a pool of
    one head and one row: the copied blocks decode like the oracle's copy."""
    step = wl.build_step("i8cow", [40, 600, 17], 32, 8, 128, cache_dtype="int8", seed=21)
    nb = step.num_blocks
    rng = np.random.default_rng(4)
    perm = rng.permutation(nb)
    used = sorted({int(b) for b in step.block_tables.ravel() if b >= 0})
    free = [int(b) for b in perm if int(b) not in used]
    mapping = np.array([[used[i], free[i]] for i in range(min(6, len(free)))], np.int64)
    kc, vc = _dev(step.k_cache), _dev(step.v_cache)
    ks, vs = _dev(step.k_row_scales), _dev(step.v_row_scales)
    md = _dev(mapping)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(kc, vc, md, error_word=err)
    hkv, bs = step.num_kv_heads, step.block_size
    pa.pa_copy_blocks(ks.view(nb, 1, 1, hkv * bs), vs.view(nb, 1, 1, hkv * bs), md, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wk, wv = step.k_cache.copy(), step.v_cache.copy()
    wks, wvs = step.k_row_scales.copy(), step.v_row_scales.copy()
    for src, dst in mapping:
        wk[dst], wv[dst], wks[dst], wvs[dst] = wk[src], wv[src], wks[src], wvs[src]
    for dv, want in zip((kc, vc, ks, vs), (wk, wv, wks, wvs)):
        np.testing.assert_array_equal(dv.cpu().numpy(), want)


def _tie_rows(d, dtype):
    """The hand-checked half-way rows of the oracle pin, zero-padded to d
    elements (the row maximum, hence the scale, is unchanged)."""
    import pins
    cases = [r for r in pins.INT8_TIE_ROWS if dtype in r[3]]
    rows = np.zeros((len(cases), d), np.float32)
    want = np.zeros((len(cases), d), np.int8)
    for t, (qs, sc, codes, _) in enumerate(cases):
        rows[t, :16] = [q * sc for q in qs]
        want[t, :16] = codes
    return rows, want, np.array([c[1] for c in cases], np.float32)


@pytest.mark.parametrize("new_dtype", ["bf16", "f32"])
def test_int8_append_rounds_exact_halves_to_even(new_dtype):
    d, hkv = 128, 1
    rows, want, scales = _tie_rows(d, new_dtype)
    T = rows.shape[0]
    nb, bs = T, 16
    kn = wl.to_cache_dtype(rows[:, None, :], new_dtype)
    vn = wl.to_cache_dtype(-rows[:, None, :], new_dtype)
    kc = torch.zeros(nb, hkv, bs, d, dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros(nb, hkv, bs, dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    slots = np.array([t * bs + 5 for t in range(T)], np.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache_int8(to_torch(kn, new_dtype), to_torch(vn, new_dtype),
                                 to_torch(slots), kc, vc, ks, vs, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    k, v = kc.cpu().numpy(), vc.cpu().numpy()
    for t in range(T):
        np.testing.assert_array_equal(k[t, 0, 5], want[t])
        np.testing.assert_array_equal(v[t, 0, 5], -want[t])
    np.testing.assert_array_equal(ks.cpu().numpy()[:, 0, 5], scales)


def test_int8_fused_append_rounds_exact_halves_to_even():
    """The decode kernel's own quantisation of the new rows (pa_append_decode_int8)."""
    rows, want, _ = _tie_rows(128, "bf16")
    T = rows.shape[0]
    step = wl.build_step("ties", [40] * T, 4, 1, 128, cache_dtype="int8", seed=9)
    kn = wl.to_cache_dtype(rows[:, None, :], "bf16")
    vn = wl.to_cache_dtype(-rows[:, None, :], "bf16")
    kc, vc = _dev(step.k_cache), _dev(step.v_cache)
    ks, vs = _dev(step.k_row_scales), _dev(step.v_row_scales)
    q = to_torch(step.q, "bf16")
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_append_decode_int8(to_torch(kn, "bf16"), to_torch(vn, "bf16"),
                             to_torch(step.slot_mapping), kc, vc, ks, vs, q,
                             to_torch(step.block_tables), to_torch(step.context_lens),
                             step.scale, out, step.max_context_len, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    k, v = kc.cpu().numpy(), vc.cpu().numpy()
    for t, slot in enumerate(step.slot_mapping):
        b, o = int(slot) // 16, int(slot) % 16
        np.testing.assert_array_equal(k[b, 0, o], want[t])
        np.testing.assert_array_equal(v[b, 0, o], -want[t])

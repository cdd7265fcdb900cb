"""Parity of the CUDA path with the fp64 oracle, through the C ABI (GPU only).

Bars: the append is bit-exact; attention outputs are within max-abs 1e-4 (fp32
caches) or 2e-2 (bf16 caches) of the oracle run on the same rounded inputs.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import DeviceStep, assert_parity, from_torch, oracle_reference
from parity import assert_elements
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

_CACHE = {}


def named(name):
    """Full-size named workload with its oracle result (generated once)."""
    if name not in _CACHE:
        step = wl.make(name)
        _CACHE[name] = (step, oracle_reference(step))
    return _CACHE[name]


KERNELS_FOR = {"f32": ["auto", "simt", "generic"], "bf16": ["auto", "mma", "simt", "generic"]}


@pytest.mark.parametrize("name", ["tiny", "7b_mha", "8b_gqa", "long_skew", "prefix_shared"])
def test_named_workload_append_and_decode(name):
    step, (k_ref, v_ref, out_ref) = named(name)
    for kernel in KERNELS_FOR[step.cache_dtype]:
        dev = DeviceStep(step)
        out = dev.run(kernel)
        assert dev.error_word() == 0
        if kernel == "auto":   # the append is bit-exact: compare whole pools
            assert np.array_equal(from_torch(dev.k_cache), k_ref)
            assert np.array_equal(from_torch(dev.v_cache), v_ref)
        assert np.isfinite(out).all()
        assert_parity(out, out_ref, step.cache_dtype, f"{name}/{kernel}")


def ragged_step(dtype, hq, hkv, d, bs=16, lens=None, seed=0):
    lens = lens or [1, 15, 16, 17, 31, 100, 511, 512, 513, 1000, 1025, 2047]
    return wl.build_step("ragged", lens, hq, hkv, d, cache_dtype=dtype, block_size=bs, seed=seed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4)])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_shapes_all_kernels(dtype, hq, hkv, d):
    step = ragged_step(dtype, hq, hkv, d, seed=hq + d)
    _, _, ref = oracle_reference(step)
    for kernel in KERNELS_FOR[dtype]:
        dev = DeviceStep(step)
        out = dev.run(kernel)
        assert dev.error_word() == 0
        assert_parity(out, ref, dtype, kernel)


@pytest.mark.parametrize("partition", [16, 48, 64, 512, 1024, 4096])
def test_partition_sizes(partition):
    step = ragged_step("bf16", 32, 8, 128, seed=partition)
    _, _, ref = oracle_reference(step)
    for kernel in ["mma", "simt", "generic"]:
        dev = DeviceStep(step, partition_size=partition)
        out = dev.run(kernel)
        assert_parity(out, ref, "bf16", (kernel, partition))


@pytest.mark.parametrize("long_p,long_from", [(1024, 1000), (2048, 600), (4096, 512)])
def test_long_partitions(long_p, long_from):
    """Larger partitions for sequences past a length (pa_decode_ex option):
    parity on every kernel, lengths on both sides of the threshold, and a
    sequence's result bitwise the same alone and inside the batch."""
    lens = [1, 17, 511, 512, 599, 600, 601, 999, 1000, 1001, 2047, 4096, 4097, 9000, 20000]
    step = ragged_step("bf16", 32, 8, 128, lens=lens, seed=long_p)
    _, _, ref = oracle_reference(step)
    opts = dict(long_partition_size=long_p, long_partition_from=long_from)
    for kernel in ["mma", "simt", "generic"]:
        dev = DeviceStep(step)
        dev.append()
        pa.pa_decode(dev.q, dev.k_cache, dev.v_cache, dev.tables, dev.lens, step.scale, dev.out,
                     step.max_context_len, workspace=dev.workspace, error_word=dev.err,
                     kernel=kernel, **opts)
        torch.cuda.synchronize()
        assert dev.error_word() == 0
        out = dev.result()
        assert_parity(out, ref, "bf16", (kernel, long_p, long_from))
        if kernel == "mma":
            # the 20,000-row sequence alone gives the same bits
            one = wl.DecodeStep(**{**step.__dict__, "q": step.q[-1:],
                                   "block_tables": step.block_tables[-1:],
                                   "context_lens": step.context_lens[-1:]})
            sub = DeviceStep(one)
            sub.k_cache.copy_(dev.k_cache)
            sub.v_cache.copy_(dev.v_cache)
            pa.pa_decode(sub.q, sub.k_cache, sub.v_cache, sub.tables, sub.lens, step.scale,
                         sub.out, 20000, workspace=sub.workspace, error_word=sub.err,
                         kernel="mma", **opts)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(from_torch(sub.out)[0], from_torch(dev.out)[-1])


@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 32, 64])
def test_block_sizes(bs):
    step = ragged_step("bf16", 8, 2, 128, bs=bs, lens=[1, 7, 16, 33, 300, 777], seed=bs)
    k_ref, v_ref, ref = oracle_reference(step)
    dev = DeviceStep(step)
    out = dev.run("auto")
    assert np.array_equal(from_torch(dev.k_cache), k_ref)
    assert_parity(out, ref, "bf16")
    if bs % 16 == 0:
        dev2 = DeviceStep(step)
        assert_parity(dev2.run("simt"), ref, "bf16")


def test_garbage_rows_do_not_leak():
    """Unused pool rows (past each sequence and in unused blocks) set to NaN."""
    for dtype in ("f32", "bf16"):
        step = ragged_step(dtype, 32, 8, 128, seed=5)
        used = np.zeros(step.k_cache.shape[:1] + step.k_cache.shape[2:3], dtype=bool)
        for s, n in enumerate(step.context_lens):
            for i in range(int(n)):
                used[step.block_tables[s, i // 16], i % 16] = True
        nan = np.float32(np.nan)
        fill = wl.to_cache_dtype(np.array([nan], np.float32), dtype)[0] if dtype == "f32" \
            else np.uint16(0x7fc0)
        for pool in (step.k_cache, step.v_cache):
            pool.transpose(0, 2, 1, 3)[~used] = fill
        # the appended rows must still come from k_new/v_new
        _, _, ref = oracle_reference(step)
        for kernel in KERNELS_FOR[dtype][1:]:
            out = DeviceStep(step).run(kernel)
            assert np.isfinite(out).all(), kernel
            assert_parity(out, ref, dtype, kernel)


def _run_subset(step, dev, idx, kernel):
    """Decode only the sequences `idx` (in that order) against dev's appended pool."""
    sub = DeviceStep(wl.DecodeStep(**{**step.__dict__, "q": step.q[idx],
                                      "block_tables": step.block_tables[idx],
                                      "context_lens": step.context_lens[idx]}))
    sub.k_cache.copy_(dev.k_cache)
    sub.v_cache.copy_(dev.v_cache)
    sub.decode(kernel, max_context_len=int(step.context_lens[idx].max()))
    torch.cuda.synchronize()
    assert sub.error_word() == 0
    return from_torch(sub.out)


def test_batch_invariance_and_determinism():
    """A sequence's output bits do not depend on the rest of the batch: run
    alone, inside a batch large enough that every persistent CTA processes
    many items, and inside a permuted batch with a 40,000-row sequence."""
    rng = np.random.default_rng(77)
    lens = list(rng.integers(1, 3000, size=95)) + [40_000]
    step = wl.build_step("invariance", lens, 32, 8, 128, seed=21)
    B = step.num_seqs
    for kernel in ["mma", "simt", "generic"]:
        dev = DeviceStep(step)
        dev.run(kernel)
        batch_out = from_torch(dev.out)
        dev.decode(kernel)
        torch.cuda.synchronize()
        assert np.array_equal(from_torch(dev.out), batch_out), "not deterministic"
        for s in [0, 7, 50, B - 1]:
            single = _run_subset(step, dev, np.array([s]), kernel)
            assert np.array_equal(single[0], batch_out[s]), (kernel, s)
        perm = rng.permutation(B)
        shuffled = _run_subset(step, dev, perm, kernel)
        assert np.array_equal(shuffled, batch_out[perm]), kernel


def test_block_permutation_is_invisible():
    step = ragged_step("bf16", 32, 8, 128, seed=13)
    base = DeviceStep(step).run("mma")
    perm = np.random.default_rng(0).permutation(step.num_blocks)
    k2, v2 = np.empty_like(step.k_cache), np.empty_like(step.v_cache)
    k2[perm], v2[perm] = step.k_cache, step.v_cache
    bt2 = np.where(step.block_tables >= 0, perm[np.maximum(step.block_tables, 0)], -1)
    slots2 = perm[step.slot_mapping // 16] * 16 + step.slot_mapping % 16
    step2 = wl.DecodeStep(**{**step.__dict__, "k_cache": k2, "v_cache": v2,
                             "block_tables": bt2.astype(np.int32),
                             "slot_mapping": slots2.astype(np.int64)})
    for kernel in ["mma", "simt", "generic"]:
        a = DeviceStep(step).run(kernel)
        b = DeviceStep(step2).run(kernel)
        assert np.array_equal(a, b), kernel
    assert np.isfinite(base).all()


def test_empty_sequences_give_zeros():
    step = ragged_step("bf16", 8, 2, 64, lens=[0, 5, 0, 600, 0])
    _, _, ref = oracle_reference(step)
    for kernel in ["mma", "simt", "generic"]:
        dev = DeviceStep(step)
        dev.out.fill_(7.0)
        out = dev.run(kernel)
        assert np.all(out[[0, 2, 4]] == 0.0)
        assert_parity(out, ref, "bf16")


def test_device_errors_are_flagged_not_faulted():
    step = ragged_step("bf16", 8, 2, 128, lens=[40, 700, 33], seed=3)
    _, _, ref = oracle_reference(step)
    for kernel in ["mma", "simt", "generic"]:
        dev = DeviceStep(step)
        dev.append()
        bad = dev.tables.clone()
        bad[1, 2] = step.num_blocks + 5            # outside the pool
        dev.tables = bad
        dev.decode(kernel)
        torch.cuda.synchronize()
        assert dev.error_word() & pa.PA_DEVERR_BLOCK_ID, kernel
        out = dev.result()
        assert_parity(out[[0, 2]], ref[[0, 2]], "bf16")
    dev = DeviceStep(step)
    dev.append()
    dev.lens[2] = 10_000                           # past max_context_len
    dev.decode("mma")
    torch.cuda.synchronize()
    assert dev.error_word() & pa.PA_DEVERR_CONTEXT
    dev = DeviceStep(step)
    dev.slots[0] = step.num_blocks * 16            # past the pool
    dev.append()
    torch.cuda.synchronize()
    assert dev.error_word() & pa.PA_DEVERR_SLOT


def test_host_argument_errors():
    step = ragged_step("bf16", 8, 2, 128, lens=[600, 20])
    dev = DeviceStep(step)
    with pytest.raises(pa.PagedAttentionError) as e:          # workspace too small
        pa.pa_decode(dev.q, dev.k_cache, dev.v_cache, dev.tables, dev.lens, 0.1, dev.out, 600,
                     workspace=dev.workspace[:8])
    assert e.value.status == pa.PA_ERR_WORKSPACE
    with pytest.raises(pa.PagedAttentionError) as e:          # max_context_len past the table
        pa.pa_decode(dev.q, dev.k_cache, dev.v_cache, dev.tables, dev.lens, 0.1, dev.out,
                     dev.tables.shape[1] * 16 + 1, workspace=dev.workspace)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    with pytest.raises(pa.PagedAttentionError) as e:          # partition not a multiple of 16
        pa.pa_decode(dev.q, dev.k_cache, dev.v_cache, dev.tables, dev.lens, 0.1, dev.out, 600,
                     workspace=dev.workspace, partition_size=40)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    f32 = DeviceStep(ragged_step("f32", 8, 2, 128, lens=[10]))
    with pytest.raises(pa.PagedAttentionError) as e:
        f32.decode("mma")
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


def test_incremental_steps_follow_the_oracle():
    """Three decode steps in a row: every step appends one row and attends."""
    import oracle
    from paged_kv_cache_29_gb300.block_manager import BlockManager
    rng = np.random.default_rng(1)
    hq, hkv, d, bs, nb = 8, 2, 128, 16, 64
    lens0 = [15, 16, 200]
    mgr = BlockManager(nb, bs, free_order=rng.permutation(nb), prefix_caching=False)
    for s, n in enumerate(lens0):
        mgr.admit(f"s{s}", [0] * n)
    k = wl.to_cache_dtype(rng.standard_normal((nb, hkv, bs, d), dtype=np.float32), "bf16")
    v = wl.to_cache_dtype(rng.standard_normal((nb, hkv, bs, d), dtype=np.float32), "bf16")
    kd = torch.from_numpy(k.copy()).view(torch.bfloat16).cuda()
    vd = torch.from_numpy(v.copy()).view(torch.bfloat16).cuda()
    for _ in range(3):
        slots = np.array([mgr.append(f"s{s}", 0).slot for s in range(3)], np.int64)
        lens = np.array([mgr.num_tokens(f"s{s}") for s in range(3)], np.int32)
        bt = np.full((3, 16), -1, np.int32)
        for s in range(3):
            t = mgr.block_table(f"s{s}")
            bt[s, :len(t)] = t
        q = wl.to_cache_dtype(rng.standard_normal((3, hq, d), dtype=np.float32), "bf16")
        kn = wl.to_cache_dtype(rng.standard_normal((3, hkv, d), dtype=np.float32), "bf16")
        vn = wl.to_cache_dtype(rng.standard_normal((3, hkv, d), dtype=np.float32), "bf16")
        oracle.append(kn, vn, slots, k, v)
        ref = oracle.decode(q, k, v, bt, lens, 1 / np.sqrt(d))
        dq = torch.from_numpy(q).view(torch.bfloat16).cuda()
        out = torch.empty_like(dq)
        pa.pa_reshape_and_cache(torch.from_numpy(kn).view(torch.bfloat16).cuda(),
                                torch.from_numpy(vn).view(torch.bfloat16).cuda(),
                                torch.from_numpy(slots).cuda(), kd, vd)
        pa.pa_decode(dq, kd, vd, torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda(),
                     1 / np.sqrt(d), out, int(lens.max()))
        torch.cuda.synchronize()
        got = wl.as_f32(from_torch(out), "bf16").astype(np.float64)
        assert_parity(got, ref, "bf16")
        assert np.array_equal(from_torch(kd), k) and np.array_equal(from_torch(vd), v)


# Element bound for the structured inputs (checked for sensitivity on the CPU
# in tests/test_parity_bounds.py): one bf16 ulp of the element plus 2^-16 of
# the row's largest element for the fp32 weight arithmetic.
STRUCT_ULPS, STRUCT_REL = 1.0, 2.0 ** -16


@pytest.mark.parametrize("variant", ["uniform", "weighted"])
def test_structured_long_context(variant):
    """long_skew's shape (one 100,000-row sequence, seven of 1,500) with V
    rows that carry a Walsh pattern of their tile index and K rows that give
    every row the same weight ("uniform") or a different weight per 512-row
    chunk ("weighted"). Many output elements are then exactly zero, and a
    dropped, repeated or re-weighted tile or partition moves them far past
    the element bound (tests/test_parity_bounds.py shows this on the CPU).
    The 100,000-row sequence spans well over 32 partitions, so its heads go
    through the merge kernel's multi-warp branch."""
    step = wl.structured_long(variant)
    assert -(-100_000 // pa.pa_default_partition_size("bf16")) > 32
    k_ref, v_ref, ref = oracle_reference(step)
    runs = {}
    for kernel in ("auto", "simt"):
        dev = DeviceStep(step)
        runs[kernel] = dev.run(kernel)
        assert dev.error_word() == 0
        if kernel == "auto":
            assert np.array_equal(from_torch(dev.k_cache), k_ref)
            assert np.array_equal(from_torch(dev.v_cache), v_ref)
    fused = DeviceStep(step)
    pa.pa_append_decode(fused.k_new, fused.v_new, fused.slots, fused.k_cache, fused.v_cache,
                        fused.q, fused.tables, fused.lens, step.scale, fused.out,
                        step.max_context_len, workspace=fused.workspace, error_word=fused.err)
    torch.cuda.synchronize()
    assert fused.error_word() == 0
    runs["fused"] = fused.result()
    for what, out in runs.items():
        assert_elements(out, ref, "bf16", STRUCT_ULPS, STRUCT_REL, f"{variant}/{what}")
        assert_parity(out, ref, "bf16", f"{variant}/{what}")

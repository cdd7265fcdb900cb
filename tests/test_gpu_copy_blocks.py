"""pa_copy_blocks (copy-on-write of whole cache blocks) against the oracle,
through the C ABI (GPU only). The copy is bit-exact."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_parity, from_torch, max_abs, to_torch
import oracle
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl
from paged_kv_cache_29_gb300.block_manager import BlockManager

pytestmark = pytest.mark.gpu


def _pool(rng, nb, hkv, bs, d, dtype):
    k = wl.to_cache_dtype(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
    v = wl.to_cache_dtype(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
    return k, v


def _mapping(rng, nb, pairs, extra=()):
    perm = rng.permutation(nb)
    m = np.stack([perm[:pairs], perm[pairs:2 * pairs]], axis=1).astype(np.int64)
    if extra:
        m = np.concatenate([m, np.array(extra, np.int64).reshape(-1, 2)])
    return m


def _run(k, v, mapping, dtype):
    kd, vd = to_torch(k, dtype), to_torch(v, dtype)
    md = torch.from_numpy(np.ascontiguousarray(mapping)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(kd, vd, md, error_word=err)
    torch.cuda.synchronize()
    return from_torch(kd), from_torch(vd), int(err.item())


@pytest.mark.parametrize("dtype,hkv,bs,d,pairs", [
    ("f32", 2, 16, 64, 37), ("bf16", 8, 16, 128, 300), ("bf16", 1, 1, 8, 5),
    ("f32", 4, 5, 12, 64), ("bf16", 32, 16, 128, 17)])
def test_copy_blocks_bit_exact(dtype, hkv, bs, d, pairs):
    rng = np.random.default_rng(pairs)
    nb = 2 * pairs + 11
    k, v = _pool(rng, nb, hkv, bs, d, dtype)
    mapping = _mapping(rng, nb, pairs, extra=[[-1, 0], [3, -1]])   # skipped pairs
    gk, gv, err = _run(k, v, mapping, dtype)
    wk, wv = k.copy(), v.copy()
    assert oracle.copy_blocks(wk, wv, mapping) == 0
    assert err == 0
    np.testing.assert_array_equal(gk, wk)
    np.testing.assert_array_equal(gv, wv)


def test_copy_blocks_out_of_range_is_flagged_and_skipped():
    rng = np.random.default_rng(5)
    nb = 40
    k, v = _pool(rng, nb, 2, 16, 64, "bf16")
    mapping = _mapping(rng, nb, 10, extra=[[nb, 1], [2, nb + 7]])
    gk, gv, err = _run(k, v, mapping, "bf16")
    wk, wv = k.copy(), v.copy()
    assert oracle.copy_blocks(wk, wv, mapping) == 2
    assert err == pa.PA_DEVERR_BLOCK_ID
    np.testing.assert_array_equal(gk, wk)
    np.testing.assert_array_equal(gv, wv)


def test_copy_blocks_empty_and_host_errors():
    k = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    pa.pa_copy_blocks(k, v, torch.zeros(0, 2, dtype=torch.int64, device="cuda"))
    with pytest.raises(TypeError):
        pa.pa_copy_blocks(k, v, torch.zeros(1, 2, dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        pa.pa_copy_blocks(k, v, torch.zeros(1, 3, dtype=torch.int64, device="cuda"))
    L = pa.lib()
    assert L.pa_copy_blocks(k.data_ptr(), v.data_ptr(), None, 1, 2, 64, 16, 4, 1, None,
                            None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_copy_blocks(k.data_ptr(), v.data_ptr(), None, 1, 2, 3, 16, 4, 1, None,
                            None) == pa.PA_ERR_UNSUPPORTED   # 6-byte rows


def test_fork_copy_append_decode_follows_the_oracle():
    """A forked sequence writes into its shared partial block: the copy, the
    append and the decode on the GPU match the oracle doing the same."""
    rng = np.random.default_rng(77)
    nb, bs, hkv, hq, d = 64, 16, 8, 32, 128
    mgr = BlockManager(nb, bs, free_order=rng.permutation(nb), prefix_caching=False)
    mgr.admit("p", list(range(600)))            # 37.5 blocks: the last is partial
    for c in range(1, 4):
        mgr.fork("p", f"c{c}")
    k, v = _pool(rng, nb, hkv, bs, d, "bf16")
    seqs = ["p", "c1", "c2", "c3"]
    pairs, slots = [], []
    for s in seqs[1:] + seqs[:1]:
        r = mgr.append(s, 1)
        if r.copy_on_write:
            pairs.append(r.copy_on_write)
        slots.append(r.slot)
    assert len(pairs) == 3                       # every writer but the last copies
    order = seqs[1:] + seqs[:1]
    slot_of = dict(zip(order, slots))
    slots = np.array([slot_of[s] for s in seqs], np.int64)
    tables = np.full((4, 40), -1, np.int32)
    for i, s in enumerate(seqs):
        t = mgr.block_table(s)
        tables[i, :len(t)] = t
    lens = np.full(4, 601, np.int32)
    q = wl.to_cache_dtype(rng.standard_normal((4, hq, d)).astype(np.float32), "bf16")
    kn = wl.to_cache_dtype(rng.standard_normal((4, hkv, d)).astype(np.float32), "bf16")
    vn = wl.to_cache_dtype(rng.standard_normal((4, hkv, d)).astype(np.float32), "bf16")
    mapping = np.array(pairs, np.int64)
    scale = 1.0 / np.sqrt(d)
    # oracle
    wk, wv = k.copy(), v.copy()
    oracle.copy_blocks(wk, wv, mapping)
    oracle.append(kn, vn, slots, wk, wv)
    want = oracle.decode(q, wk, wv, tables, lens, scale)
    # GPU
    kd, vd = to_torch(k, "bf16"), to_torch(v, "bf16")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(kd, vd, torch.from_numpy(mapping).cuda(), error_word=err)
    pa.pa_reshape_and_cache(to_torch(kn, "bf16"), to_torch(vn, "bf16"),
                            torch.from_numpy(slots).cuda(), kd, vd, error_word=err)
    out = torch.empty(4, hq, d, dtype=torch.bfloat16, device="cuda")
    pa.pa_decode(to_torch(q, "bf16"), kd, vd, torch.from_numpy(tables).cuda(),
                 torch.from_numpy(lens).cuda(), scale, out, 601, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(from_torch(kd), wk)
    np.testing.assert_array_equal(from_torch(vd), wv)
    got = wl.as_f32(from_torch(out), "bf16").astype(np.float64)
    assert_parity(got, want, "bf16")
    # the four sequences now differ only in their last row
    assert max_abs(want[0], want[1]) > 0


def test_copy_blocks_at_bench_size():
    """The bench's copy measurement: 4096 random distinct pairs over the 8B GQA
    pool (8 KV heads, 16 rows, head_dim 128, bf16), compared in full."""
    step = wl.make("8b_gqa")
    rng = np.random.default_rng(123)
    nb = step.num_blocks
    mapping = _mapping(rng, nb, 4096)
    gk, gv, err = _run(step.k_cache, step.v_cache, mapping, "bf16")
    wk, wv = step.k_cache.copy(), step.v_cache.copy()
    oracle.copy_blocks(wk, wv, mapping)
    assert err == 0
    np.testing.assert_array_equal(gk, wk)
    np.testing.assert_array_equal(gv, wv)

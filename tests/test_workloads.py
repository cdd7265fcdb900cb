"""Seeded inputs: shapes, lengths, rounding and determinism (small configs only)."""
import numpy as np
import torch

from paged_kv_cache_29_gb300 import workloads as wl
from paged_kv_cache_29_gb300.block_manager import BlockManager


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100_000).astype(np.float32) * 10,
                        np.array([1.00390625, 1.01171875, -2.00390625, 0.0, -0.0],
                                 dtype=np.float32)])   # exact ties round to even
    ours = wl.round_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = wl.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_tiny_workload_shape():
    s = wl.tiny()
    assert s.cache_dtype == "f32" and s.k_cache.shape == (32, 2, 16, 64)
    assert s.context_lens.tolist() == [5, 17, 33, 64]
    assert s.q.shape == (4, 4, 64) and s.k_new.shape == (4, 2, 64)
    used = s.block_tables[s.block_tables >= 0]
    assert len(used) == 10 and len(set(used.tolist())) == 10
    for seq, n in enumerate(s.context_lens):
        i = n - 1
        assert s.slot_mapping[seq] == s.block_tables[seq, i // 16] * 16 + i % 16
    assert abs(s.scale - 1 / 8) < 1e-15


def test_generation_is_deterministic():
    a, b = wl.tiny(), wl.tiny()
    for name in ("q", "k_new", "v_new", "k_cache", "v_cache", "block_tables", "slot_mapping"):
        assert np.array_equal(getattr(a, name), getattr(b, name))
    c = wl.tiny(seed=5)
    assert not np.array_equal(a.k_cache, c.k_cache)


def test_8b_gqa_lengths_follow_the_recipe():
    lens = wl.gqa_8b_lengths(np.random.default_rng(wl.WORKLOAD_SEEDS["8b_gqa"]))
    assert lens.shape == (128,) and lens.min() >= 16 and lens.max() <= 8192 + 300
    assert 1400 < lens.mean() < 1900


def test_small_prefix_shared_structure():
    s = wl.prefix_shared(samples=4, prefix=64, max_tail=20)
    shared = s.block_tables[:, :4]
    assert (shared == shared[0]).all()
    assert s.meta["shared_refcount_min"] == 4
    tails = [set(r[4:][r[4:] >= 0].tolist()) for r in s.block_tables]
    for i in range(4):
        for j in range(i + 1, 4):
            assert not tails[i] & tails[j]


def test_chunked_values_do_not_depend_on_threads(monkeypatch):
    rng1 = np.random.default_rng(3)
    a = wl._normal(rng1, (3, 1 << 21), "bf16")
    monkeypatch.setattr(wl.os, "cpu_count", lambda: 1)
    rng2 = np.random.default_rng(3)
    b = wl._normal(rng2, (3, 1 << 21), "bf16")
    assert np.array_equal(a, b)


def test_idle_sequence_has_no_append():
    s = wl.build_step("x", [0, 3], 2, 1, 8, cache_dtype="f32")
    assert s.slot_mapping[0] == -1 and (s.block_tables[0] == -1).all()
    assert BlockManager  # imported for the module's public surface

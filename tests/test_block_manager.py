"""Host block manager: the pages' printed demo, fragmentation, sharing, LRU."""
import numpy as np
import pytest

import golden_io
from paged_kv_cache_29_gb300.block_manager import BlockManager, OutOfBlocks


def test_demo_matches_printed_output():
    """Same scenario as the printed demo of "Batching and the KV Cache"."""
    want = golden_io.read("block_manager_demo.txt")["printed"]
    m = BlockManager(num_blocks=64)
    system = list(range(1000, 1040))
    got = [m.admit("a", system + [1, 2, 3]), m.admit("b", system + [7, 8])]
    m.fork("b", "b2")
    m.append("b2", 99)
    got.append(m.num_free)
    got.append(m.admit("c", [999] + system[1:]))
    got.append(m.admit("d", system, salt="tenant-42"))
    for seq in ("a", "b", "b2"):
        m.release(seq)
    got.append(m.admit("e", system))
    m.check()
    assert got == want


def test_fragmentation_at_most_one_partial_block():
    """At most block_size - 1 = 15 wasted slots per sequence, at every step."""
    rng = np.random.default_rng(0)
    m = BlockManager(4096, 16, free_order=rng.permutation(4096))
    lens = rng.integers(0, 700, size=40)
    for s, n in enumerate(lens):
        m.admit(f"s{s}", rng.integers(0, 50_000, size=int(n)).tolist())
        assert 0 <= m.wasted_slots(f"s{s}") <= 15
    for _ in range(100):
        s = int(rng.integers(0, len(lens)))
        m.append(f"s{s}", int(rng.integers(0, 50_000)))
        assert 0 <= m.wasted_slots(f"s{s}") <= 15
    m.check()


def test_fork_shares_and_copy_on_write_copies_once():
    m = BlockManager(16, 16, prefix_caching=False)
    m.admit("p", list(range(40)))
    m.fork("p", "c")
    t = m.block_table("p")
    assert m.block_table("c") == t and all(m.refcount(b) == 2 for b in t)
    r = m.append("c", 1)
    assert r.copy_on_write == (t[-1], m.block_table("c")[-1])
    assert m.refcount(t[-1]) == 1 and m.block_table("c")[:2] == t[:2]
    assert r.slot == m.block_table("c")[-1] * 16 + 8
    r2 = m.append("c", 2)                       # now private: no second copy
    assert r2.copy_on_write is None and r2.slot == r.slot + 1
    m.check()


def test_full_shared_block_needs_no_copy():
    """Forking on a block boundary: the first append opens a private block."""
    m = BlockManager(8, 16, prefix_caching=False)
    m.admit("p", list(range(32)))
    m.fork("p", "c")
    r = m.append("c", 0)
    assert r.copy_on_write is None
    assert m.block_table("c")[:2] == m.block_table("p")
    m.check()


def test_out_of_blocks_raises_and_leaves_state_intact():
    m = BlockManager(3, 16, prefix_caching=False)
    m.admit("a", list(range(32)))
    with pytest.raises(OutOfBlocks):
        m.admit("b", list(range(40)))
    assert m.num_free == 1 and m.sequences() == ["a"]
    m.check()
    m.admit("c", [1])
    with pytest.raises(OutOfBlocks):
        m.append("a", 5)
    m.check()


def test_slots_follow_the_block_table():
    rng = np.random.default_rng(4)
    m = BlockManager(32, 4, free_order=rng.permutation(32), prefix_caching=False)
    m.admit("s", [])
    slots = [m.append("s", i).slot for i in range(23)]
    table = m.block_table("s")
    assert slots == [table[i // 4] * 4 + i % 4 for i in range(23)]
    assert len(set(slots)) == 23 and m.num_tokens("s") == 23


def test_release_order_and_lru_reuse():
    """Released blocks join the queue tail, last block first; untouched free
    blocks are handed out before them."""
    m = BlockManager(6, 2, prefix_caching=False)
    m.admit("a", [1, 2, 3, 4, 5])               # blocks 0, 1, 2
    m.release("a")
    m.admit("b", [9] * 6)                       # 3, 4, 5 first, never 2, 1, 0
    assert m.block_table("b") == [3, 4, 5]
    m.admit("c", [8] * 2)
    assert m.block_table("c") == [2]
    m.check()


def test_incremental_rows_match_naive_decoder():
    g = golden_io.read("naive_decoder.txt")
    m = BlockManager(4, 16)
    m.admit("s", list(range(g["prompt"])))
    for t in range(g["decoded"]):
        m.append("s", 100 + t)
    assert m.num_tokens("s") == g["cache_rows"]


def test_prefix_reuse_shares_full_blocks_only():
    """A second request with the same prompt reuses the unbroken run of full
    cached blocks from its start (reference counts go up, no new blocks); its
    partly filled last block is its own."""
    m = BlockManager(32, 4)
    prompt = list(range(10))                     # 2 full blocks + 2 tokens
    assert m.admit("a", prompt) == 0
    free_before = m.num_free
    assert m.admit("b", prompt) == 8
    ta, tb = m.block_table("a"), m.block_table("b")
    assert ta[:2] == tb[:2] and ta[2] != tb[2]
    assert [m.refcount(x) for x in tb] == [2, 2, 1]
    assert m.num_free == free_before - 1         # only the partial block is new
    m.check()


def test_salt_isolates_prefix_caches():
    m = BlockManager(32, 4)
    prompt = list(range(12))
    m.admit("a", prompt, salt="tenant-1")
    assert m.admit("b", prompt, salt="tenant-2") == 0
    assert set(m.block_table("a")).isdisjoint(m.block_table("b"))
    assert m.admit("c", prompt, salt="tenant-1") == 12
    m.check()


def test_chain_key_breaks_at_the_first_differing_block():
    """Blocks match only as an unbroken run from the start: a prompt that
    differs in block 1 reuses block 0 and nothing after it, even where a later
    block's tokens are the same."""
    m = BlockManager(32, 4)
    m.admit("a", list(range(12)))
    other = list(range(12))
    other[5] = 99                                # block 1 differs, block 2 identical
    assert m.admit("b", other) == 4
    ta, tb = m.block_table("a"), m.block_table("b")
    assert ta[0] == tb[0] and ta[1] != tb[1] and ta[2] != tb[2]
    m.check()


def test_released_blocks_stay_reusable_until_handed_out_again():
    """A finished request's blocks join the LRU free queue with their keys: a
    new identical prompt revives them; once the free queue hands a block out
    to other data, its key is gone."""
    m = BlockManager(4, 4)
    prompt = list(range(8))
    m.admit("a", prompt)
    blocks = m.block_table("a")
    m.release("a")
    assert m.num_free == 4
    assert m.admit("b", prompt) == 8              # revived from the free queue
    assert m.block_table("b") == blocks
    m.release("b")
    # Allocate every block for other tokens: the cached blocks are reused and
    # their keys evicted.
    m.admit("c", list(range(100, 116)))
    m.release("c")
    assert m.admit("d", prompt) == 0
    m.check()

"""Byte and block accounting against the pages' worked examples."""
import numpy as np

import golden_io
from paged_kv_cache_29_gb300 import accounting as acc

G = golden_io.read("kv_accounting.txt")


def test_bytes_per_token_examples():
    assert acc.kv_bytes_per_token(80, 8, 128, 2) == G["llama33_70b_bf16_bytes_per_token"]
    assert acc.mla_bytes_per_token(512, 64, 61, 2) == G["deepseek_v3_mla_bytes_per_token"]
    assert 61 * 128 * (192 + 128) * 2 == G["deepseek_v3_mha_bytes_per_token"]
    assert acc.kv_bytes_per_token(32, 32, 128, 2) == G["mha_7b_bytes_per_token"]
    assert acc.kv_bytes_per_token(32, 8, 128, 2) == G["gqa_7b_bytes_per_token"]
    assert acc.kv_bytes_per_token(32, 32, 128, 2) * 4096 == G["mha_7b_bytes_4096"]
    assert acc.kv_bytes_per_token(32, 8, 128, 2) * 4096 == G["gqa_7b_bytes_4096"]
    assert acc.kv_bytes_per_token(32, 32, 128, 2) * 4096 * 32 == G["mha_7b_bytes_4096_x32"]


def test_block_budget_worked_example():
    per_token = acc.kv_bytes_per_token(32, 8, 128, 2)
    assert per_token == G["llama3_8b_bytes_per_token"]
    block = 16 * per_token
    assert block == G["llama3_8b_block_bytes"]
    blocks = acc.budget_blocks(62 * 1024 * 2**20, block)
    assert blocks == G["budget_blocks_62gb"]
    assert acc.blocks_for_tokens(5000) == G["blocks_per_5k_request"]
    assert acc.admissible_requests(blocks, acc.blocks_for_tokens(5000)) == \
        G["requests_without_sharing"]
    assert acc.blocks_for_tokens(1000) == G["shared_prefix_blocks"]
    assert acc.blocks_for_tokens(4000) == G["private_blocks_per_request"]
    assert acc.admissible_requests(blocks, 250, shared_blocks=63) == \
        G["requests_with_shared_prefix"]


def test_step_bytes_closed_form():
    lens = np.array([1, 16, 17, 0])
    b = acc.step_bytes(lens, num_heads=8, num_kv_heads=2, head_dim=64, elem_bytes=2)
    row = 2 * 64 * 2
    assert b.kv == 34 * row * 2
    assert b.q_out == 4 * 8 * 64 * 2 * 2
    assert b.tables == (1 + 1 + 2 + 0) * 4 + 4 * 4
    assert b.append == 3 * 2 * 64 * 2 * 2 * 2 + 4 * 8   # K and V, read and written
    assert b.decode == b.kv + b.q_out + b.tables and b.total == b.decode + b.append


def test_unique_bytes_count_shared_rows_once():
    bt = np.array([[0, 1, -1], [0, 2, -1]])
    lens = np.array([20, 30])
    b = acc.step_bytes(lens, 4, 1, 8, 2, block_size=16, block_tables=bt)
    # rows: block 0 (16 shared), block 1 (4), block 2 (14)
    assert b.kv_unique == (16 + 4 + 14) * 8 * 2 * 2
    assert b.kv == 50 * 8 * 2 * 2

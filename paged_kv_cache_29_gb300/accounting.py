"""Byte and block accounting for the paged KV cache and one decode step.

Formulas:
  * KV bytes per token = 2 x layers x KV heads x head dim x bytes per element
    ("Batching and the KV Cache", section 6, and "LLM inference and serving",
    "KV-cache size"); for latent attention (r_kv + d_rope) x layers x bytes
    (same chapter, the MLA formula).
  * blocks for T tokens = ceil(T / block_size) ("Chapter 29 Building a
    Production LLM Serving Stack", 29.1.2, the worked example).
  * A decode step's algorithmic bytes: every attended K and V row once, q read
    and out written once, the block-table entries the sequences use, the
    context lengths, and the append (new K/V rows read and written, slots read).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int,
                       bytes_per_elem: int) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_elem


def mla_bytes_per_token(kv_lora_rank: int, rope_dim: int, num_layers: int,
                        bytes_per_elem: int) -> int:
    return (kv_lora_rank + rope_dim) * num_layers * bytes_per_elem


def blocks_for_tokens(tokens: int, block_size: int = 16) -> int:
    return -(-int(tokens) // block_size)


@dataclass(frozen=True)
class StepBytes:
    kv: int            # K and V rows attended (logical: shared blocks counted per reader)
    q_out: int         # q read + out written
    tables: int        # block-table entries used + context lengths
    append: int        # new K/V rows read and written + slot mapping read
    kv_unique: int     # K and V bytes of the distinct physical rows attended

    @property
    def decode(self) -> int:
        """Bytes the attention kernel must move: kv + q/out + tables."""
        return self.kv + self.q_out + self.tables

    @property
    def total(self) -> int:
        return self.decode + self.append


def step_bytes(context_lens, num_heads: int, num_kv_heads: int, head_dim: int,
               elem_bytes: int, block_size: int = 16, block_tables=None,
               act_bytes: int | None = None, num_queries: int = 1,
               window: int = 0, row_scale_bytes: int = 0) -> StepBytes:
    """elem_bytes: bytes per cache element; act_bytes: bytes per element of q,
    out and the new K/V rows (default: elem_bytes); num_queries: new tokens
    (queries) per sequence; window: a sliding window of rows attended (0 =
    all): K/V and table bytes count the attended rows only; row_scale_bytes:
    bytes of scale stored per (row, KV head) of K and of V (4 for an INT8
    cache), read and written with the rows."""
    act = elem_bytes if act_bytes is None else act_bytes
    lens = np.asarray(context_lens, dtype=np.int64)
    B = int(lens.shape[0])
    first = np.maximum(lens - window, 0) if window > 0 else np.zeros_like(lens)
    row = num_kv_heads * (head_dim * elem_bytes + row_scale_bytes)   # one token, K or V
    kv = int((lens - first).sum()) * row * 2
    Q = int(num_queries)
    q_out = B * Q * num_heads * head_dim * act * 2
    used_entries = int(sum(blocks_for_tokens(int(n), block_size) - int(f) // block_size
                           for n, f in zip(lens, first)))
    tables = used_entries * 4 + B * 4
    active = int((lens > 0).sum())
    # new K and V rows read (act dtype) and written (cache dtype), slots read
    append = (active * Q * num_kv_heads * 2 * (head_dim * (act + elem_bytes) + row_scale_bytes)
              + B * Q * 8)
    if block_tables is None:
        kv_unique = kv
    else:
        bt = np.asarray(block_tables, dtype=np.int64)
        slots = [bt[s, np.arange(f, n) // block_size] * block_size + np.arange(f, n) % block_size
                 for s, (n, f) in enumerate(zip(lens, first)) if n > 0]
        distinct = np.unique(np.concatenate(slots)).size if slots else 0
        kv_unique = int(distinct) * row * 2
    return StepBytes(kv=kv, q_out=q_out, tables=tables, append=append, kv_unique=kv_unique)


def step_bytes_for(step) -> StepBytes:
    """StepBytes of a workloads.DecodeStep."""
    return step_bytes(step.context_lens, step.num_heads, step.num_kv_heads, step.head_dim,
                      step.elem_bytes, step.block_size, step.block_tables, step.act_bytes,
                      step.num_queries, step.window,
                      4 if step.k_row_scales is not None else 0)


def decode_flops(context_lens, num_heads: int, head_dim: int) -> int:
    """2 flops per multiply-add of q.K and p.V for every query head."""
    return int(np.asarray(context_lens, dtype=np.int64).sum()) * num_heads * head_dim * 4


def admissible_requests(budget_blocks: int, blocks_per_request: int,
                        shared_blocks: int = 0) -> int:
    """Requests that fit when each needs blocks_per_request private blocks and
    all share shared_blocks blocks held once."""
    return (budget_blocks - shared_blocks) // blocks_per_request


def budget_blocks(budget_bytes: int, block_bytes: int) -> int:
    return budget_bytes // block_bytes


def ceil_div(a: int, b: int) -> int:
    return -(-a // b) if b else 0


__all__ = ["kv_bytes_per_token", "mla_bytes_per_token", "blocks_for_tokens", "StepBytes",
           "step_bytes", "step_bytes_for", "decode_flops", "admissible_requests",
           "budget_blocks", "ceil_div"]

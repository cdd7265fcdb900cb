"""Pure-Python brute force of the decode step, for tiny inputs only.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``). A second implementation of
the same definition as ``pa_oracle.c``, written with plain Python loops and
floats (IEEE double), so that the two can be checked against each other:

* the slot of a token is block * block_size + offset, and row i of a sequence
  sits in block_table[i // block_size] at offset i % block_size ("MLSys
  Engineer -- Inference Systems Q&A", Q1 "How does PagedAttention work?");
* the step appends, then attends with softmax(scale * K q) . V over every row
  ("LLM inference and serving", the naive incremental decoder);
* query head qh reads KV head qh // (num_heads // num_kv_heads).

Inputs are nested Python lists of floats (already rounded to the cache dtype).
"""
from __future__ import annotations

import math


def append(k_new, v_new, slot_mapping, k_cache, v_cache, block_size):
    """In-place copy of the new rows; k_cache[blk][h][off] = k_new[t][h]."""
    num_slots = len(k_cache) * block_size
    for t, slot in enumerate(slot_mapping):
        if slot < 0 or slot >= num_slots:
            continue
        blk, off = slot // block_size, slot % block_size
        for h in range(len(k_new[t])):
            k_cache[blk][h][off] = list(k_new[t][h])
            v_cache[blk][h][off] = list(v_new[t][h])


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, block_size):
    """out[s][qh][d] = sum_i softmax_i(scale * <q, K_i>) * V_i[d]."""
    num_heads = len(q[0]) if q else 0
    num_kv_heads = len(k_cache[0]) if k_cache else 1
    group = num_heads // num_kv_heads
    out = []
    for s, n in enumerate(context_lens):
        rows = []
        for qh in range(num_heads):
            h = qh // group
            keys, vals = [], []
            for i in range(n):
                blk = block_tables[s][i // block_size]
                keys.append(k_cache[blk][h][i % block_size])
                vals.append(v_cache[blk][h][i % block_size])
            d_model = len(q[s][qh])
            if n == 0:
                rows.append([0.0] * d_model)
                continue
            scores = []
            for key in keys:
                acc = 0.0
                for a, b in zip(q[s][qh], key):
                    acc += a * b
                scores.append(scale * acc)
            top = max(scores)
            ex = [math.exp(x - top) for x in scores]
            z = sum(ex)
            row = [0.0] * d_model
            for e, val in zip(ex, vals):
                for d in range(d_model):
                    row[d] += (e / z) * val[d]
            rows.append(row)
        out.append(rows)
    return out

"""Seeded synthetic inputs for one paged-attention decode step.

This module only draws inputs: random values, sequence lengths, block tables
and slot mappings. It holds none of the attention arithmetic, and both the CUDA
path and the CPU oracle take their inputs from it.

The traffic shape follows "Design an LLM Inference API with GPU Batching"
(clarifying questions: prompts average 1,500 tokens, answers 300, some prompts
reach 100,000) with 16-token blocks ("Batching and the KV Cache"). Five
workloads:

  tiny           fp32, B=4, Hq=4, Hkv=2, d=64, lengths {5, 17, 33, 64}, a 32-block
                 pool handed out in a random permutation
  7b_mha         bf16, B=32, Hq=Hkv=32, d=128, lengths uniform in [512, 2048]
  8b_gqa         bf16, B=128, Hq=32, Hkv=8, d=128, length = prompt + generated,
                 prompt lognormal with mean 1,500 (sigma 0.8) clipped to
                 [16, 8192], generated uniform in [0, 300]
  long_skew      bf16, B=8, Hq=32, Hkv=8, d=128, one 100,000-token sequence and
                 seven of 1,500
  prefix_shared  bf16, 64 samples forked from one 4,096-token prompt (256
                 shared blocks, reference count 64) plus private tails of
                 uniform [0, 300] tokens and the token appended this step
  8b_gqa_fp8     the 8b_gqa batch over an FP8 (e4m3) cache with per-tensor
                 scales 1.0 (uncalibrated); q and the new K/V rows stay bf16
                 and the append quantises them
  8b_gqa_mq2     the 8b_gqa batch with two new tokens per sequence verified
                 together (multi-query decode: each query attends causally)
  8b_gqa_win1024 the 8b_gqa batch under a 1,024-row sliding window (a local
                 attention layer)
  8b_gqa_int8    the 8b_gqa batch over an INT8 cache with one fp32 scale per
                 (row, KV head); q and the new K/V rows stay bf16 and the
                 append quantises them

Every value of q, of the new K/V rows and of the whole pool (used or not) is
drawn N(0, 1) in fp32 and stored in the cache dtype (bf16 by round to nearest
even). An FP8 pool holds e4m3 codes of N(0, 1) draws, made by PyTorch's
float8_e4m3fn conversion; q and the new rows of an FP8 step are bf16. An
INT8 pool holds codes drawn uniformly from [-127, 127] with per-row scales
drawn uniformly from [0.01, 0.03] (values of about unit size). The pool holds 1.25x the blocks the batch needs (the tiny workload: 32)
and hands them out in a seeded random order, so a sequence's blocks are
scattered. Lengths count the token appended by this step: the cache holds
n - 1 rows before the step and n after it. Unused block-table entries hold -1.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

from .block_manager import BlockManager

# Seeds of the five named workloads, in the order listed above.
WORKLOAD_SEEDS = {"tiny": 0, "7b_mha": 1, "8b_gqa": 2, "long_skew": 3, "prefix_shared": 4,
                  "8b_gqa_fp8": 2, "8b_gqa_mq2": 2,
                  "8b_gqa_win1024": 2, "8b_gqa_int8": 2}   # variants of the 8b_gqa batch
PAD_BLOCK = -1


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even.
    Inputs here are finite normals, so no NaN handling is needed."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _torch_e4m3():
    import torch
    return torch, torch.float8_e4m3fn


def to_cache_dtype(x: np.ndarray, cache_dtype: str) -> np.ndarray:
    if cache_dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if cache_dtype == "bf16":
        return round_to_bf16_bits(x)
    if cache_dtype == "fp8":
        torch, e4m3 = _torch_e4m3()
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(e4m3)
        return t.view(torch.uint8).numpy().copy()
    raise ValueError(f"unknown cache dtype {cache_dtype!r}")


def as_f32(x: np.ndarray, cache_dtype: str) -> np.ndarray:
    """Values of a cache-dtype array as fp32 (exact)."""
    if cache_dtype == "bf16":
        return bf16_bits_to_f32(x)
    if cache_dtype == "fp8":
        torch, e4m3 = _torch_e4m3()
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint8)).view(e4m3).float().numpy()
    return np.asarray(x, dtype=np.float32)


_STORAGE = {"f32": np.float32, "bf16": np.uint16, "fp8": np.uint8, "int8": np.int8}
_BYTES = {"f32": 4, "bf16": 2, "fp8": 1, "int8": 1}


_CHUNK = 1 << 22


def _int8_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Codes uniform in [-127, 127], drawn in the same fixed chunks as
    _normal."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.int8)
    root = np.random.SeedSequence(int(rng.integers(0, 2**63 - 1)))
    chunks = list(range(0, n, _CHUNK))
    for i, seed in enumerate(root.spawn(len(chunks))):
        lo = chunks[i]
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = np.random.default_rng(seed).integers(-127, 128, hi - lo, dtype=np.int8)
    return out.reshape(shape)


def _normal(rng: np.random.Generator, shape, cache_dtype: str) -> np.ndarray:
    """N(0,1) fp32 stored in the cache dtype. The array is cut into fixed
    chunks, each drawn from its own child seed of one SeedSequence taken from
    ``rng``, so the values do not depend on how many threads fill them."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=_STORAGE[cache_dtype])
    root = np.random.SeedSequence(int(rng.integers(0, 2**63 - 1)))
    chunks = list(range(0, n, _CHUNK))
    seeds = root.spawn(len(chunks))

    def fill(i: int) -> None:
        lo = chunks[i]
        hi = min(n, lo + _CHUNK)
        vals = np.random.default_rng(seeds[i]).standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi] = to_cache_dtype(vals, cache_dtype)

    if len(chunks) <= 1:
        for i in range(len(chunks)):
            fill(i)
    else:
        workers = min(len(chunks), max(1, os.cpu_count() or 1), 32)
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(len(chunks))))
    return out.reshape(shape)


@dataclass
class DecodeStep:
    """Inputs of one decode step, host side, in the layouts the library takes.

    k_cache / v_cache hold the pool BEFORE the step's append. Applying the
    append (k_new/v_new into slot_mapping) and then attending over
    context_lens tokens per sequence is the step."""
    name: str
    cache_dtype: str                  # "f32", "bf16", "fp8" (e4m3 codes) or "int8" (codes)
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    q: np.ndarray                     # [B][Hq][D]; [B][Q][Hq][D] with Q > 1 queries
    k_new: np.ndarray                 # [B * Q][Hkv][D] (token t = s * Q + j)
    v_new: np.ndarray                 # [B * Q][Hkv][D]
    slot_mapping: np.ndarray          # int64 [B * Q]; -1 = no append
    k_cache: np.ndarray               # [NB][Hkv][bs][D]
    v_cache: np.ndarray               # [NB][Hkv][bs][D]
    block_tables: np.ndarray          # int32 [B][max_blocks]
    context_lens: np.ndarray          # int32 [B]
    scale: float
    seed: int
    meta: dict = field(default_factory=dict)
    act_dtype: str = ""               # dtype of q, out, k_new, v_new ("" = cache_dtype)
    num_queries: int = 1              # new tokens per sequence, the last rows of each
    window: int = 0                   # sliding window: attend to the last `window` rows
    k_row_scales: np.ndarray | None = None   # INT8 caches: fp32 [NB][Hkv][bs], value = scale * code
    v_row_scales: np.ndarray | None = None
    k_scale: float = 1.0              # FP8 caches: value = scale * e4m3(code)
    v_scale: float = 1.0

    def __post_init__(self):
        if not self.act_dtype:
            self.act_dtype = self.cache_dtype

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def elem_bytes(self) -> int:
        """Bytes per cache element."""
        return _BYTES[self.cache_dtype]

    @property
    def act_bytes(self) -> int:
        """Bytes per element of q, out and the new K/V rows."""
        return _BYTES[self.act_dtype]


def build_step(name: str, context_lens, num_heads: int, num_kv_heads: int, head_dim: int,
               cache_dtype: str = "bf16", block_size: int = 16, seed: int = 0,
               pool_factor: float = 1.25, num_blocks: int | None = None,
               scale: float | None = None, rng: np.random.Generator | None = None,
               num_queries: int = 1) -> DecodeStep:
    """A decode step over independent sequences of the given lengths.

    Each sequence is admitted with n - Q tokens and then gets Q appended
    tokens (Q = num_queries, 1 for plain decode); the block manager hands out
    blocks from a seeded permutation of the pool. Length 0 means an idle
    sequence: no blocks, no append."""
    rng = np.random.default_rng(seed) if rng is None else rng
    lens = [int(n) for n in context_lens]
    Q = int(num_queries)
    if any(n < 0 for n in lens) or Q < 1 or any(0 < n < Q for n in lens):
        raise ValueError("context lengths must be 0 or >= the number of queries")
    need = sum(math.ceil(n / block_size) for n in lens)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * need))
    if num_blocks < need:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
    mgr = BlockManager(num_blocks, block_size, free_order=rng.permutation(num_blocks),
                       prefix_caching=False)
    slots = np.full(len(lens) * Q, -1, dtype=np.int64)
    for s, n in enumerate(lens):
        mgr.admit(f"s{s}", [0] * max(n - Q, 0))
        if n > 0:
            for j in range(Q):
                slots[s * Q + j] = mgr.append(f"s{s}", 0).slot
    tables = [mgr.block_table(f"s{s}") for s in range(len(lens))]
    return _materialise(name, cache_dtype, num_heads, num_kv_heads, head_dim, block_size,
                        lens, tables, slots, num_blocks, rng, seed, scale, cow_pairs=[],
                        meta={"pool_factor": pool_factor, "blocks_needed": need},
                        num_queries=Q)


def _materialise(name, cache_dtype, num_heads, num_kv_heads, head_dim, block_size, lens,
                 tables, slots, num_blocks, rng, seed, scale, cow_pairs, meta, num_queries=1):
    if num_heads % num_kv_heads:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    B = len(lens)
    max_blocks = max([len(t) for t in tables] + [1])
    bt = np.full((B, max_blocks), PAD_BLOCK, dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = t
    pool_shape = (num_blocks, num_kv_heads, block_size, head_dim)
    k_rs = v_rs = None
    if cache_dtype == "int8":
        k_cache = _int8_codes(rng, pool_shape)
        v_cache = _int8_codes(rng, pool_shape)
        k_rs = rng.uniform(0.01, 0.03, pool_shape[:3]).astype(np.float32)
        v_rs = rng.uniform(0.01, 0.03, pool_shape[:3]).astype(np.float32)
    else:
        k_cache = _normal(rng, pool_shape, cache_dtype)
        v_cache = _normal(rng, pool_shape, cache_dtype)
    for src, dst in cow_pairs:           # copy-on-write copies made while building
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]
        if k_rs is not None:
            k_rs[dst] = k_rs[src]
            v_rs[dst] = v_rs[src]
    act = "bf16" if cache_dtype in ("fp8", "int8") else cache_dtype
    Q = num_queries
    q = _normal(rng, (B, num_heads, head_dim) if Q == 1 else (B, Q, num_heads, head_dim), act)
    k_new = _normal(rng, (B * Q, num_kv_heads, head_dim), act)
    v_new = _normal(rng, (B * Q, num_kv_heads, head_dim), act)
    used = sorted({b for t in tables for b in t})
    meta = dict(meta, unique_blocks=len(used), max_blocks_per_seq=max_blocks)
    return DecodeStep(name=name, cache_dtype=cache_dtype, num_heads=num_heads,
                      num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                      q=q, k_new=k_new, v_new=v_new, slot_mapping=slots,
                      k_cache=k_cache, v_cache=v_cache, block_tables=bt,
                      context_lens=np.asarray(lens, dtype=np.int32),
                      scale=(1.0 / math.sqrt(head_dim)) if scale is None else float(scale),
                      seed=seed, meta=meta, act_dtype=act, num_queries=Q,
                      k_row_scales=k_rs, v_row_scales=v_rs)


# ---- the five named workloads ------------------------------------------------

def tiny(seed: int = WORKLOAD_SEEDS["tiny"]) -> DecodeStep:
    return build_step("tiny", [5, 17, 33, 64], num_heads=4, num_kv_heads=2, head_dim=64,
                      cache_dtype="f32", seed=seed, num_blocks=32)


def mha_7b(seed: int = WORKLOAD_SEEDS["7b_mha"]) -> DecodeStep:
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 2048, size=32, endpoint=True)
    return build_step("7b_mha", lens, num_heads=32, num_kv_heads=32, head_dim=128,
                      seed=seed, rng=rng)


def gqa_8b_lengths(rng: np.random.Generator, batch: int = 128) -> np.ndarray:
    """prompt ~ lognormal (mean 1,500, sigma 0.8) clipped to [16, 8192], plus
    generated ~ uniform [0, 300]; the sum counts the appended token."""
    sigma = 0.8
    mu = math.log(1500.0) - sigma * sigma / 2.0
    prompt = np.clip(np.rint(rng.lognormal(mu, sigma, size=batch)), 16, 8192).astype(np.int64)
    generated = rng.integers(0, 300, size=batch, endpoint=True)
    return prompt + generated


def gqa_8b(seed: int = WORKLOAD_SEEDS["8b_gqa"], batch: int = 128) -> DecodeStep:
    rng = np.random.default_rng(seed)
    lens = gqa_8b_lengths(rng, batch)
    return build_step("8b_gqa", lens, num_heads=32, num_kv_heads=8, head_dim=128,
                      seed=seed, rng=rng)


def gqa_8b_fp8(seed: int = WORKLOAD_SEEDS["8b_gqa_fp8"], batch: int = 128) -> DecodeStep:
    rng = np.random.default_rng(seed)
    lens = gqa_8b_lengths(rng, batch)
    return build_step("8b_gqa_fp8", lens, num_heads=32, num_kv_heads=8, head_dim=128,
                      cache_dtype="fp8", seed=seed, rng=rng)


def gqa_8b_mq2(seed: int = WORKLOAD_SEEDS["8b_gqa_mq2"], batch: int = 128) -> DecodeStep:
    rng = np.random.default_rng(seed)
    lens = gqa_8b_lengths(rng, batch)
    return build_step("8b_gqa_mq2", lens, num_heads=32, num_kv_heads=8, head_dim=128,
                      seed=seed, rng=rng, num_queries=2)


def gqa_8b_win1024(seed: int = WORKLOAD_SEEDS["8b_gqa_win1024"], batch: int = 128) -> DecodeStep:
    step = gqa_8b(seed, batch)
    step.name = "8b_gqa_win1024"
    step.window = 1024
    return step


def gqa_8b_int8(seed: int = WORKLOAD_SEEDS["8b_gqa_int8"], batch: int = 128) -> DecodeStep:
    rng = np.random.default_rng(seed)
    lens = gqa_8b_lengths(rng, batch)
    return build_step("8b_gqa_int8", lens, num_heads=32, num_kv_heads=8, head_dim=128,
                      cache_dtype="int8", seed=seed, rng=rng)


def long_skew(seed: int = WORKLOAD_SEEDS["long_skew"]) -> DecodeStep:
    return build_step("long_skew", [100_000] + [1_500] * 7, num_heads=32, num_kv_heads=8,
                      head_dim=128, seed=seed)


def prefix_shared(seed: int = WORKLOAD_SEEDS["prefix_shared"], samples: int = 64,
                  prefix: int = 4096, max_tail: int = 300) -> DecodeStep:
    """Parallel samples of one prompt: the prompt's blocks are shared by fork
    (reference count = samples), each sample owns its tail blocks."""
    rng = np.random.default_rng(seed)
    bs = 16
    tails = rng.integers(0, max_tail, size=samples, endpoint=True)
    need = math.ceil(prefix / bs) + sum(math.ceil((prefix + int(t) + 1) / bs) -
                                        prefix // bs for t in tails)
    num_blocks = math.ceil(1.25 * need)
    mgr = BlockManager(num_blocks, bs, free_order=rng.permutation(num_blocks),
                       prefix_caching=False)
    mgr.admit("s0", [0] * prefix)
    for s in range(1, samples):
        mgr.fork("s0", f"s{s}")
    cow_pairs = []
    slots = np.full(samples, -1, dtype=np.int64)
    for s in range(samples):
        for _ in range(int(tails[s])):
            r = mgr.append(f"s{s}", 0)
            if r.copy_on_write:
                cow_pairs.append(r.copy_on_write)
        r = mgr.append(f"s{s}", 0)          # the token this decode step appends
        if r.copy_on_write:
            cow_pairs.append(r.copy_on_write)
        slots[s] = r.slot
    tables = [mgr.block_table(f"s{s}") for s in range(samples)]
    lens = [prefix + int(t) + 1 for t in tails]
    shared = prefix // bs
    refs = [mgr.refcount(b) for b in tables[0][:shared]]
    return _materialise("prefix_shared", "bf16", 32, 8, 128, bs, lens, tables, slots,
                        num_blocks, rng, seed, None, cow_pairs,
                        meta={"prefix": prefix, "shared_blocks": shared,
                              "shared_refcount_min": min(refs) if refs else 0,
                              "blocks_needed": need})


# ---- structured inputs for parity at long contexts ------------------------------

def tile_signs(num_tiles: int, head_dim: int) -> np.ndarray:
    """[num_tiles][head_dim] of +-1: element d of every row of logical tile t
    (16 rows) is (-1)^popcount(t & (d + 1)), a Walsh function of the tile
    index. Tiles 2k and 2k + 1 cancel in every odd-mask column and aligned
    runs of 2^(b+1) tiles cancel in the columns whose mask has lowest bit b,
    so the mean over a whole sequence is small or exactly zero, while one
    missing, repeated or re-weighted tile (or run of tiles) moves it by a
    large multiple of its own size."""
    t = np.arange(num_tiles, dtype=np.int64)[:, None]
    m = np.arange(1, head_dim + 1, dtype=np.int64)[None, :]
    odd = np.bitwise_count(t & m) & 1
    return (1 - 2 * odd).astype(np.int8)


_BF16_ONE, _BF16_MINUS_ONE = np.uint16(0x3F80), np.uint16(0xBF80)


def structured_long(variant: str = "uniform", lens=(100_000,) + (1_500,) * 7,
                    seed: int = WORKLOAD_SEEDS["long_skew"],
                    partition_rows: int = 512) -> DecodeStep:
    """long_skew's shape (bf16, Hq=32, Hkv=8, d=128) with structured K and V
    in every attended row (the rest of the pool stays random):
      V  row i of sequence s, KV head h: (-1)^(s + h) * tile_signs[i // 16]
      K  "uniform": all zero, so every row gets the same softmax weight;
         "weighted": zero except element 0, which is 0.5 * ((5 p + s) mod 4)
         for the rows of chunk p = i // partition_rows, with q's element 0
         set to 8 and its others to 0, so the weight is constant within a
         chunk and differs between chunks (up to e^1.06 apart).
    The step's new rows (k_new, v_new) carry the same pattern for row n - 1."""
    if variant not in ("uniform", "weighted"):
        raise ValueError(f"unknown variant {variant!r}")
    step = build_step(f"structured_{variant}", list(lens), num_heads=32, num_kv_heads=8,
                      head_dim=128, seed=seed)
    bs, D, Hkv, G = step.block_size, step.head_dim, step.num_kv_heads, 32 // 8
    signs_h = np.array([1 if h % 2 == 0 else -1 for h in range(Hkv)], np.int8)
    c_bits = round_to_bf16_bits(np.array([0.0, 0.5, 1.0, 1.5], np.float32))
    if variant == "weighted":
        step.q[...] = 0
        step.q[:, :, 0] = round_to_bf16_bits(np.array([8.0], np.float32))[0]
    for s, n in enumerate(step.context_lens):
        n = int(n)
        if n == 0:
            continue
        nt = (n + bs - 1) // bs
        blocks = step.block_tables[s, :nt]
        sg = tile_signs(nt, D)[:, None, :] * signs_h[None, :, None] * (1 if s % 2 == 0 else -1)
        vbits = np.where(sg > 0, _BF16_ONE, _BF16_MINUS_ONE)          # [nt][Hkv][D]
        step.v_cache[blocks] = vbits[:, :, None, :]
        step.k_cache[blocks] = 0
        last = n - 1
        step.v_new[s] = vbits[last // bs]
        step.k_new[s] = 0
        if variant == "weighted":
            chunk = (np.arange(nt * bs) // partition_rows).reshape(nt, bs)
            cbits = c_bits[(5 * chunk + s) % 4]                         # [nt][bs]
            step.k_cache[blocks, :, :, 0] = cbits[:, None, :]
            step.k_new[s, :, 0] = c_bits[(5 * (last // partition_rows) + s) % 4]
    step.meta = dict(step.meta, structured=variant, partition_rows=partition_rows)
    return step

WORKLOADS = {
    "tiny": tiny,
    "7b_mha": mha_7b,
    "8b_gqa": gqa_8b,
    "long_skew": long_skew,
    "prefix_shared": prefix_shared,
    "8b_gqa_fp8": gqa_8b_fp8,
    "8b_gqa_mq2": gqa_8b_mq2,
    "8b_gqa_win1024": gqa_8b_win1024,
    "8b_gqa_int8": gqa_8b_int8,
}


def make(name: str, seed: int | None = None) -> DecodeStep:
    fn = WORKLOADS[name]
    return fn() if seed is None else fn(seed)

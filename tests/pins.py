"""Pins of the fp64 oracle: checks against facts the pages and the mathematics
fix, not against the oracle itself. Each pin is a plain function that raises
AssertionError on failure, so that test_oracle_pins.py runs them against the
oracle and test_oracle_mutants.py runs them against copies of the oracle with a
planted mistake (at least one pin must catch every such mistake).
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import softmax

import oracle
from oracle import brute
from paged_kv_cache_29_gb300 import workloads as wl
from paged_kv_cache_29_gb300.block_manager import BlockManager


def _f64(step, a):
    return wl.as_f32(a, step.cache_dtype).astype(np.float64)


def _after_append(step):
    k = step.k_cache.copy()
    v = step.v_cache.copy()
    oracle.append(step.k_new, step.v_new, step.slot_mapping, k, v)
    return k, v


def _decode(step, k, v, **kw):
    return oracle.decode(step.q, k, v, step.block_tables, step.context_lens, step.scale, **kw)


def small_step(lens=(5, 17, 33, 64), hq=4, hkv=2, d=16, dtype="f32", bs=16, seed=11,
               num_blocks=None):
    return wl.build_step("pin", list(lens), hq, hkv, d, cache_dtype=dtype, block_size=bs,
                         seed=seed, num_blocks=num_blocks)


# ---- P1: an independent pure-Python implementation on tiny inputs ------------

def pin_brute_force():
    for dtype, hq, hkv, bs, d in [("f32", 4, 2, 16, 8), ("bf16", 6, 3, 4, 8),
                                  ("f32", 2, 2, 1, 4), ("bf16", 8, 1, 16, 8)]:
        step = small_step((1, 7, 16, 23), hq, hkv, d, dtype, bs, seed=3)
        k, v = _after_append(step)
        got = _decode(step, k, v)
        kb, vb = _f64(step, step.k_cache).tolist(), _f64(step, step.v_cache).tolist()
        brute.append(_f64(step, step.k_new).tolist(), _f64(step, step.v_new).tolist(),
                     step.slot_mapping.tolist(), kb, vb, bs)
        want = np.array(brute.decode(_f64(step, step.q).tolist(), kb, vb,
                                     step.block_tables.tolist(), step.context_lens.tolist(),
                                     step.scale, bs))
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# ---- P2: paged == contiguous, the contiguous side through a library softmax --

def pin_paged_equals_contiguous():
    rng = np.random.default_rng(5)
    hq, hkv, d, bs = 6, 2, 12, 4
    G = hq // hkv
    lens = [1, 4, 9, 30]
    nb = 40
    perm = rng.permutation(nb)
    pool_k = rng.standard_normal((nb, hkv, bs, d))
    pool_v = rng.standard_normal((nb, hkv, bs, d))
    q = rng.standard_normal((len(lens), hq, d))
    scale = 0.37
    tables = np.full((len(lens), 8), -1, dtype=np.int32)
    contig = []
    nxt = 0
    for s, n in enumerate(lens):
        nblk = -(-n // bs)
        tables[s, :nblk] = perm[nxt:nxt + nblk]
        nxt += nblk
        K = rng.standard_normal((n, hkv, d))
        V = rng.standard_normal((n, hkv, d))
        idx = np.arange(n)
        pool_k[tables[s, idx // bs], :, idx % bs, :] = K     # scatter into the pool
        pool_v[tables[s, idx // bs], :, idx % bs, :] = V
        contig.append((K, V))
    got = oracle.decode(q.astype(np.float32), pool_k.astype(np.float32),
                        pool_v.astype(np.float32), tables, np.array(lens, np.int32), scale)
    for s, (K, V) in enumerate(contig):
        K32 = K.astype(np.float32).astype(np.float64)
        V32 = V.astype(np.float32).astype(np.float64)
        for qh in range(hq):
            qv = q[s, qh].astype(np.float32).astype(np.float64)
            w = softmax(scale * (K32[:, qh // G, :] @ qv))
            np.testing.assert_allclose(got[s, qh], w @ V32[:, qh // G, :], rtol=0, atol=1e-12)


# ---- P3: permuting physical blocks is invisible -------------------------------

def pin_block_permutation():
    step = small_step(dtype="bf16", seed=21)
    k, v = _after_append(step)
    base = _decode(step, k, v)
    perm = np.random.default_rng(1).permutation(step.num_blocks)
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    bt2 = np.where(step.block_tables >= 0, perm[np.maximum(step.block_tables, 0)], -1)
    got = oracle.decode(step.q, k2, v2, bt2.astype(np.int32), step.context_lens, step.scale)
    assert np.array_equal(got, base), "block permutation changed the result"


# ---- P4: block size 1 and 16 give the same result ----------------------------

def pin_block_size_invariance():
    step = small_step(dtype="f32", seed=8)
    k, v = _after_append(step)
    base = _decode(step, k, v)
    bs = step.block_size
    B = step.num_seqs
    total = int(step.context_lens.sum())
    order = np.random.default_rng(2).permutation(total + 3)
    k1 = np.random.default_rng(3).standard_normal(
        (total + 3, step.num_kv_heads, 1, step.head_dim)).astype(np.float32)
    v1 = k1.copy()
    bt1 = np.full((B, int(step.context_lens.max())), -1, dtype=np.int32)
    nxt = 0
    for s in range(B):
        for i in range(int(step.context_lens[s])):
            blk = order[nxt]
            nxt += 1
            src = step.block_tables[s, i // bs]
            k1[blk, :, 0, :] = k[src, :, i % bs, :]
            v1[blk, :, 0, :] = v[src, :, i % bs, :]
            bt1[s, i] = blk
    got = oracle.decode(step.q, k1, v1, bt1, step.context_lens, step.scale)
    assert np.array_equal(got, base), "block size 1 and 16 disagree"


# ---- P5: weights sum to one; the output is a convex combination ---------------

def pin_softmax_weights_and_hull():
    step = small_step(dtype="bf16", seed=4, hq=4, hkv=1)
    k, v = _after_append(step)
    out = _decode(step, k, v)
    for s in range(step.num_seqs):
        n = int(step.context_lens[s])
        rows = np.array([_f64(step, v[step.block_tables[s, i // 16], 0, i % 16])
                         for i in range(n)])
        for qh in range(step.num_heads):
            w = oracle.attention_weights(step.q, k, step.block_tables, step.context_lens,
                                         step.scale, s, qh)
            assert w.shape == (n,) and np.all(w >= 0)
            assert abs(w.sum() - 1.0) < 1e-12
            np.testing.assert_allclose(out[s, qh], w @ rows, rtol=0, atol=1e-12)
            assert np.all(out[s, qh] <= rows.max(axis=0) + 1e-12)
            assert np.all(out[s, qh] >= rows.min(axis=0) - 1e-12)


# ---- P7: copy-on-write sharing gives the result of private copies ------------

def pin_copy_on_write():
    bs, hkv, hq, d = 16, 2, 4, 8
    rng = np.random.default_rng(9)
    nb = 24
    mgr = BlockManager(nb, bs, free_order=rng.permutation(nb), prefix_caching=False)
    mgr.admit("p", list(range(40)))              # last block holds 8 of 16 slots
    mgr.fork("p", "c")
    k = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    v = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    q = rng.standard_normal((2, hq, d)).astype(np.float32)

    def tables():
        t = [mgr.block_table("p"), mgr.block_table("c")]
        out = np.full((2, 4), -1, np.int32)
        for s, row in enumerate(t):
            out[s, :len(row)] = row
        return out

    lens = np.array([40, 40], np.int32)
    before = oracle.decode(q, k, v, tables(), lens, 0.3)
    res_c = mgr.append("c", 99)                  # child writes into the shared block
    assert res_c.copy_on_write is not None, "a shared partial block must be copied first"
    src, dst = res_c.copy_on_write
    k[dst], v[dst] = k[src], v[src]
    new_k = rng.standard_normal((2, hkv, d)).astype(np.float32)
    new_v = rng.standard_normal((2, hkv, d)).astype(np.float32)
    oracle.append(new_k[1:], new_v[1:], np.array([res_c.slot], np.int64), k, v)
    mid = oracle.decode(q, k, v, tables(), np.array([40, 41], np.int32), 0.3)
    np.testing.assert_array_equal(mid[0], before[0])      # the parent never sees the write
    res_p = mgr.append("p", 77)                  # now the parent appends its own token
    assert res_p.copy_on_write is None and res_p.slot != res_c.slot
    oracle.append(new_k[:1], new_v[:1], np.array([res_p.slot], np.int64), k, v)
    lens2 = np.array([41, 41], np.int32)
    shared = oracle.decode(q, k, v, tables(), lens2, 0.3)
    # Same contents with every block private to its sequence.
    t = tables()
    kp = np.zeros((8, hkv, bs, d), np.float32)
    vp = np.zeros_like(kp)
    priv = np.full_like(t, -1)
    nxt = 0
    for s in range(2):
        for j in range(-(-int(lens2[s]) // bs)):
            kp[nxt], vp[nxt] = k[t[s, j]], v[t[s, j]]
            priv[s, j] = nxt
            nxt += 1
    private = oracle.decode(q, kp, vp, priv, lens2, 0.3)
    np.testing.assert_array_equal(private, shared)
    # and the private layout holds each sequence's own new row
    for s, slot_owner in ((0, new_k[0]), (1, new_k[1])):
        blk = priv[s, 40 // bs]
        np.testing.assert_array_equal(kp[blk, :, 40 % bs, :], slot_owner)


# ---- P7b: the copy-on-write block copy ---------------------------------------

def pin_copy_blocks():
    """After a fork, the child's append copies the shared partial block
    (oracle.copy_blocks) and then writes its row: the child must see the
    parent's 40 rows followed by its own, the parent must see nothing new, and
    no block but the copy's destination may change."""
    bs, hkv, hq, d = 16, 2, 4, 8
    for dtype in ("f32", "bf16"):
        rng = np.random.default_rng(21)
        nb = 24
        mgr = BlockManager(nb, bs, free_order=rng.permutation(nb), prefix_caching=False)
        mgr.admit("p", list(range(40)))          # last block holds 8 of 16 slots
        mgr.fork("p", "c")
        k = wl.to_cache_dtype(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
        v = wl.to_cache_dtype(rng.standard_normal((nb, hkv, bs, d)).astype(np.float32), dtype)
        q = wl.to_cache_dtype(rng.standard_normal((1, hq, d)).astype(np.float32), dtype)
        new_k = wl.to_cache_dtype(rng.standard_normal((1, hkv, d)).astype(np.float32), dtype)
        new_v = wl.to_cache_dtype(rng.standard_normal((1, hkv, d)).astype(np.float32), dtype)
        parent_table = mgr.block_table("p")
        # the parent's 40 rows per KV head, read before anything is written
        rows_k = np.stack([k[parent_table[i // bs], :, i % bs, :] for i in range(40)])
        rows_v = np.stack([v[parent_table[i // bs], :, i % bs, :] for i in range(40)])
        k0, v0 = k.copy(), v.copy()
        res = mgr.append("c", 99)
        assert res.copy_on_write is not None
        src, dst = res.copy_on_write
        assert oracle.copy_blocks(k, v, [[src, dst]]) == 0
        changed = [b for b in range(nb) if not (np.array_equal(k[b], k0[b]) and
                                                np.array_equal(v[b], v0[b]))]
        assert changed == [dst], changed
        oracle.append(new_k, new_v, np.array([res.slot], np.int64), k, v)
        # The child's expected rows in one private block of 41 rows.
        kc = np.concatenate([rows_k, new_k]).transpose(1, 0, 2)[None].copy()
        vc = np.concatenate([rows_v, new_v]).transpose(1, 0, 2)[None].copy()
        table_c = np.array([mgr.block_table("c") + [-1]], np.int32)
        got = oracle.decode(q, k, v, table_c, np.array([41], np.int32), 0.3)
        want = oracle.decode(q, kc, vc, np.zeros((1, 1), np.int32), np.array([41], np.int32), 0.3)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
        table_p = np.array([parent_table + [-1]], np.int32)
        kp = np.stack([rows_k]).transpose(0, 2, 1, 3).copy()
        vp = np.stack([rows_v]).transpose(0, 2, 1, 3).copy()
        got_p = oracle.decode(q, k, v, table_p, np.array([40], np.int32), 0.3)
        want_p = oracle.decode(q, kp, vp, np.zeros((1, 1), np.int32), np.array([40], np.int32), 0.3)
        np.testing.assert_allclose(got_p, want_p, rtol=0, atol=1e-12)
    # Skipped and out-of-range pairs: nothing is written, the latter are counted.
    k1, v1 = k.copy(), v.copy()
    assert oracle.copy_blocks(k1, v1, [[-1, 3], [2, -1], [nb, 1], [0, nb + 5]]) == 2
    assert np.array_equal(k1, k) and np.array_equal(v1, v)


# ---- FP8 (e4m3) cache: the format, the quantising append, the dequantised decode

# Code -> value from the OCP 8-bit e4m3 definition (bias 7, 3 mantissa bits,
# subnormals at exponent 0, 0x7F/0xFF NaN): written out by hand.
E4M3_KNOWN = [(0x00, 0.0), (0x01, 2.0 ** -9), (0x02, 2.0 ** -8), (0x07, 7 * 2.0 ** -9),
              (0x08, 2.0 ** -6), (0x09, 1.125 * 2.0 ** -6), (0x30, 0.5), (0x38, 1.0),
              (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x44, 3.0), (0x50, 8.0),
              (0x78, 256.0), (0x7D, 416.0), (0x7E, 448.0), (0x80, -0.0), (0xB8, -1.0),
              (0xC4, -3.0), (0xFE, -448.0)]


def _e4m3_brute(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code by searching every finite code's value (ties to the
    even code, saturating at +-448): a table search, unlike the oracle's
    binade arithmetic."""
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.int64)
    vals = np.array([dict(E4M3_TABLE)[c] for c in codes])
    out = np.empty(x.shape, dtype=np.uint8)
    for i, xv in enumerate(np.asarray(x, dtype=np.float64).ravel()):
        neg = math.copysign(1.0, xv) < 0
        if abs(xv) >= 448.0:
            out.flat[i] = 0xFE if neg else 0x7E
            continue
        same = codes[(codes >= 0x80) == neg]
        d = np.abs(vals[(codes >= 0x80) == neg] - xv)
        best = np.flatnonzero(d == d.min())
        cand = same[best]
        out.flat[i] = int(cand[0]) if len(cand) == 1 else int([c for c in cand if c % 2 == 0][0])
    return out


def _e4m3_table():
    t = []
    for c in range(256):
        e, m = (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        t.append((c, -mag if c & 0x80 else mag))
    return t


E4M3_TABLE = _e4m3_table()


def pin_e4m3_format():
    table = dict(E4M3_TABLE)
    for code, val in E4M3_KNOWN:
        assert table[code] == val and math.copysign(1, table[code]) == math.copysign(1, val)
    got = oracle.e4m3_decode(np.arange(256))
    for c in range(256):
        if c & 0x7F == 0x7F:
            assert math.isnan(got[c]), c
        else:
            assert got[c] == table[c] and math.copysign(1, got[c]) == math.copysign(1, table[c]), c
    pos = got[:0x7F]
    assert np.all(np.diff(pos) > 0)                       # strictly increasing magnitudes
    np.testing.assert_array_equal(got[0x80:0xFF], -pos)
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F])
    np.testing.assert_array_equal(oracle.e4m3_encode(got[finite].astype(np.float32)), finite)
    rng = np.random.default_rng(8)
    mids = (pos[:-1] + pos[1:]) / 2                       # exact in binary32
    xs = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.uniform(-4, 2.8, 3000),
        mids, -mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
        np.nextafter(mids.astype(np.float32), np.float32(1e9)),
        [440.0, 447.9, 448.0, 455.9, 464.0, 470.0, 479.9, 480.0, 1e6, -1e9, 2.0 ** -10,
         3 * 2.0 ** -11, 1e-30, -1e-30, 0.0, -0.0]]).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(xs), _e4m3_brute(xs))
    assert int(oracle.e4m3_encode(np.array([np.nan], np.float32))[0]) == 0x7F


def pin_fp8_append():
    rng = np.random.default_rng(31)
    nb, hkv, bs, d, T = 6, 2, 4, 16, 5
    for new_dtype in ("bf16", "f32"):
        for k_scale, v_scale in ((1.0, 1.0), (0.37, 3.0), (2.0, 0.5)):
            kn = wl.to_cache_dtype(rng.standard_normal((T, hkv, d)).astype(np.float32) * 3, new_dtype)
            vn = wl.to_cache_dtype(rng.standard_normal((T, hkv, d)).astype(np.float32) * 3, new_dtype)
            kc = rng.integers(0, 256, (nb, hkv, bs, d)).astype(np.uint8)
            vc = rng.integers(0, 256, (nb, hkv, bs, d)).astype(np.uint8)
            slots = np.array([3, -1, 17, 0, nb * bs + 2], np.int64)
            k0, v0 = kc.copy(), vc.copy()
            assert oracle.append_fp8(kn, vn, slots, kc, vc, k_scale, v_scale) == 1
            kx = wl.as_f32(kn, new_dtype) / np.float32(k_scale)     # binary32 division
            vx = wl.as_f32(vn, new_dtype) / np.float32(v_scale)
            for t, slot in enumerate(slots):
                if 0 <= slot < nb * bs:
                    k0[slot // bs, :, slot % bs, :] = _e4m3_brute(kx[t])
                    v0[slot // bs, :, slot % bs, :] = _e4m3_brute(vx[t])
            np.testing.assert_array_equal(kc, k0)
            np.testing.assert_array_equal(vc, v0)


def pin_fp8_decode():
    """Attention over an e4m3 cache equals attention over a binary32 cache
    holding scale * value(code) (exact for power-of-two scales)."""
    rng = np.random.default_rng(41)
    step = small_step((1, 9, 16, 40), hq=8, hkv=2, d=16, dtype="bf16", bs=4, seed=5)
    codes_ok = np.array([c for c, _ in E4M3_TABLE], dtype=np.uint8)
    kc = codes_ok[rng.integers(0, len(codes_ok), step.k_cache.shape)]
    vc = codes_ok[rng.integers(0, len(codes_ok), step.v_cache.shape)]
    vals = dict(E4M3_TABLE)
    for k_scale, v_scale in ((1.0, 1.0), (0.5, 2.0), (0.015625, 8.0)):
        got = oracle.decode_kv(step.q, kc, vc, step.block_tables, step.context_lens,
                               step.scale, k_scale, v_scale)
        kf = (np.vectorize(vals.get)(kc) * k_scale).astype(np.float32)
        vf = (np.vectorize(vals.get)(vc) * v_scale).astype(np.float32)
        qf = wl.as_f32(step.q, "bf16")
        want = oracle.decode(qf, kf, vf, step.block_tables, step.context_lens, step.scale)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# ---- multi-query decode: causal within the new tokens ------------------------

def pin_multi_query():
    """Query j of a sequence with n rows and Q new tokens equals the pinned
    single-query decode of the same sequence cut to its first n - Q + j + 1
    rows; Q = 1 equals decode(); empty sequences give zeros."""
    for Q, dtype in ((3, "bf16"), (1, "f32"), (5, "f32")):
        lens = (0, Q, 9, 16, 40) if Q < 9 else (Q, 40)
        step = wl.build_step("mq", list(lens), 6, 2, 8, cache_dtype=dtype, block_size=4,
                             seed=13 + Q, num_queries=Q)
        k, v = step.k_cache.copy(), step.v_cache.copy()
        oracle.append(step.k_new, step.v_new, step.slot_mapping, k, v)
        q4 = step.q if Q > 1 else step.q[:, None]
        got = oracle.decode_multi(q4, k, v, step.block_tables, step.context_lens, step.scale)
        for s_, n in enumerate(step.context_lens):
            for j in range(Q):
                if n == 0:
                    assert not got[s_, j].any()
                    continue
                want = oracle.decode(q4[s_:s_ + 1, j], k, v, step.block_tables[s_:s_ + 1],
                                     np.array([n - Q + j + 1], np.int32), step.scale)
                np.testing.assert_allclose(got[s_, j], want[0], rtol=0, atol=1e-12)
        if Q == 1:
            np.testing.assert_array_equal(got[:, 0], oracle.decode(step.q, k, v, step.block_tables,
                                                                   step.context_lens, step.scale))
    # a sequence shorter than its query count is an error
    step = wl.build_step("mq", [5], 4, 2, 8, cache_dtype="f32", seed=3, num_queries=2)
    q4 = step.q
    try:
        oracle.decode_multi(q4, step.k_cache, step.v_cache, step.block_tables,
                            np.array([1], np.int32), step.scale)
    except oracle.OracleError:
        pass
    else:
        raise AssertionError("n < Q must be rejected")


# ---- INT8 cache with per-row scales --------------------------------------------

def pin_int8_append():
    """Every appended row's codes reconstruct it within half a step of its
    scale, stay within +-127 and reach 127 in magnitude at the row's largest
    element; an all-zero row gets scale 0 and codes 0; nothing else moves."""
    rng = np.random.default_rng(51)
    nb, hkv, bs, d, T = 6, 2, 4, 16, 6
    for new_dtype in ("f32", "bf16"):
        x = rng.standard_normal((T, 2, hkv, d)).astype(np.float32)
        x *= 10.0 ** rng.uniform(-3, 3, (T, 2, hkv, 1)).astype(np.float32)
        x[2, :, 1] = 0.0                                       # an all-zero row
        kn = wl.to_cache_dtype(x[:, 0], new_dtype)
        vn = wl.to_cache_dtype(x[:, 1], new_dtype)
        kc = rng.integers(-128, 128, (nb, hkv, bs, d)).astype(np.int8)
        vc = rng.integers(-128, 128, (nb, hkv, bs, d)).astype(np.int8)
        ks = rng.uniform(0.1, 1.0, (nb, hkv, bs)).astype(np.float32)
        vs = rng.uniform(0.1, 1.0, (nb, hkv, bs)).astype(np.float32)
        before = [a.copy() for a in (kc, vc, ks, vs)]
        slots = np.array([3, -1, 17, 0, nb * bs + 2, 9], np.int64)
        assert oracle.append_int8(kn, vn, slots, kc, vc, ks, vs) == 1
        written = set()
        for t, slot in enumerate(slots):
            if not 0 <= slot < nb * bs:
                continue
            b, o = slot // bs, slot % bs
            for new, codes, scales in ((kn, kc, ks), (vn, vc, vs)):
                vals = wl.as_f32(new[t], new_dtype).astype(np.float64)
                for h in range(hkv):
                    row, c, sc = vals[h], codes[b, h, o].astype(np.float64), float(scales[b, h, o])
                    written.add((b, h, o))
                    if not row.any():
                        assert sc == 0.0 and not c.any()
                        continue
                    assert np.abs(c).max() <= 127 and np.abs(c[np.argmax(np.abs(row))]) == 127
                    assert np.all(np.abs(row - sc * c) <= sc / 2 * (1 + 1e-6)), (t, h)
        for a, a0 in zip((kc, vc, ks, vs), before):
            for idx in np.ndindex(nb, hkv, bs):
                if idx not in written:
                    np.testing.assert_array_equal(a[idx], a0[idx])


# Rows whose quotients x / scale are exact halves k + 1/2: scale = amax / 127 is
# exact when amax = 127 * 2^-3, 127 * 3 or 127 * 4, and so is every quotient
# below. Expected codes written out by hand under round-half-to-even
# (half-away rounding would give 1, 2, 3, 4, 5, 126, 127, -1, -2, -3, -4, 8,
# 11, 65 in the first row). The rows with power-of-two scales are exact in
# bf16 as well as fp32; 127 * 3 needs 9 significant bits, fp32 only.
INT8_TIE_ROWS = [
    # (values / scale, scale, expected codes, input types)
    ([0.5, 1.5, 2.5, 3.5, 4.5, 125.5, 126.5, -0.5, -1.5, -2.5, -3.5, 7.5, 10.5, 64.5, 127.0,
      0.0], 0.125,
     [0, 2, 2, 4, 4, 126, 126, 0, -2, -2, -4, 8, 10, 64, 127, 0], ("f32", "bf16")),
    ([1.5, 2.5, -2.5, 127.0, 0.5, 3.5, -127.0, 5.5, -5.5, 6.5, 8.5, 9.5, -0.5, 11.5, 12.5,
      13.5], 3.0,
     [2, 2, -2, 127, 0, 4, -127, 6, -6, 6, 8, 10, 0, 12, 12, 14], ("f32",)),
    ([-127.0, 21.5, 22.5, -23.5, 0.5, 1.5, 33.5, 34.5, -99.5, 100.5, 101.5, 0.0, 1.0, -1.0,
      -64.5, 63.5], 4.0,
     [-127, 22, 22, -24, 0, 2, 34, 34, -100, 100, 102, 0, 1, -1, -64, 64], ("f32", "bf16")),
]


def pin_int8_tie_rounding():
    """INT8 codes of exact half-way quotients round to the even neighbour
    ("MLSys Engineer -- Inference Systems Q&A", Q3 gives scale = max|row| / 127
    and rounding to int8; the tie rule is round-half-to-even, the IEEE default),
    for fp32 and bf16 input rows."""
    d = 16
    for new_dtype in ("f32", "bf16"):
        cases = [r for r in INT8_TIE_ROWS if new_dtype in r[3]]
        T = len(cases)
        rows = np.array([[np.float32(q * sc) for q in qs] for qs, sc, _, _ in cases], np.float32)
        assert np.all(rows.astype(np.float64) ==
                      np.array([[q * sc for q in qs] for qs, sc, _, _ in cases]))
        kn = wl.to_cache_dtype(rows[:, None, :], new_dtype)
        vn = wl.to_cache_dtype(-rows[:, None, :], new_dtype)
        assert np.all(wl.as_f32(kn, new_dtype) == rows[:, None, :])   # exact in the input type
        nb, bs = T, 2
        kc = np.zeros((nb, 1, bs, d), np.int8)
        vc = np.zeros_like(kc)
        ks = np.zeros((nb, 1, bs), np.float32)
        vs = np.zeros_like(ks)
        slots = np.array([t * bs + (t % 2) for t in range(T)], np.int64)
        assert oracle.append_int8(kn, vn, slots, kc, vc, ks, vs) == 0
        for t, (qs, sc, want, _) in enumerate(cases):
            b, o = t, t % 2
            assert ks[b, 0, o] == np.float32(sc) and vs[b, 0, o] == np.float32(sc)
            assert kc[b, 0, o].tolist() == want, (new_dtype, kc[b, 0, o].tolist(), want)
            assert vc[b, 0, o].tolist() == [-c for c in want]

def pin_int8_decode():
    """Attention over INT8 codes with per-row scales equals the pure-Python
    brute force over the fp64 values scale * code."""
    rng = np.random.default_rng(52)
    step = small_step((1, 7, 16, 23), hq=4, hkv=2, d=8, dtype="bf16", bs=4, seed=6)
    kc = rng.integers(-127, 128, step.k_cache.shape).astype(np.int8)
    vc = rng.integers(-127, 128, step.v_cache.shape).astype(np.int8)
    ks = rng.uniform(0.005, 0.05, step.k_cache.shape[:3]).astype(np.float32)
    vs = rng.uniform(0.005, 0.05, step.v_cache.shape[:3]).astype(np.float32)
    got = oracle.decode_int8(step.q, kc, vc, ks, vs, step.block_tables, step.context_lens,
                             step.scale)
    kf = (ks[..., None].astype(np.float64) * kc).tolist()
    vf = (vs[..., None].astype(np.float64) * vc).tolist()
    want = np.array(brute.decode(_f64(step, step.q).tolist(), kf, vf, step.block_tables.tolist(),
                                 step.context_lens.tolist(), step.scale, 4))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# ---- sliding window ----------------------------------------------------------

def pin_sliding_window():
    """A window of W rows equals plain attention (scipy's softmax) over the
    last W rows laid out contiguously; W >= n equals decode(); W = 1 returns
    the last V row exactly."""
    for dtype, bs in (("f32", 16), ("bf16", 4)):
        step = small_step((1, 9, 16, 17, 40, 64), hq=6, hkv=3, d=8, dtype=dtype, bs=bs, seed=17)
        k, v = _after_append(step)
        full = oracle.decode(step.q, k, v, step.block_tables, step.context_lens, step.scale)
        np.testing.assert_array_equal(
            oracle.decode_window(step.q, k, v, step.block_tables, step.context_lens,
                                 step.scale, 64), full)
        kf, vf, qf = _f64(step, k), _f64(step, v), _f64(step, step.q)
        G = step.num_heads // step.num_kv_heads
        for W in (1, 5, 16, 17, 33):
            got = oracle.decode_window(step.q, k, v, step.block_tables, step.context_lens,
                                       step.scale, W)
            for s_, n in enumerate(step.context_lens):
                rows = [(step.block_tables[s_, i // bs], i % bs) for i in range(max(0, n - W), n)]
                for qh in range(step.num_heads):
                    h = qh // G
                    K = np.array([kf[b, h, o] for b, o in rows])
                    V = np.array([vf[b, h, o] for b, o in rows])
                    w = softmax(step.scale * (K @ qf[s_, qh]))
                    np.testing.assert_allclose(got[s_, qh], w @ V, rtol=0, atol=1e-12)
                    if W == 1:
                        np.testing.assert_array_equal(got[s_, qh], V[-1])


# ---- P8: closed forms ---------------------------------------------------------

def pin_closed_forms():
    rng = np.random.default_rng(12)
    hkv, hq, d, bs = 2, 4, 16, 16
    nb = 8
    k = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    v = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    q = rng.standard_normal((4, hq, d)).astype(np.float32)
    bt = np.array([[3, -1], [5, 1], [6, 2], [7, 4]], np.int32)
    # one row: the output is that V row exactly
    out = oracle.decode(q, k, v, bt, np.array([1, 0, 0, 0], np.int32), 0.125)
    assert np.array_equal(out[0], v[3, np.arange(hq) // 2, 0, :].astype(np.float64))
    assert np.all(out[1:] == 0.0), "empty sequences give zero rows"
    # equal keys: uniform weights, the output is the mean of the V rows
    k2 = k.copy()
    k2[5] = k2[5, :, :1, :]
    k2[1] = k2[5, :, :1, :]
    out = oracle.decode(q, k2, v, bt, np.array([0, 20, 0, 0], np.int32), 0.125)
    rows = np.concatenate([v[5], v[1, :, :4]], axis=1).astype(np.float64)   # [hkv][20][d]
    for qh in range(hq):
        np.testing.assert_allclose(out[1, qh], rows[qh // 2].mean(axis=0), rtol=0, atol=1e-12)
    # q = 0: uniform weights as well
    out = oracle.decode(np.zeros_like(q), k, v, bt, np.array([0, 0, 29, 0], np.int32), 0.125)
    rows = np.concatenate([v[6], v[2, :, :13]], axis=1).astype(np.float64)
    for qh in range(hq):
        np.testing.assert_allclose(out[2, qh], rows[qh // 2].mean(axis=0), rtol=0, atol=1e-12)
    # one key far ahead of the rest: the output is that key's V row. Both query
    # heads of a group get the same q so that one key can lead for both.
    q3 = q.copy()
    q3[3, 1], q3[3, 3] = q3[3, 0], q3[3, 2]
    k3 = k.copy()
    for h in range(hkv):
        k3[4, h, 9, :] = 1000.0 * np.sign(q3[3, 2 * h])
    out = oracle.decode(q3, k3, v, bt, np.array([0, 0, 0, 26], np.int32), 1.0)
    for qh in range(hq):
        np.testing.assert_array_equal(out[3, qh], v[4, qh // 2, 9].astype(np.float64))


# ---- P9: the split form merges back to the single pass ------------------------

def pin_split_invariance():
    step = small_step((1, 16, 17, 100, 257), hq=4, hkv=2, d=16, dtype="bf16", seed=31)
    k, v = _after_append(step)
    base = _decode(step, k, v)
    for P in (1, 2, 3, 7, 16, 64, 512):
        m, l, o, parts = oracle.decode_partitions(step.q, k, v, step.block_tables,
                                                  step.context_lens, step.scale, P)
        got = oracle.combine_partitions(m, l, o, parts)
        np.testing.assert_allclose(got, base, rtol=0, atol=1e-12)
        assert np.all(parts == -(-step.context_lens // P))


# ---- GQA: G query heads on one KV head == the same KV head repeated G times ----

def pin_gqa_grouping():
    step = small_step(hq=8, hkv=2, d=8, dtype="f32", seed=17)
    k, v = _after_append(step)
    grouped = _decode(step, k, v)
    G = step.num_heads // step.num_kv_heads
    k_rep = np.repeat(k, G, axis=1)              # KV head h -> query heads h*G .. h*G+G-1
    v_rep = np.repeat(v, G, axis=1)
    mha = oracle.decode(step.q, k_rep, v_rep, step.block_tables, step.context_lens,
                        step.scale)
    assert np.array_equal(grouped, mha)


# ---- append: bit copy into the slot, checked by numpy fancy indexing ----------

def pin_append_slots():
    step = small_step(dtype="bf16", d=8, seed=6, bs=4)
    slots = step.slot_mapping.copy()
    slots[1] = -1                                 # padding token: skipped
    k, v = step.k_cache.copy(), step.v_cache.copy()
    bad = oracle.append(step.k_new, step.v_new, slots, k, v)
    assert bad == 0
    ek, ev = step.k_cache.copy(), step.v_cache.copy()
    for t, slot in enumerate(slots):
        if slot >= 0:
            ek[slot // 4, :, slot % 4, :] = step.k_new[t]
            ev[slot // 4, :, slot % 4, :] = step.v_new[t]
    assert np.array_equal(k, ek) and np.array_equal(v, ev)
    over = np.array([step.num_blocks * 4, 0], np.int64)
    assert oracle.append(step.k_new[:2], step.v_new[:2], over, k, v) == 1


# ---- incremental decoding: the cache grows by one row a step ------------------

def pin_incremental_decoder():
    rng = np.random.default_rng(40)
    d, bs, nb = 16, 4, 8
    mgr = BlockManager(nb, bs, free_order=rng.permutation(nb), prefix_caching=False)
    prompt = 4
    k = np.zeros((nb, 1, bs, d), np.float32)
    v = np.zeros_like(k)
    rows_k, rows_v = [], []
    mgr.admit("s", [])
    for step in range(prompt + 6):
        kn = rng.standard_normal((1, 1, d)).astype(np.float32)
        vn = rng.standard_normal((1, 1, d)).astype(np.float32)
        res = mgr.append("s", step)
        oracle.append(kn, vn, np.array([res.slot], np.int64), k, v)
        rows_k.append(kn[0, 0].astype(np.float64))
        rows_v.append(vn[0, 0].astype(np.float64))
        n = mgr.num_tokens("s")
        assert n == step + 1
        qv = rng.standard_normal((1, 1, d)).astype(np.float32)
        bt = np.full((1, 3), -1, np.int32)
        table = mgr.block_table("s")
        bt[0, :len(table)] = table
        out = oracle.decode(qv, k, v, bt, np.array([n], np.int32), 1 / math.sqrt(d))
        w = softmax(np.array(rows_k) @ qv[0, 0].astype(np.float64) / math.sqrt(d))
        np.testing.assert_allclose(out[0, 0], w @ np.array(rows_v), rtol=0, atol=1e-12)
    assert mgr.num_tokens("s") == 10 == prompt + 6


ALL_PINS = [pin_brute_force, pin_paged_equals_contiguous, pin_block_permutation,
            pin_block_size_invariance, pin_softmax_weights_and_hull, pin_copy_on_write,
            pin_copy_blocks, pin_e4m3_format, pin_fp8_append, pin_fp8_decode, pin_multi_query,
            pin_sliding_window, pin_int8_append, pin_int8_tie_rounding, pin_int8_decode,
            pin_closed_forms, pin_split_invariance, pin_gqa_grouping, pin_append_slots,
            pin_incremental_decoder]

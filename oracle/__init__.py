"""fp64 CPU oracle for the paged-attention decode step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import this package. The CUDA library and
its Python binding never import it, and it imports nothing from them.

The arithmetic lives in ``pa_oracle.c`` (plain C, fp64; see its header for the
definition and the passages it follows). This module compiles it with gcc on
first use and wraps it for numpy arrays. ``brute.py`` holds a second,
pure-Python implementation for tiny inputs.

Array conventions (numpy, C-contiguous):
  * fp32 caches are ``np.float32``; bf16 caches are ``np.uint16`` holding the
    raw bf16 bit patterns;
  * q, k_new, v_new, k_cache, v_cache use the cache dtype;
  * block_tables ``int32 [B][max_blocks]``, context_lens ``int32 [B]``,
    slot_mapping ``int64 [T]``;
  * results are ``np.float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpaoracle.so")

_lock = threading.Lock()
_lib = None
_has_openmp = False


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into oracle/_build/libpaoracle.so (OpenMP if gcc has it)."""
    global _has_openmp
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.pao_append.argtypes = [P, P, P, P, P, I, I, I, I, I, I]
        lib.pao_append.restype = I
        lib.pao_copy_blocks.argtypes = [P, P, P, I, I, I, I, I, I]
        lib.pao_copy_blocks.restype = I
        F = ctypes.c_float
        lib.pao_e4m3_decode.argtypes = [I]
        lib.pao_e4m3_decode.restype = D
        lib.pao_e4m3_encode.argtypes = [F]
        lib.pao_e4m3_encode.restype = I
        lib.pao_append_fp8.argtypes = [P, P, I, P, P, P, I, I, I, I, I, F, F]
        lib.pao_append_fp8.restype = I
        lib.pao_decode_kv.argtypes = [P, I, P, P, I, D, D, P, P, D, P, I, I, I, I, I, I, I, I]
        lib.pao_decode_kv.restype = I
        lib.pao_decode_multi.argtypes = [P, I, P, P, I, D, D, P, P, D, P, I, I, I, I, I, I, I, I, I]
        lib.pao_decode_multi.restype = I
        lib.pao_decode_window.argtypes = [P, P, P, P, P, D, I, P, I, I, I, I, I, I, I, I, I]
        lib.pao_decode_window.restype = I
        lib.pao_append_int8.argtypes = [P, P, I, P, P, P, P, P, I, I, I, I, I]
        lib.pao_append_int8.restype = I
        lib.pao_decode_int8.argtypes = [P, I, P, P, P, P, P, P, D, P, I, I, I, I, I, I, I, I]
        lib.pao_decode_int8.restype = I
        lib.pao_decode.argtypes = [P, P, P, P, P, D, P, I, I, I, I, I, I, I, I, I]
        lib.pao_decode.restype = I
        lib.pao_attention_weights.argtypes = [P, P, P, P, D, I, I, P, I, I, I, I, I, I, I, I]
        lib.pao_attention_weights.restype = I
        lib.pao_decode_partitions.argtypes = [P, P, P, P, P, D, I, I, P, P, P,
                                              I, I, I, I, I, I, I, I]
        lib.pao_decode_partitions.restype = I
        lib.pao_combine_partitions.argtypes = [P, P, P, P, I, P, I, I, I]
        lib.pao_combine_partitions.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.uint8:
        return 2
    raise OracleError("cache dtype must be float32, uint16 (bf16 bits) or uint8 (e4m3 codes), "
                      f"got {a.dtype}")


def _c(a: np.ndarray, dtype=None) -> np.ndarray:
    return np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        names = {-1: "invalid argument", -2: "block id outside the pool",
                 -3: "context length outside the block table", -4: "out of memory"}
        raise OracleError(f"{what}: {names.get(rc, rc)}")


def append(k_new, v_new, slot_mapping, k_cache, v_cache) -> int:
    """Copy new K/V rows into their slots, in place. Returns out-of-range slot count."""
    for a in (k_cache, v_cache):
        if not a.flags.c_contiguous:
            raise OracleError("caches must be C-contiguous (they are written in place)")
    nb, hkv, bs, d = k_cache.shape
    k_new, v_new = _c(k_new, k_cache.dtype), _c(v_new, k_cache.dtype)
    slots = _c(slot_mapping, np.int64)
    rc = _load().pao_append(_ptr(k_new), _ptr(v_new), _ptr(slots), _ptr(k_cache),
                            _ptr(v_cache), int(slots.shape[0]), hkv, d, bs, nb,
                            _dtype_code(k_cache))
    if rc < 0:
        _check(rc, "append")
    return rc


def copy_blocks(k_cache, v_cache, block_mapping) -> int:
    """Copy-on-write, in place: block dst := block src of K and V for each
    (src, dst) row of block_mapping (int64 [n][2]), in order. Negative entries
    skip a pair; returns the count of pairs with an entry past the pool."""
    for a in (k_cache, v_cache):
        if not a.flags.c_contiguous:
            raise OracleError("caches must be C-contiguous (they are written in place)")
    nb, hkv, bs, d = k_cache.shape
    mapping = _c(np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2))
    rc = _load().pao_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(mapping),
                                 int(mapping.shape[0]), hkv, d, bs, nb, _dtype_code(k_cache))
    if rc < 0:
        _check(rc, "copy_blocks")
    return rc


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of e4m3 codes (any integer array; NaN for 0x7F/0xFF)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.int64)
    return np.array([lib.pao_e4m3_decode(int(x)) for x in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def e4m3_encode(values) -> np.ndarray:
    """Nearest e4m3 codes (uint8) of binary32 values (ties to even, saturating)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    return np.array([lib.pao_e4m3_encode(float(x)) for x in v.ravel()],
                    dtype=np.uint8).reshape(v.shape)


def append_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale=1.0, v_scale=1.0) -> int:
    """Quantising append into an FP8 cache (uint8 codes, in place): code =
    e4m3(x / scale). k_new/v_new are fp32 or bf16 bits. Returns the
    out-of-range slot count."""
    for a in (k_cache, v_cache):
        if not a.flags.c_contiguous or a.dtype != np.uint8:
            raise OracleError("fp8 caches must be C-contiguous uint8 (written in place)")
    nb, hkv, bs, d = k_cache.shape
    k_new, v_new = _c(k_new), _c(v_new, k_new.dtype)
    slots = _c(slot_mapping, np.int64)
    rc = _load().pao_append_fp8(_ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(slots),
                                _ptr(k_cache), _ptr(v_cache), int(slots.shape[0]), hkv, d, bs,
                                nb, float(k_scale), float(v_scale))
    if rc < 0:
        _check(rc, "append_fp8")
    return rc


def decode_kv(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale=1.0,
              v_scale=1.0, num_threads=0):
    """fp64 decode attention with q and the caches in their own dtypes (the
    caches may be e4m3 codes) and per-tensor K/V scales."""
    q = _c(q)
    k_cache, v_cache = _c(k_cache), _c(v_cache, k_cache.dtype)
    bt, cl = _c(block_tables, np.int32), _c(context_lens, np.int32)
    B, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    out = np.zeros((B, hq, d), dtype=np.float64)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    rc = _load().pao_decode_kv(_ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache),
                               _dtype_code(k_cache), float(k_scale), float(v_scale), _ptr(bt),
                               _ptr(cl), float(scale), _ptr(out), B, hq, hkv, d, bs, nb, mb,
                               int(num_threads))
    _check(rc, "decode_kv")
    return out


def decode_multi(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale=1.0,
                 v_scale=1.0, num_threads=0):
    """Multi-query decode, fp64. q: [B][Q][Hq][D]; query j of sequence s attends
    to rows 0 .. n - Q + j. Returns [B][Q][Hq][D] float64."""
    q = _c(q)
    k_cache, v_cache = _c(k_cache), _c(v_cache, k_cache.dtype)
    bt, cl = _c(block_tables, np.int32), _c(context_lens, np.int32)
    B, Q, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    out = np.zeros((B, Q, hq, d), dtype=np.float64)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    rc = _load().pao_decode_multi(_ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache),
                                  _dtype_code(k_cache), float(k_scale), float(v_scale),
                                  _ptr(bt), _ptr(cl), float(scale), _ptr(out), B, Q, hq, hkv,
                                  d, bs, nb, mb, int(num_threads))
    _check(rc, "decode_multi")
    return out


def decode_window(q, k_cache, v_cache, block_tables, context_lens, scale, window,
                  num_threads=0):
    """fp64 sliding-window decode: each sequence attends to its last `window`
    rows. q: [B][Hq][D] in the cache dtype -> [B][Hq][D] float64."""
    q = _c(q, k_cache.dtype)
    k_cache, v_cache = _c(k_cache), _c(v_cache)
    bt, cl = _c(block_tables, np.int32), _c(context_lens, np.int32)
    B, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    out = np.zeros((B, hq, d), dtype=np.float64)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    rc = _load().pao_decode_window(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl),
                                   float(scale), int(window), _ptr(out), B, hq, hkv, d, bs, nb,
                                   mb, _dtype_code(k_cache), int(num_threads))
    _check(rc, "decode_window")
    return out


def append_int8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scales, v_scales) -> int:
    """Quantising append into an INT8 cache (in place): codes int8
    [NB][Hkv][bs][D], scales float32 [NB][Hkv][bs]; scale = max|row| / 127,
    code = round-half-even(x / scale). Returns the out-of-range slot count."""
    for a, dt in ((k_cache, np.int8), (v_cache, np.int8), (k_scales, np.float32),
                  (v_scales, np.float32)):
        if not a.flags.c_contiguous or a.dtype != dt:
            raise OracleError("INT8 caches and scales must be C-contiguous int8 / float32")
    nb, hkv, bs, d = k_cache.shape
    k_new, v_new = _c(k_new), _c(v_new, k_new.dtype)
    slots = _c(slot_mapping, np.int64)
    rc = _load().pao_append_int8(_ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(slots),
                                 _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
                                 int(slots.shape[0]), hkv, d, bs, nb)
    if rc < 0:
        _check(rc, "append_int8")
    return rc


def decode_int8(q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens, scale,
                num_threads=0):
    """fp64 decode attention over an INT8 cache with per-row scales."""
    q = _c(q)
    k_cache, v_cache = _c(k_cache, np.int8), _c(v_cache, np.int8)
    k_scales, v_scales = _c(k_scales, np.float32), _c(v_scales, np.float32)
    bt, cl = _c(block_tables, np.int32), _c(context_lens, np.int32)
    B, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    out = np.zeros((B, hq, d), dtype=np.float64)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    rc = _load().pao_decode_int8(_ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(k_scales), _ptr(v_scales), _ptr(bt), _ptr(cl), float(scale),
                                 _ptr(out), B, hq, hkv, d, bs, nb, mb, int(num_threads))
    _check(rc, "decode_int8")
    return out


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, num_threads=0):
    """fp64 decode attention. q: [B][Hq][D] in the cache dtype -> [B][Hq][D] float64."""
    q = _c(q, k_cache.dtype)
    k_cache, v_cache = _c(k_cache), _c(v_cache)
    bt, cl = _c(block_tables, np.int32), _c(context_lens, np.int32)
    B, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    out = np.zeros((B, hq, d), dtype=np.float64)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    rc = _load().pao_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl),
                            float(scale), _ptr(out), B, hq, hkv, d, bs, nb, mb,
                            _dtype_code(k_cache), int(num_threads))
    _check(rc, "decode")
    return out


def attention_weights(q, k_cache, block_tables, context_lens, scale, seq, head):
    """Normalised softmax weights of one (seq, query head) over its context."""
    q = _c(q, k_cache.dtype)
    k_cache = _c(k_cache)
    bt, cl = _c(block_tables, np.int32), _c(context_lens, np.int32)
    B, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    w = np.zeros(max(int(cl[seq]), 1), dtype=np.float64)
    rc = _load().pao_attention_weights(_ptr(q), _ptr(k_cache), _ptr(bt), _ptr(cl),
                                       float(scale), int(seq), int(head), _ptr(w), B, hq,
                                       hkv, d, bs, nb, bt.shape[1], _dtype_code(k_cache))
    _check(rc, "attention_weights")
    return w[: int(cl[seq])]


def decode_partitions(q, k_cache, v_cache, block_tables, context_lens, scale,
                      partition_size):
    """Split form: returns (m, l, o, parts) with m/l [B][Hq][P], o [B][Hq][P][D]."""
    q = _c(q, k_cache.dtype)
    k_cache, v_cache = _c(k_cache), _c(v_cache)
    bt, cl = _c(block_tables, np.int32), _c(context_lens, np.int32)
    B, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    parts = ((cl.astype(np.int64) + partition_size - 1) // partition_size).astype(np.int32)
    P = max(int(parts.max()) if B else 0, 1)
    m = np.zeros((B, hq, P), dtype=np.float64)
    l = np.zeros((B, hq, P), dtype=np.float64)
    o = np.zeros((B, hq, P, d), dtype=np.float64)
    rc = _load().pao_decode_partitions(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                       _ptr(cl), float(scale), int(partition_size), P,
                                       _ptr(m), _ptr(l), _ptr(o), B, hq, hkv, d, bs, nb,
                                       bt.shape[1], _dtype_code(k_cache))
    _check(rc, "decode_partitions")
    return m, l, o, parts


def combine_partitions(m, l, o, parts):
    """Merge per-partition (m, l, o) into the normalised output, fp64."""
    m, l, o = _c(m, np.float64), _c(l, np.float64), _c(o, np.float64)
    parts = _c(parts, np.int32)
    B, hq, P, d = o.shape
    out = np.zeros((B, hq, d), dtype=np.float64)
    rc = _load().pao_combine_partitions(_ptr(m), _ptr(l), _ptr(o), _ptr(parts), P,
                                        _ptr(out), B, hq, d)
    _check(rc, "combine_partitions")
    return out


class use_library:
    """Context manager for tests: route this module's calls to another build of
    the oracle (for example a copy with a planted mistake) for its duration."""

    def __init__(self, path: str):
        self.path = path
        self._saved = None

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        lib = ctypes.CDLL(self.path)
        for name in ("pao_append", "pao_copy_blocks", "pao_e4m3_decode", "pao_e4m3_encode",
                     "pao_append_fp8", "pao_decode_kv", "pao_decode_multi", "pao_decode_window",
                     "pao_append_int8", "pao_decode_int8",
                     "pao_decode",
                     "pao_attention_weights",
                     "pao_decode_partitions", "pao_combine_partitions"):
            src = getattr(self._saved, name)
            dst = getattr(lib, name)
            dst.argtypes, dst.restype = src.argtypes, src.restype
        _lib = lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile C source text (a variant of pa_oracle.c) into a shared library."""
    src_path = out_path + ".c"
    with open(src_path, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", out_path, src_path,
                    "-lm"], check=True, capture_output=True, text=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()

"""ctypes binding of libpagedattn.so (include/pagedattn.h).

Argument marshalling only: every function takes torch tensors (or plain
integers), checks that they are CUDA tensors of the expected dtype and shape,
passes their device pointers and the current torch stream to the C entry point
of the same name, and raises PagedAttentionError on a non-OK status. There is
no CPU fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpagedattn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "pagedattn.h")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_CUDA = 4
PA_ERR_DEVICE_BOUNDS = 5

PA_DEVERR_BLOCK_ID = 0x1
PA_DEVERR_SLOT = 0x2
PA_DEVERR_CONTEXT = 0x4
PA_DEVERR_TIMEOUT = 0x8

KERNELS = {"auto": 0, "simt": 1, "mma": 2, "generic": 3, "tc": 4}
DEFAULT_PARTITION = 512

_lock = threading.Lock()
_lib = None


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {pa_status_string(status)} (status {status})")


class _Options(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("partition_size", ctypes.c_int),
                ("long_partition_size", ctypes.c_int), ("long_partition_from", ctypes.c_int)]


def lib() -> ctypes.CDLL:
    """The loaded library. Raises if it has not been built."""
    global _lib
    if _lib is not None:            # loaded: no lock needed to read the reference
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_29_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.pa_reshape_and_cache.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P]
        L.pa_reshape_and_cache.restype = I
        L.pa_reshape_and_cache_fp8.argtypes = [P, P, I, P, P, P, I, I, I, I, I, F, F, P, P]
        L.pa_reshape_and_cache_fp8.restype = I
        L.pa_decode_fp8.argtypes = [P, P, P, P, P, F, F, F, P, I, I, I, I, I, I, I, I, P, S, P, P]
        L.pa_decode_fp8.restype = I
        L.pa_decode_fp8_ex.argtypes = [P, P, P, P, P, F, F, F, P, I, I, I, I, I, I, I, I, P, S, P,
                                       ctypes.POINTER(_Options), P]
        L.pa_decode_fp8_ex.restype = I
        L.pa_test_withhold_tile.argtypes = [P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, I, P, S, P,
                                            I, P]
        L.pa_test_withhold_tile.restype = I
        L.pa_decode_multi.argtypes = [P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, I, I, P, S, P, P]
        L.pa_decode_multi.restype = I
        L.pa_decode_workspace_size_multi.argtypes = [I, I, I, I, I]
        L.pa_decode_workspace_size_multi.restype = S
        L.pa_decode_window.argtypes = [P, P, P, P, P, F, I, P, I, I, I, I, I, I, I, I, I, P, S,
                                       P, P]
        L.pa_decode_window.restype = I
        L.pa_reshape_and_cache_int8.argtypes = [P, P, I, P, P, P, P, P, I, I, I, I, I, P, P]
        L.pa_reshape_and_cache_int8.restype = I
        L.pa_decode_int8.argtypes = [P, P, P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, P, S, P, P]
        L.pa_decode_int8.restype = I
        L.pa_copy_blocks.argtypes = [P, P, P, I, I, I, I, I, I, P, P]
        L.pa_copy_blocks.restype = I
        L.pa_decode.argtypes = [P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, I, P, S, P, P]
        L.pa_decode.restype = I
        L.pa_append_decode.argtypes = [P, P, P, P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, I,
                                       P, S, P, P]
        L.pa_append_decode.restype = I
        L.pa_append_decode_fp8.argtypes = [P, P, P, P, P, F, F, P, P, P, F, P, I, I, I, I, I, I, I,
                                           I, P, S, P, P]
        L.pa_append_decode_fp8.restype = I
        L.pa_append_decode_int8.argtypes = [P, P, P, P, P, P, P, P, P, P, F, P, I, I, I, I, I, I,
                                            I, I, P, S, P, P]
        L.pa_append_decode_int8.restype = I
        L.pa_decode_ex.argtypes = [P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, I, P, S, P,
                                   ctypes.POINTER(_Options), P]
        L.pa_decode_ex.restype = I
        L.pa_decode_noalloc.argtypes = [P, P, P, P, P, F, P, I, I, I, I, I, I, I, I, I, P, P]
        L.pa_decode_noalloc.restype = I
        L.pa_decode_workspace_size.argtypes = [I, I, I, I]
        L.pa_decode_workspace_size.restype = S
        L.pa_decode_workspace_size_ex.argtypes = [I, I, I, I, I]
        L.pa_decode_workspace_size_ex.restype = S
        L.pa_status_string.argtypes = [I]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_check_error_word.argtypes = [ctypes.c_int32]
        L.pa_check_error_word.restype = I
        L.pa_version.argtypes = []
        L.pa_version.restype = I
        L.pa_default_partition_size.argtypes = [I]
        L.pa_default_partition_size.restype = I
        _lib = L
        return L


def declared_functions() -> list[str]:
    """Names of the functions include/pagedattn.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def pa_status_string(status: int) -> str:
    try:
        return lib().pa_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def pa_version() -> int:
    return lib().pa_version()


def pa_default_partition_size(cache_dtype: str) -> int:
    """Rows per split-K partition used when none is requested, for a cache
    of this type ("f32", "bf16", "fp8" or "int8")."""
    codes = {"f32": 0, "bf16": 1, "fp8": 2, "int8": 3}
    if cache_dtype not in codes:
        raise ValueError(f"unknown cache dtype {cache_dtype!r}")
    return lib().pa_default_partition_size(codes[cache_dtype])


def _dtype_code(t) -> int:
    """float32 -> 0, bfloat16 -> 1; an FP8 cache is uint8 (e4m3 codes) or
    torch.float8_e4m3fn -> 2."""
    import torch
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    if t.dtype == torch.uint8 or t.dtype == getattr(torch, "float8_e4m3fn", None):
        return 2
    if t.dtype == torch.int8:
        return 3
    raise TypeError(f"dtype must be float32, bfloat16 or e4m3 codes, got {t.dtype}")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _current_raw_stream():
    """A function returning torch's current CUDA stream handle as an int: the
    raw accessor when this torch has it (no Stream object is built, ~3 us less
    per call), else the public API."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return lambda: raw(torch.cuda.current_device())
    return lambda: torch.cuda.current_stream().cuda_stream


_raw_stream = None


def _stream(stream) -> int | None:
    global _raw_stream
    if stream is None:
        if _raw_stream is None:
            _raw_stream = _current_raw_stream()
        return _raw_stream() or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _check_cuda(name, t, dtype=None, ndim=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")


def _check_device(stream, *tensors):
    """Every tensor (and an explicit torch stream) on torch's current CUDA
    device. The library launches on the current device and takes the SM count,
    the tensor maps, the fixed scratch of pa_decode_noalloc and the default
    stream from it, so a tensor on another GPU would hand that GPU's pointers
    to kernels running here."""
    import torch
    cur = torch.cuda.current_device()
    for t in tensors:
        if t is not None and t.device.index != cur:
            raise ValueError(f"a tensor is on {t.device} but the current CUDA device is cuda:{cur}:"
                             f" run the call under torch.cuda.device({t.device.index})")
    dev = getattr(stream, "device", None)
    if dev is not None and getattr(dev, "index", cur) != cur:
        raise ValueError(f"the stream belongs to {dev} but the current CUDA device is cuda:{cur}")


def pa_reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, error_word=None,
                         stream=None) -> None:
    """Append new K/V rows ([T][Hkv][D]) into their slots of the paged pools
    ([NB][Hkv][bs][D]). slot_mapping: int64 [T], negative = skip."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _check_cuda("k_new", k_new, k_cache.dtype, 3)
    _check_cuda("v_new", v_new, k_cache.dtype, 3)
    _check_cuda("slot_mapping", slot_mapping, torch.int64, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    if tuple(v_cache.shape) != (nb, hkv, bs, d) or tuple(k_new.shape[1:]) != (hkv, d) \
            or k_new.shape != v_new.shape or slot_mapping.shape[0] != k_new.shape[0]:
        raise ValueError("shape mismatch between k_new/v_new/slot_mapping and the caches")
    _check_device(stream, k_new, v_new, slot_mapping, k_cache, v_cache, error_word)
    rc = lib().pa_reshape_and_cache(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                    _ptr(k_cache), _ptr(v_cache), int(k_new.shape[0]), hkv, d,
                                    bs, nb, _dtype_code(k_cache), _ptr(error_word),
                                    _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_reshape_and_cache")


def pa_reshape_and_cache_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale=1.0,
                             v_scale=1.0, error_word=None, stream=None) -> None:
    """Quantising append: k_new/v_new (bf16 or fp32, [T][Hkv][D]) -> e4m3 codes
    of x / scale in the FP8 pools (uint8 [NB][Hkv][bs][D])."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    if _dtype_code(k_cache) != 2:
        raise TypeError("FP8 caches are uint8 (e4m3 codes) or float8_e4m3fn")
    _check_cuda("k_new", k_new, ndim=3)
    _check_cuda("v_new", v_new, k_new.dtype, 3)
    _check_cuda("slot_mapping", slot_mapping, torch.int64, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    if tuple(v_cache.shape) != (nb, hkv, bs, d) or tuple(k_new.shape[1:]) != (hkv, d) \
            or k_new.shape != v_new.shape or slot_mapping.shape[0] != k_new.shape[0]:
        raise ValueError("shape mismatch between k_new/v_new/slot_mapping and the caches")
    _check_device(stream, k_new, v_new, slot_mapping, k_cache, v_cache, error_word)
    rc = lib().pa_reshape_and_cache_fp8(_ptr(k_new), _ptr(v_new), _dtype_code(k_new),
                                        _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                        int(k_new.shape[0]), hkv, d, bs, nb, float(k_scale),
                                        float(v_scale), _ptr(error_word), _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_reshape_and_cache_fp8")


def pa_decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale, out, max_context_len,
                  k_scale=1.0, v_scale=1.0, workspace=None, error_word=None,
                  stream=None, kernel: str = "auto") -> None:
    """Decode attention over FP8 pools (uint8 e4m3 codes) with bf16 q/out.
    kernel: "auto", "mma" (tile ring, mma.sync) or "tc" (tcgen05)."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    if _dtype_code(k_cache) != 2:
        raise TypeError("FP8 caches are uint8 (e4m3 codes) or float8_e4m3fn")
    _check_cuda("q", q, torch.bfloat16, 3)
    _check_cuda("out", out, torch.bfloat16, 3)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape) or tuple(v_cache.shape) != tuple(k_cache.shape) \
            or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("shape mismatch between q/out/block_tables/context_lens and the caches")
    _check_device(stream, q, out, k_cache, v_cache, block_tables, context_lens, error_word,
                  workspace)
    if workspace is None:
        need = pa_decode_workspace_size(B, hq, d, int(max_context_len))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda("workspace", workspace)
    opts = _Options(KERNELS[kernel], 0, 0, 0)
    rc = lib().pa_decode_fp8_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                _ptr(context_lens), float(scale), float(k_scale), float(v_scale),
                                _ptr(out), B, hq, hkv, d, bs, nb, int(block_tables.shape[1]),
                                int(max_context_len), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _ptr(error_word),
                                ctypes.byref(opts), _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_decode_fp8")


def pa_test_withhold_tile(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                          max_context_len, withhold_tile, error_word, workspace=None,
                          stream=None) -> None:
    """Failure test of the bounded waits: a decode call (fp32/bf16 caches, or
    FP8 codes with unit scales) whose CTA 0 withholds tile `withhold_tile` of
    its stream; the waiting consumer gives up after about 2 s and the kernel
    sets PA_DEVERR_TIMEOUT in error_word. Not for production use."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    code = _dtype_code(k_cache)
    act = torch.bfloat16 if code == 2 else k_cache.dtype
    _check_cuda("q", q, act, 3)
    _check_cuda("out", out, act, 3)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape) or tuple(v_cache.shape) != tuple(k_cache.shape) \
            or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("shape mismatch between q/out/block_tables/context_lens and the caches")
    _check_device(stream, q, out, k_cache, v_cache, block_tables, context_lens, error_word,
                  workspace)
    if workspace is None:
        need = pa_decode_workspace_size(B, hq, d, int(max_context_len))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda("workspace", workspace)
    rc = lib().pa_test_withhold_tile(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                     _ptr(context_lens), float(scale), _ptr(out), B, hq, hkv, d,
                                     bs, nb, int(block_tables.shape[1]), int(max_context_len),
                                     code, _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _ptr(error_word), int(withhold_tile), _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_test_withhold_tile")


def pa_decode_workspace_size_multi(num_seqs: int, num_queries: int, num_heads: int,
                                   head_dim: int, max_context_len: int) -> int:
    return int(lib().pa_decode_workspace_size_multi(num_seqs, num_queries, num_heads, head_dim,
                                                     max_context_len))


def pa_decode_multi(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                    max_context_len, workspace=None, error_word=None, stream=None) -> None:
    """Multi-query decode: q/out [B][Q][Hq][D] bf16; query token j of sequence
    s attends to rows 0 .. n - Q + j of its n = context_lens[s] rows."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _check_cuda("q", q, k_cache.dtype, 4)
    _check_cuda("out", out, k_cache.dtype, 4)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, Q, hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape) or tuple(v_cache.shape) != tuple(k_cache.shape) \
            or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("shape mismatch between q/out/block_tables/context_lens and the caches")
    _check_device(stream, q, out, k_cache, v_cache, block_tables, context_lens, error_word,
                  workspace)
    if workspace is None:
        need = pa_decode_workspace_size_multi(B, Q, hq, d, int(max_context_len))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda("workspace", workspace)
    rc = lib().pa_decode_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               _ptr(context_lens), float(scale), _ptr(out), B, Q, hq, hkv, d, bs,
                               nb, int(block_tables.shape[1]), int(max_context_len),
                               _dtype_code(k_cache), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _ptr(error_word),
                               _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_decode_multi")


def pa_decode_window(q, k_cache, v_cache, block_tables, context_lens, scale, window, out,
                     max_context_len, workspace=None, error_word=None, stream=None) -> None:
    """Sliding-window decode: each sequence attends to its last `window` rows."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _check_cuda("q", q, k_cache.dtype, 3)
    _check_cuda("out", out, k_cache.dtype, 3)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape) or tuple(v_cache.shape) != tuple(k_cache.shape) \
            or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("shape mismatch between q/out/block_tables/context_lens and the caches")
    _check_device(stream, q, out, k_cache, v_cache, block_tables, context_lens, error_word,
                  workspace)
    if workspace is None:
        need = pa_decode_workspace_size(B, hq, d, int(max_context_len))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda("workspace", workspace)
    rc = lib().pa_decode_window(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                _ptr(context_lens), float(scale), int(window), _ptr(out), B, hq,
                                hkv, d, bs, nb, int(block_tables.shape[1]), int(max_context_len),
                                _dtype_code(k_cache), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _ptr(error_word),
                                _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_decode_window")


def _check_int8_pool(k_cache, v_cache, k_scales, v_scales):
    import torch
    _check_cuda("k_cache", k_cache, torch.int8, 4)
    _check_cuda("v_cache", v_cache, torch.int8, 4)
    _check_cuda("k_scales", k_scales, torch.float32, 3)
    _check_cuda("v_scales", v_scales, torch.float32, 3)
    if tuple(v_cache.shape) != tuple(k_cache.shape) or \
            tuple(k_scales.shape) != tuple(k_cache.shape[:3]) or \
            tuple(v_scales.shape) != tuple(k_cache.shape[:3]):
        raise ValueError("INT8 pools are [NB][Hkv][bs][D] codes with [NB][Hkv][bs] scales")


def pa_reshape_and_cache_int8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scales, v_scales,
                              error_word=None, stream=None) -> None:
    """Quantising append into an INT8 cache: one fp32 scale per (row, KV head)."""
    import torch
    _check_int8_pool(k_cache, v_cache, k_scales, v_scales)
    _check_cuda("k_new", k_new, ndim=3)
    _check_cuda("v_new", v_new, k_new.dtype, 3)
    _check_cuda("slot_mapping", slot_mapping, torch.int64, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    if tuple(k_new.shape[1:]) != (hkv, d) or k_new.shape != v_new.shape \
            or slot_mapping.shape[0] != k_new.shape[0]:
        raise ValueError("shape mismatch between k_new/v_new/slot_mapping and the caches")
    _check_device(stream, k_new, v_new, slot_mapping, k_cache, v_cache, k_scales, v_scales,
                  error_word)
    rc = lib().pa_reshape_and_cache_int8(_ptr(k_new), _ptr(v_new), _dtype_code(k_new),
                                         _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(k_scales), _ptr(v_scales), int(k_new.shape[0]), hkv,
                                         d, bs, nb, _ptr(error_word), _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_reshape_and_cache_int8")


def pa_decode_int8(q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens, scale,
                   out, max_context_len, workspace=None, error_word=None, stream=None) -> None:
    """Decode attention over an INT8 cache with per-row scales, bf16 q/out."""
    import torch
    _check_int8_pool(k_cache, v_cache, k_scales, v_scales)
    _check_cuda("q", q, torch.bfloat16, 3)
    _check_cuda("out", out, torch.bfloat16, 3)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape) or block_tables.shape[0] != B \
            or context_lens.shape[0] != B:
        raise ValueError("shape mismatch between q/out/block_tables/context_lens and the caches")
    _check_device(stream, q, out, k_cache, v_cache, k_scales, v_scales, block_tables,
                  context_lens, error_word, workspace)
    if workspace is None:
        need = pa_decode_workspace_size(B, hq, d, int(max_context_len))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda("workspace", workspace)
    rc = lib().pa_decode_int8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales),
                              _ptr(v_scales), _ptr(block_tables), _ptr(context_lens),
                              float(scale), _ptr(out), B, hq, hkv, d, bs, nb,
                              int(block_tables.shape[1]), int(max_context_len), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(error_word),
                              _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_decode_int8")


def pa_copy_blocks(k_cache, v_cache, block_mapping, error_word=None, stream=None) -> None:
    """Copy-on-write: block dst := block src of both pools for each (src, dst)
    row of block_mapping (int64 [n][2]); negative entries skip a pair. The
    pools are [NB][Hkv][bs][D]; for an INT8 cache call it again on the row
    scales viewed as [NB][1][1][Hkv * bs]."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _check_cuda("block_mapping", block_mapping, torch.int64, 2)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    if tuple(v_cache.shape) != (nb, hkv, bs, d) or block_mapping.shape[1] != 2:
        raise ValueError("v_cache must match k_cache and block_mapping must be [n][2]")
    _check_device(stream, k_cache, v_cache, block_mapping, error_word)
    rc = lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_mapping),
                              int(block_mapping.shape[0]), hkv, d, bs, nb,
                              _dtype_code(k_cache), _ptr(error_word), _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_copy_blocks")


def pa_decode_workspace_size(num_seqs: int, num_heads: int, head_dim: int,
                             max_context_len: int, partition_size: int = 0) -> int:
    return int(lib().pa_decode_workspace_size_ex(num_seqs, num_heads, head_dim,
                                                 max_context_len, partition_size))


def pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, max_context_len,
              workspace=None, error_word=None, stream=None, kernel: str = "auto",
              partition_size: int = 0, long_partition_size: int = 0,
              long_partition_from: int = 0) -> None:
    """Decode attention for every sequence, written into ``out`` ([B][Hq][D]).

    max_context_len bounds context_lens (host value; sizes the work list and
    the workspace). workspace: a CUDA tensor of at least
    pa_decode_workspace_size(...) bytes; when None, one is allocated from
    torch's caching allocator for this call. long_partition_size /
    long_partition_from: partitions of that many rows for sequences longer
    than long_partition_from rows (0 = one size for all)."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _check_cuda("q", q, k_cache.dtype, 3)
    _check_cuda("out", out, k_cache.dtype, 3)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape) or tuple(v_cache.shape) != tuple(k_cache.shape) \
            or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("shape mismatch between q/out/block_tables/context_lens and the caches")
    _check_device(stream, q, out, k_cache, v_cache, block_tables, context_lens, error_word,
                  workspace)
    if workspace is None:
        # The C library allocates nothing; the binding takes the scratch from
        # torch's allocator for callers that do not manage their own.
        need = pa_decode_workspace_size(B, hq, d, int(max_context_len), int(partition_size))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    opts = _Options(KERNELS[kernel], int(partition_size), int(long_partition_size),
                    int(long_partition_from))
    rc = lib().pa_decode_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                            _ptr(context_lens), float(scale), _ptr(out), B, hq, hkv, d, bs, nb,
                            int(block_tables.shape[1]), int(max_context_len),
                            _dtype_code(k_cache), _ptr(workspace), ws_bytes, _ptr(error_word),
                            ctypes.byref(opts), _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_decode")


def pa_append_decode(k_new, v_new, slot_mapping, k_cache, v_cache, q, block_tables, context_lens,
                     scale, out, max_context_len, workspace=None, error_word=None,
                     stream=None) -> None:
    """One decode step: append one new K/V row per sequence (k_new/v_new
    [B][Hkv][D], slot_mapping int64 [B], the slot of each sequence's last row
    or negative), then decode attention into out ([B][Hq][D])."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _check_cuda("k_new", k_new, k_cache.dtype, 3)
    _check_cuda("v_new", v_new, k_cache.dtype, 3)
    _check_cuda("slot_mapping", slot_mapping, torch.int64, 1)
    _check_cuda("q", q, k_cache.dtype, 3)
    _check_cuda("out", out, k_cache.dtype, 3)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape) or tuple(v_cache.shape) != tuple(k_cache.shape) \
            or tuple(k_new.shape) != (B, hkv, d) or tuple(v_new.shape) != (B, hkv, d) \
            or slot_mapping.shape[0] != B or block_tables.shape[0] != B \
            or context_lens.shape[0] != B:
        raise ValueError("shape mismatch between the step's tensors and the caches")
    _check_device(stream, k_new, v_new, slot_mapping, q, out, k_cache, v_cache, block_tables,
                  context_lens, error_word, workspace)
    if workspace is None:
        need = pa_decode_workspace_size(B, hq, d, int(max_context_len))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pa_append_decode(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache),
                                _ptr(v_cache), _ptr(q), _ptr(block_tables), _ptr(context_lens),
                                float(scale), _ptr(out), B, hq, hkv, d, bs, nb,
                                int(block_tables.shape[1]), int(max_context_len),
                                _dtype_code(k_cache), _ptr(workspace), ws_bytes,
                                _ptr(error_word), _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_append_decode")


def _check_step_rows(k_new, v_new, slot_mapping, q, out, block_tables, context_lens, hkv, d):
    import torch
    _check_cuda("k_new", k_new, torch.bfloat16, 3)
    _check_cuda("v_new", v_new, torch.bfloat16, 3)
    _check_cuda("slot_mapping", slot_mapping, torch.int64, 1)
    _check_cuda("q", q, torch.bfloat16, 3)
    _check_cuda("out", out, torch.bfloat16, 3)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    B, hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape) or tuple(k_new.shape) != (B, hkv, d) \
            or tuple(v_new.shape) != (B, hkv, d) or slot_mapping.shape[0] != B \
            or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("shape mismatch between the step's tensors and the caches")
    return B, hq


def pa_append_decode_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, q, block_tables,
                         context_lens, scale, out, max_context_len, k_scale=1.0, v_scale=1.0,
                         workspace=None, error_word=None, stream=None) -> None:
    """One decode step over FP8 pools: quantise one new bf16 K/V row per
    sequence into its slot (the sequence's last row), then decode."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    if _dtype_code(k_cache) != 2:
        raise TypeError("FP8 caches are uint8 (e4m3 codes) or float8_e4m3fn")
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, hq = _check_step_rows(k_new, v_new, slot_mapping, q, out, block_tables, context_lens, hkv, d)
    _check_device(stream, k_new, v_new, slot_mapping, q, out, k_cache, v_cache, block_tables,
                  context_lens, error_word, workspace)
    if workspace is None:
        need = pa_decode_workspace_size(B, hq, d, int(max_context_len))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda("workspace", workspace)
    rc = lib().pa_append_decode_fp8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache),
                                    _ptr(v_cache), float(k_scale), float(v_scale), _ptr(q),
                                    _ptr(block_tables), _ptr(context_lens), float(scale),
                                    _ptr(out), B, hq, hkv, d, bs, nb, int(block_tables.shape[1]),
                                    int(max_context_len), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _ptr(error_word), _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_append_decode_fp8")


def pa_append_decode_int8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scales, v_scales, q,
                          block_tables, context_lens, scale, out, max_context_len,
                          workspace=None, error_word=None, stream=None) -> None:
    """One decode step over INT8 pools with row scales: quantise one new bf16
    K/V row per sequence into its slot (the sequence's last row), then decode."""
    import torch
    _check_int8_pool(k_cache, v_cache, k_scales, v_scales)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, hq = _check_step_rows(k_new, v_new, slot_mapping, q, out, block_tables, context_lens, hkv, d)
    _check_device(stream, k_new, v_new, slot_mapping, q, out, k_cache, v_cache, k_scales,
                  v_scales, block_tables, context_lens, error_word, workspace)
    if workspace is None:
        need = pa_decode_workspace_size(B, hq, d, int(max_context_len))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda("workspace", workspace)
    rc = lib().pa_append_decode_int8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(k_scales), _ptr(v_scales), _ptr(q),
                                     _ptr(block_tables), _ptr(context_lens), float(scale),
                                     _ptr(out), B, hq, hkv, d, bs, nb, int(block_tables.shape[1]),
                                     int(max_context_len), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _ptr(error_word), _stream(stream))
    if rc != PA_OK:
        raise PagedAttentionError(rc, "pa_append_decode_int8")


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024   # PA_NOALLOC_SCRATCH_BYTES


def pa_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                      max_context_len, error_word=None, stream=None) -> None:
    """pa_decode on the library's fixed device scratch: no workspace argument
    and no allocation. Raises PagedAttentionError (PA_ERR_WORKSPACE) when the
    call needs more than NOALLOC_SCRATCH_BYTES of scratch. Calls that may
    overlap on the GPU share the one scratch and race."""
    import torch
    _check_cuda("k_cache", k_cache, ndim=4)
    _check_cuda("v_cache", v_cache, k_cache.dtype, 4)
    _check_cuda("q", q, k_cache.dtype, 3)
    _check_cuda("out", out, k_cache.dtype, 3)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    if error_word is not None:
        _check_cuda("error_word", error_word, torch.int32)
    nb, hkv, bs, d = k_cache.shape
    B, hq, dq = q.shape
    if dq != d or tuple(out.shape) != tuple(q.shape) or tuple(v_cache.shape) != tuple(k_cache.shape) \
            or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("shape mismatch between q/out/block_tables/context_lens and the caches")
    _check_device(stream, q, out, k_cache, v_cache, block_tables, context_lens, error_word)
    rc = lib().pa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                 _ptr(context_lens), float(scale), _ptr(out), B, hq, hkv, d, bs,
                                 nb, int(block_tables.shape[1]), int(max_context_len),
                                 _dtype_code(k_cache), _ptr(error_word), _stream(stream))
    if rc != PA_OK:
        need = pa_decode_workspace_size(B, hq, d, int(max_context_len))
        what = "pa_decode_noalloc"
        if rc == PA_ERR_WORKSPACE:
            what += (f" (needs {need} bytes of scratch, the fixed scratch holds "
                     f"{NOALLOC_SCRATCH_BYTES}; pass a workspace to pa_decode instead)")
        raise PagedAttentionError(rc, what)

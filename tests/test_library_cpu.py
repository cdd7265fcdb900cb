"""The C-ABI library without a GPU: it builds, loads, exports every function
the header declares, and rejects bad arguments on the host before touching
CUDA."""
import ctypes
import os

import pytest

from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import build as build_mod


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return pa.lib()


def test_exports_every_declared_function(lib):
    names = pa.declared_functions()
    assert {"pa_reshape_and_cache", "pa_decode", "pa_decode_workspace_size",
            "pa_status_string"} <= set(names)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    for code in range(6):
        assert pa.pa_status_string(code)
    assert pa.pa_status_string(99) == "unknown status"
    assert pa.pa_version() >= 10100
    assert lib.pa_check_error_word(0) == pa.PA_OK
    assert lib.pa_check_error_word(pa.PA_DEVERR_SLOT) == pa.PA_ERR_DEVICE_BOUNDS


def test_withhold_hook_argument_checks(lib):
    # Checked on the host before anything is enqueued (no GPU needed).
    P = None
    args = [P, P, P, P, P, 1.0, P, 1, 1, 1, 16, 16, 1, 1, 16, 1, P, 0]   # bf16
    assert lib.pa_test_withhold_tile(*args, P, -1, P) == pa.PA_ERR_INVALID_ARG   # negative tile
    assert lib.pa_test_withhold_tile(*args, P, 3, P) == pa.PA_ERR_INVALID_ARG    # no error word


def test_default_partition_sizes():
    # 512 rows, 1024 of FP8 codes (the same bytes per partition as 512 bf16 rows)
    assert [pa.pa_default_partition_size(d) for d in ("f32", "bf16", "fp8", "int8")] == \
        [512, 512, 1024, 512]
    assert pa.lib().pa_default_partition_size(7) == 0
    with pytest.raises(ValueError):
        pa.pa_default_partition_size("f16")


def _decode(lib, **kw):
    args = dict(q=None, k=None, v=None, bt=None, cl=None, scale=0.1, out=None, B=4, Hq=8,
                Hkv=2, D=128, bs=16, NB=10, mb=4, mcl=64, dtype=1, ws=None, wsb=0, err=None)
    args.update(kw)
    return lib.pa_decode(*args.values(), None)


FAKE = 1 << 20   # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), pa.PA_ERR_INVALID_ARG),                     # heads not a multiple
    (dict(q=None), pa.PA_ERR_INVALID_ARG),                           # null pointers
    (dict(dtype=7), pa.PA_ERR_INVALID_ARG),
    (dict(mcl=65), pa.PA_ERR_INVALID_ARG),                          # past max_blocks * bs
    (dict(B=-1), pa.PA_ERR_INVALID_ARG),
    (dict(D=512), pa.PA_ERR_UNSUPPORTED),
])
def test_decode_rejects_bad_arguments(lib, kw, status):
    ptrs = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, out=FAKE)
    if "q" in kw:
        ptrs["q"] = None
        kw = {}
    assert _decode(lib, **ptrs, **kw) == status


def workspace_formula(B, hq, d, mcl, P=512):
    """The documented workspace layout: a 256-byte header, one 16-byte work
    item per (sequence, head, partition) for at most 4096 sequences, then
    8 + 4 * d bytes of partials per (sequence, head, partition) when a sequence
    can span more than one partition."""
    if B <= 0:
        return 0
    parts = max(1, -(-mcl // P))
    seqs = min(B, 4096)
    units = seqs * hq * parts
    return 256 + 16 * units + ((8 + 4 * d) * units if parts > 1 else 0)


def test_decode_rejects_misaligned_and_missing_workspace(lib):
    ptrs = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, out=FAKE)
    assert _decode(lib, **{**ptrs, "q": FAKE + 8}) == pa.PA_ERR_INVALID_ARG
    assert _decode(lib, **ptrs, mcl=600, mb=40) == pa.PA_ERR_WORKSPACE
    need = lib.pa_decode_workspace_size(4, 8, 128, 600)
    assert need == workspace_formula(4, 8, 128, 600)
    assert _decode(lib, **ptrs, mcl=600, mb=40, ws=FAKE, wsb=need - 4) == pa.PA_ERR_WORKSPACE
    assert _decode(lib, **ptrs, mcl=600, mb=40, ws=FAKE + 8, wsb=need) == pa.PA_ERR_WORKSPACE


def test_empty_batch_is_a_no_op(lib):
    assert _decode(lib, B=0) == pa.PA_OK
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 2, 128, 16, 8, 1, None,
                                    None) == pa.PA_OK


def test_append_rejects_bad_arguments(lib):
    P = FAKE
    assert lib.pa_reshape_and_cache(P, P, P, P, P, 4, 2, 128, 0, 8, 1, None, None) == \
        pa.PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(P, P, P, P, P, 4, 2, 3, 16, 8, 1, None, None) == \
        pa.PA_ERR_UNSUPPORTED                                         # 6-byte rows
    assert lib.pa_reshape_and_cache(None, P, P, P, P, 4, 2, 128, 16, 8, 1, None, None) == \
        pa.PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(P + 4, P, P, P, P, 4, 2, 128, 16, 8, 1, None, None) == \
        pa.PA_ERR_INVALID_ARG


def test_workspace_size_formula(lib):
    for args in [(8, 32, 128, 512), (8, 32, 128, 100_000), (128, 32, 128, 7811), (1, 1, 64, 0),
                 (5000, 8, 64, 1000)]:
        assert lib.pa_decode_workspace_size(*args) == workspace_formula(*args), args
    assert lib.pa_decode_workspace_size(0, 32, 128, 512) == 0
    assert lib.pa_decode_workspace_size_ex(2, 4, 64, 100, 16) == workspace_formula(2, 4, 64, 100, 16)


def test_python_binding_has_no_cpu_fallback():
    """The binding refuses CPU tensors instead of computing anything itself."""
    import torch
    x = torch.zeros(1, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.pa_reshape_and_cache(x, x, torch.zeros(1, dtype=torch.int64),
                                torch.zeros(1, 2, 16, 128, dtype=torch.bfloat16),
                                torch.zeros(1, 2, 16, 128, dtype=torch.bfloat16))


def test_noalloc_rejects_oversize_requests_on_the_host(lib):
    """pa_decode_noalloc refuses a call whose scratch need exceeds its fixed
    scratch before any CUDA call, so this runs without a GPU."""
    too_big = (128, 32, 128, 1 << 20)
    assert lib.pa_decode_workspace_size(*too_big) > pa.NOALLOC_SCRATCH_BYTES
    B, hq, d, mcl = too_big
    rc = lib.pa_decode_noalloc(None, None, None, None, None, 0.1, None, B, hq, 8, d, 16, 1000,
                               mcl // 16, mcl, 1, None, None)
    assert rc == pa.PA_ERR_WORKSPACE
    # The 8B GQA decode batch (128 sequences up to ~8K rows) fits.
    assert lib.pa_decode_workspace_size(128, 32, 128, 8192) <= pa.NOALLOC_SCRATCH_BYTES


def test_fused_step_calls_reject_bad_arguments_on_the_host(lib):
    """pa_append_decode and its FP8/INT8 forms check their extra arguments (the
    new rows, the slots, the scales) before anything is enqueued."""
    P = FAKE
    common = (P, P, P, 0.1, P, 4, 8, 2, 128, 16, 10, 4, 64)   # q .. max_context_len
    tail = (None, 0, None, None)                                # workspace, bytes, error word, stream
    # pa_append_decode(k_new, v_new, slots, k_cache, v_cache, q, tables, lens, scale, out, B, ...)
    ok = dict(k_new=P, v_new=P, slots=P, kc=P, vc=P)

    def fused(dtype=1, **kw):
        a = {**ok, **kw}
        return lib.pa_append_decode(a["k_new"], a["v_new"], a["slots"], a["kc"], a["vc"],
                                    *common, dtype, *tail)
    assert fused(k_new=None) == pa.PA_ERR_INVALID_ARG
    assert fused(slots=P + 4) == pa.PA_ERR_INVALID_ARG       # int64 slots, 8-byte aligned
    assert fused(v_new=P + 8) == pa.PA_ERR_INVALID_ARG       # 16-byte aligned rows
    assert fused(dtype=7) == pa.PA_ERR_INVALID_ARG
    assert fused() == pa.PA_ERR_WORKSPACE                    # valid, but no workspace given
    # pa_append_decode_fp8(..., k_scale, v_scale, q, ...): scales must be finite and > 0
    for ks, vs in [(0.0, 1.0), (1.0, -2.0), (float("inf"), 1.0)]:
        assert lib.pa_append_decode_fp8(P, P, P, P, P, ks, vs, *common, *tail) == \
            pa.PA_ERR_INVALID_ARG
    assert lib.pa_append_decode_fp8(None, P, P, P, P, 1.0, 1.0, *common, *tail) == \
        pa.PA_ERR_INVALID_ARG
    # pa_append_decode_int8(..., k_scales, v_scales, q, ...): the row scales are required
    assert lib.pa_append_decode_int8(P, P, P, P, P, None, P, *common, *tail) == \
        pa.PA_ERR_INVALID_ARG
    assert lib.pa_append_decode_int8(P, P, None, P, P, P, P, *common, *tail) == \
        pa.PA_ERR_INVALID_ARG


def test_c99_program_builds_links_and_runs(lib, tmp_path):
    """The header is plain C99 and the library links into a C program."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not installed")
    here = os.path.dirname(os.path.abspath(__file__))
    lib = pa.LIB_PATH
    exe = str(tmp_path / "abi_check")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(here, "..", "include"), os.path.join(here, "c", "abi_check.c"),
                    "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib),
                    "-Wl,-rpath," + os.path.dirname(lib), "-o", exe], check=True)
    run = subprocess.run([exe], capture_output=True, text=True)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stdout)


class _OnDevice:
    """A stand-in for a CUDA tensor on device `index` (no GPU needed): the
    binding reads only these attributes before it calls the library."""

    def __init__(self, shape, dtype, index):
        import torch
        self._t = torch.empty(shape, dtype=dtype)
        self.shape, self.dtype = self._t.shape, dtype
        self.device = torch.device("cuda", index)
        self.is_cuda = True

    def is_contiguous(self):
        return True

    def dim(self):
        return self._t.dim()

    def numel(self):
        return self._t.numel()

    def element_size(self):
        return self._t.element_size()

    def data_ptr(self):
        return FAKE


def test_binding_refuses_tensors_on_another_device_before_any_call(monkeypatch):
    import torch

    def no_library():
        raise AssertionError("the library was reached")

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(pa, "lib", no_library)
    B, hq, hkv, d, nb, bs = 2, 8, 2, 128, 8, 16

    def tensors(q_dev=0, cache_dev=0, ws_dev=0):
        bf = torch.bfloat16
        return dict(q=_OnDevice((B, hq, d), bf, q_dev),
                    k_cache=_OnDevice((nb, hkv, bs, d), bf, cache_dev),
                    v_cache=_OnDevice((nb, hkv, bs, d), bf, cache_dev),
                    block_tables=_OnDevice((B, 4), torch.int32, 0),
                    context_lens=_OnDevice((B,), torch.int32, 0),
                    out=_OnDevice((B, hq, d), bf, 0),
                    workspace=_OnDevice((4096,), torch.uint8, ws_dev))

    for kw in (dict(q_dev=1), dict(cache_dev=1), dict(ws_dev=1)):
        t = tensors(**kw)
        with pytest.raises(ValueError, match="current CUDA device"):
            pa.pa_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                         t["context_lens"], 0.1, t["out"], 64, workspace=t["workspace"])
    t = tensors(q_dev=1)
    with pytest.raises(ValueError, match="current CUDA device"):
        pa.pa_decode_noalloc(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                             t["context_lens"], 0.1, t["out"], 64)
    k_new = _OnDevice((B, hkv, d), torch.bfloat16, 1)
    slots = _OnDevice((B,), torch.int64, 1)
    t = tensors()
    with pytest.raises(ValueError, match="current CUDA device"):
        pa.pa_reshape_and_cache(k_new, k_new, slots, t["k_cache"], t["v_cache"])
    with pytest.raises(ValueError, match="current CUDA device"):
        pa.pa_copy_blocks(t["k_cache"], t["v_cache"], _OnDevice((3, 2), torch.int64, 1))
    # everything on the current device: the checks pass and the call reaches
    # the library (here the stub)
    t = tensors()
    with pytest.raises(AssertionError, match="library was reached"):
        pa.pa_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                     0.1, t["out"], 64, workspace=t["workspace"])


@pytest.mark.parametrize("long_size,long_from,status", [
    (1024, 2048, None),                  # accepted: fails later only on the fake pointers' workspace
    (500, 2048, pa.PA_ERR_INVALID_ARG),  # not a multiple of 16
    (256, 2048, pa.PA_ERR_INVALID_ARG),  # smaller than the base partition (512)
    (8192, 2048, pa.PA_ERR_INVALID_ARG), # past 4096 rows
    (1024, -5, pa.PA_ERR_INVALID_ARG),   # negative threshold
])
def test_long_partition_options_checked_on_the_host(lib, long_size, long_from, status):
    import ctypes as C
    opts = pa._Options(0, 512, long_size, long_from)
    args = [FAKE] * 5 + [0.1, FAKE, 4, 8, 2, 128, 16, 10, 4, 64, 1, None, 0, None]
    rc = lib.pa_decode_ex(*args, C.byref(opts), None)
    # with a valid option the call gets as far as the (missing) workspace
    assert rc == (pa.PA_ERR_WORKSPACE if status is None else status)

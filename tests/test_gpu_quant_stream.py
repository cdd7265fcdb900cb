"""Work-list edge cases of the FP8 and INT8 decode kernels on the GPU, through
the C ABI. Their producer refills each consumer warp's ring stages from that
warp's own issue stream (block ids double-buffered per item), so these cases
aim at the item bookkeeping: hundreds of one-tile items per CTA (the streams
constantly one item apart), every tile count, CTAs with no item at all, empty
sequences and partition edges, and a bad block id in the middle of a CTA's
stream (flagged, the other sequences still exact)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_parity, from_torch, to_torch
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FORMATS = ["fp8", "int8"]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(fmt, step, tables=None):
    """Decode over the step's caches as they are (no append); returns the
    output (fp64) and the device error word."""
    q = to_torch(step.q, "bf16")
    kc, vc = _dev(step.k_cache), _dev(step.v_cache)
    bt = to_torch(step.block_tables if tables is None else tables)
    lens = to_torch(step.context_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, float("nan"))
    if fmt == "fp8":
        pa.pa_decode_fp8(q, kc, vc, bt, lens, step.scale, out, step.max_context_len,
                         step.k_scale, step.v_scale, error_word=err)
    else:
        pa.pa_decode_int8(q, kc, vc, _dev(step.k_row_scales), _dev(step.v_row_scales), bt, lens,
                          step.scale, out, step.max_context_len, error_word=err)
    torch.cuda.synchronize()
    return wl.as_f32(from_torch(out), "bf16").astype(np.float64), int(err.item())


def _reference(fmt, step):
    if fmt == "fp8":
        return oracle.decode_kv(step.q, step.k_cache, step.v_cache, step.block_tables,
                                step.context_lens, step.scale, step.k_scale, step.v_scale)
    return oracle.decode_int8(step.q, step.k_cache, step.v_cache, step.k_row_scales,
                              step.v_row_scales, step.block_tables, step.context_lens, step.scale)


LENS = {
    # hundreds of one-tile items: every CTA gets several, each one tile per
    # consumer warp at most
    "one_tile_items": [1] * 700 + [17, 33],
    # every tile count from 1 to 100 (rows 16 k + 1: a one-row ragged tail)
    "every_tile_count": [16 * k + 1 for k in range(100)],
    # a single item: nearly every CTA has nothing to do
    "single_item": [17],
    # empty sequences, edges of the 1024-row partitions of 8-bit caches and of
    # 512 rows, and a long sequence
    "empty_and_edges": [0, 9000, 0, 1, 511, 512, 513, 1023, 1024, 1025, 2047, 2049, 0],
}


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("case", sorted(LENS))
def test_work_list_shapes(fmt, case):
    lens = LENS[case]
    step = wl.build_step(f"qs_{case}", lens, 32, 8, 128, cache_dtype=fmt, seed=31)
    got, err = _run(fmt, step)
    want = _reference(fmt, step)
    assert err == 0
    empty = [s for s, n in enumerate(lens) if n == 0]
    assert np.all(got[empty] == 0.0)
    assert_parity(got, want, "bf16")


@pytest.mark.parametrize("fmt", FORMATS)
def test_bad_block_id_mid_stream_is_flagged(fmt):
    lens = [40, 1300, 33, 700, 5000, 16]
    step = wl.build_step("qs_bad", lens, 32, 8, 128, cache_dtype=fmt, seed=32)
    want = _reference(fmt, step)
    bad = step.block_tables.copy()
    bad[1, 40] = step.num_blocks + 3           # a full partition of sequence 1: outside the pool
    bad[4, 300] = -2                           # the last partition of sequence 4
    got, err = _run(fmt, step, tables=bad)
    assert err & pa.PA_DEVERR_BLOCK_ID
    ok = [0, 2, 3, 5]
    assert_parity(got[ok], want[ok], "bf16")
    # The next call on a clean table is exact again (no state carried over).
    got, err = _run(fmt, step)
    assert err == 0
    assert_parity(got, want, "bf16")


@pytest.mark.parametrize("mcl", [0, 16])
def test_all_empty_batch(mcl):
    """No sequence has a row: the plan yields no work item at all; every output
    row is zero and nothing is flagged, for every kernel family (max_context_len
    0, or an upper bound no sequence reaches)."""
    from gpu_helpers import DeviceStep
    lens = [0] * 5
    step = wl.build_step("all_empty", lens, 8, 2, 128, cache_dtype="bf16", seed=33)
    for kernel in ["mma", "simt", "generic"]:
        dev = DeviceStep(step)
        dev.out.fill_(7.0)
        dev.decode(kernel, max_context_len=mcl)
        torch.cuda.synchronize()
        assert dev.error_word() == 0, kernel
        assert np.all(dev.result() == 0.0), kernel
    for fmt in FORMATS:
        st = wl.build_step(f"all_empty_{fmt}", lens, 32, 8, 128, cache_dtype=fmt, seed=34)
        q = to_torch(st.q, "bf16")
        kc, vc = _dev(st.k_cache), _dev(st.v_cache)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full_like(q, 7.0)
        if fmt == "fp8":
            pa.pa_decode_fp8(q, kc, vc, to_torch(st.block_tables), to_torch(st.context_lens),
                             st.scale, out, mcl, 1.0, 1.0, error_word=err)
        else:
            pa.pa_decode_int8(q, kc, vc, _dev(st.k_row_scales), _dev(st.v_row_scales),
                              to_torch(st.block_tables), to_torch(st.context_lens), st.scale,
                              out, mcl, error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, fmt
        assert torch.all(out == 0).item(), fmt


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("bs", [32, 64])
def test_larger_blocks(fmt, bs):
    """Blocks of 32 and 64 rows: several tiles per block (and, for INT8, the
    row scales of each tile inside the block's scale rows)."""
    lens = [1, 31, 32, 33, 64, 65, 700, 2100]
    step = wl.build_step(f"qs_bs{bs}", lens, 32, 8, 128, cache_dtype=fmt, block_size=bs,
                         seed=35 + bs)
    got, err = _run(fmt, step)
    assert err == 0
    assert_parity(got, _reference(fmt, step), "bf16")

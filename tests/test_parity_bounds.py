"""The output-scaled parity bounds (tests/parity.py) on the CPU: they accept
the oracle's own result rounded to the output type, and they reject oracle
results computed as a faulty kernel would compute them, with one 16-row tile
dropped or read twice, or one 512-row partition counted twice (its weight
doubled in the softmax). No GPU: the faults are made by editing the block
table handed to the oracle, so the "faulty" result is exactly what a kernel
with that fault would produce ("MLSys Engineer -- Inference Systems Q&A", Q1:
row i is row i % 16 of block block_table[i / 16]; Q4: the online softmax
merges partial results by their maxima and sums)."""
import numpy as np
import pytest

import oracle
from parity import assert_elements, element_violation, scaled_violation, ulp
from paged_kv_cache_29_gb300 import workloads as wl

BS = 16


def _round_bf16(x):
    return wl.as_f32(wl.to_cache_dtype(np.asarray(x, np.float32), "bf16"), "bf16").astype(
        np.float64)


def _appended(step):
    k, v = step.k_cache.copy(), step.v_cache.copy()
    oracle.append(step.k_new, step.v_new, step.slot_mapping, k, v)
    return k, v


def _decode_one(step, k, v, s, table, n):
    bt = np.full((1, max(len(table), 1)), -1, np.int32)
    bt[0, :len(table)] = table
    return oracle.decode(step.q[s:s + 1], k, v, bt, np.array([n], np.int32), step.scale)


def _doctored(step, k, v, s, fault, where):
    """Oracle output of sequence s as a kernel with `fault` at tile (or
    partition) `where` would compute it."""
    n = int(step.context_lens[s])
    nt = (n + BS - 1) // BS
    table = list(step.block_tables[s, :nt])
    tail = n - (nt - 1) * BS                       # rows in the last tile
    rows_of = (lambda t: tail if t == nt - 1 else BS)
    if fault == "drop_tile":
        new = table[:where] + table[where + 1:]    # later tiles move up, keeping their rows
        n2 = n - rows_of(where)
    elif fault == "repeat_tile":
        assert where != nt - 1
        new = table[:where + 1] + [table[where]] + table[where + 1:]
        n2 = n + BS
    elif fault == "double_partition":
        lo, hi = 32 * where, 32 * (where + 1)
        assert hi < nt
        new = table[:hi] + table[lo:hi] + table[hi:]
        n2 = n + 512
    else:
        raise ValueError(fault)
    return _decode_one(step, k, v, s, new, n2)


@pytest.fixture(scope="module")
def random_steps():
    """Random N(0,1) inputs of 1,500 and 8,000 rows (the 8b_gqa lengths'
    mean and upper end); the 100,000-row case uses the structured inputs."""
    return {n: wl.build_step("bounds", [n], 32, 8, 128, seed=n) for n in (1500, 8000)}


def test_row_bound_accepts_the_rounded_oracle(random_steps):
    for step in random_steps.values():
        k, v = _appended(step)
        want = oracle.decode(step.q, k, v, step.block_tables, step.context_lens, step.scale)
        ratio, _ = scaled_violation(_round_bf16(want), want, "bf16")
        assert ratio <= 0.25          # half an ulp of the element <= a quarter of 2 row ulps
        ratio, _ = scaled_violation(want.astype(np.float32).astype(np.float64), want, "f32")
        assert ratio <= 0.25


@pytest.mark.parametrize("fault", ["drop_tile", "repeat_tile"])
def test_row_bound_rejects_tile_faults_on_random_inputs(random_steps, fault):
    for n, step in random_steps.items():
        k, v = _appended(step)
        want = _decode_one(step, k, v, 0, list(step.block_tables[0, :(n + 15) // 16]), n)
        nt = (n + BS - 1) // BS
        for t in (0, nt // 3, nt - 2):
            bad = _doctored(step, k, v, 0, fault, t)
            ratio, _ = scaled_violation(_round_bf16(bad), want, "bf16")
            assert ratio > 1.0, (n, fault, t, ratio)


def test_row_bound_rejects_a_doubled_partition_on_random_inputs(random_steps):
    step = random_steps[8000]
    k, v = _appended(step)
    want = _decode_one(step, k, v, 0, list(step.block_tables[0, :500]), 8000)
    for p in (0, 7, 14):
        bad = _doctored(step, k, v, 0, "double_partition", p)
        assert scaled_violation(_round_bf16(bad), want, "bf16")[0] > 1.0, p


def test_row_bound_rejects_zeros_and_a_scaled_output(random_steps):
    step = random_steps[8000]
    k, v = _appended(step)
    want = oracle.decode(step.q, k, v, step.block_tables, step.context_lens, step.scale)
    assert scaled_violation(np.zeros_like(want), want, "bf16")[0] > 1.0
    assert scaled_violation(_round_bf16(want * 1.02), want, "bf16")[0] > 1.0


@pytest.fixture(scope="module", params=["uniform", "weighted"])
def structured(request):
    step = wl.structured_long(request.param, lens=(100_000,))
    k, v = _appended(step)
    n = int(step.context_lens[0])
    want = _decode_one(step, k, v, 0, list(step.block_tables[0, :(n + 15) // 16]), n)
    return step, k, v, want


# The element bound the structured GPU test uses (tests/test_gpu_parity.py).
STRUCT_ULPS, STRUCT_REL = 1.0, 2.0 ** -16


def test_structured_inputs_reach_exact_zeros(structured):
    step, _, _, want = structured
    # the odd-mask columns cancel pairwise over the sequence's 6,250 tiles
    # (zero up to the fp64 summation's rounding)
    assert np.all(np.abs(want[0, :, 0::2]) < 1e-12)
    assert element_violation(_round_bf16(want), want, "bf16", STRUCT_ULPS, STRUCT_REL)[0] <= 0.5


@pytest.mark.parametrize("fault,where", [("drop_tile", 0), ("drop_tile", 3125),
                                         ("drop_tile", 6248), ("drop_tile", 6249),
                                         ("repeat_tile", 0), ("repeat_tile", 4095),
                                         ("double_partition", 0), ("double_partition", 97),
                                         ("double_partition", 194)])
def test_element_bound_rejects_structured_faults(structured, fault, where):
    step, k, v, want = structured
    bad = _round_bf16(_doctored(step, k, v, 0, fault, where))
    ratio, _ = element_violation(bad, want, "bf16", STRUCT_ULPS, STRUCT_REL)
    assert ratio > 1.0, (fault, where, ratio)
    with pytest.raises(AssertionError):
        assert_elements(bad, want, "bf16", STRUCT_ULPS, STRUCT_REL)


def test_ulp_spacing():
    # bf16 spacing: 2^-7 at 1, 2^-14 at 0.01 (2^-7 <= 0.01 < 2^-6), 0 at 0
    np.testing.assert_array_equal(ulp(np.array([1.0, 1.5, 0.01, 0.0, -3.0]), 7),
                                  [2.0 ** -7, 2.0 ** -7, 2.0 ** -14, 0.0, 2.0 ** -6])

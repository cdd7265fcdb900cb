"""Output-scaled parity bounds (pure numpy, no GPU).

The contract's absolute bars (max-abs 2e-2 for bf16 outputs, 1e-4 for fp32)
are larger than the output itself on long contexts: with unit-variance K, V
and q the attention output of an n-row sequence shrinks like 1/sqrt(n)
(about 0.016 at 100,000 rows), so an absolute bar alone would pass a kernel
that dropped a tile or wrote zeros. These bounds scale with the output.

Row bound (`row_bounds`): for each output row r (one sequence, query token and
query head; the last axis is the head dimension),

    max_d |got[r, d] - want[r, d]|  <=  C * ulp(max_d |want[r, d]|)

with ulp(x) = 2^(floor(log2 x) - p) the spacing of the output type at x (p = 7
for bf16, 23 for fp32). Where the error comes from, for a bf16 output:
  - the final rounding of each element to bf16: at most half an ulp of that
    element, so at most half an ulp of the row maximum;
  - the probabilities rounded to the 16-bit MMA operand type before the P.V
    product (bf16 or f16, relative error at most 2^-9 resp. 2^-12 each): with
    independent rounding errors the effect on an element is about
    2^-9 / sqrt(3) * sqrt(sum_i w_i^2 v_id^2), which for the workloads' N(0,1)
    V is well below one ulp of the row maximum (the row maximum is a few times
    sqrt(sum_i w_i^2), the elementwise error a few parts in a thousand of it);
  - fp32 accumulation of the scores, the online-softmax rescales, the split-K
    merge and the approximate exp2: relative errors of order 1e-6, far below
    an ulp of bf16.
C = 2 bf16 ulps covers these with margin. For fp32 outputs the same terms are
all of order 2^-20 relative; the bound is C = 2 ulps of a 16-bit significand
(2^(floor(log2 x) - 15)), about 3e-5 of the row maximum.

Element bound (`element_bounds`), for structured inputs whose exact result is
reachable in fp32 (many elements exactly zero by cancellation):

    |got - want| <= ulps * ulp(|want|) + rel * max_d |want[r, d]|

elementwise, so that an element the oracle gives as 0 must come out as (nearly)
0 whatever the size of the rest of its row.
"""
from __future__ import annotations

import numpy as np

# significand bits after the leading one
_P = {"bf16": 7, "f32": 23}
# row-bound ulps and the precision they are counted in
_ROW = {"bf16": (2.0, 7), "f32": (2.0, 15)}


def ulp(x: np.ndarray, p: int) -> np.ndarray:
    """Spacing 2^(floor(log2 |x|) - p) of a p-bit-significand format at |x|
    (0 where x is 0)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - p).astype(np.int64)), 0.0)


def _rows(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return a.reshape(-1, a.shape[-1]) if a.ndim else a.reshape(1, 1)


def row_bounds(want: np.ndarray, out_dtype: str) -> np.ndarray:
    """Per-row tolerance C * ulp(max_d |want|) (see the module docstring)."""
    c, p = _ROW[out_dtype]
    return c * ulp(np.abs(_rows(want)).max(axis=1), p)


def scaled_violation(got: np.ndarray, want: np.ndarray, out_dtype: str):
    """(worst ratio of a row's max-abs error to its bound, that row's index).
    A ratio above 1 is a violation; a row whose bound is 0 (an all-zero
    oracle row) must match exactly (ratio inf otherwise)."""
    g, w = _rows(got), _rows(want)
    if g.shape != w.shape:
        raise ValueError(f"shape mismatch {g.shape} vs {w.shape}")
    if g.size == 0:
        return 0.0, -1
    err = np.abs(g - w).max(axis=1)
    bound = row_bounds(want, out_dtype)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                         np.where(err > 0, np.inf, 0.0))
    ratio = np.where(np.isnan(err), np.inf, ratio)
    i = int(np.argmax(ratio))
    return float(ratio[i]), i


def assert_scaled(got: np.ndarray, want: np.ndarray, out_dtype: str, what: str = "") -> None:
    ratio, row = scaled_violation(got, want, out_dtype)
    assert ratio <= 1.0, (f"{what}: row {row} error is {ratio:.3g}x its output-scaled bound "
                          f"({row_bounds(want, out_dtype)[row]:.3g})")


def element_violation(got: np.ndarray, want: np.ndarray, out_dtype: str, ulps: float = 1.0,
                      rel: float = 0.0):
    """(worst ratio of an element's error to its element bound, flat index)."""
    g, w = _rows(got), _rows(want)
    if g.shape != w.shape:
        raise ValueError(f"shape mismatch {g.shape} vs {w.shape}")
    if g.size == 0:
        return 0.0, -1
    bound = ulps * ulp(w, _P[out_dtype]) + rel * np.abs(w).max(axis=1, keepdims=True)
    err = np.abs(g - w)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                         np.where(err > 0, np.inf, 0.0))
    ratio = np.where(np.isnan(err), np.inf, ratio)
    i = int(np.argmax(ratio))
    return float(ratio.flat[i]), i


def assert_elements(got, want, out_dtype, ulps=1.0, rel=0.0, what=""):
    ratio, i = element_violation(got, want, out_dtype, ulps, rel)
    assert ratio <= 1.0, f"{what}: element {i} error is {ratio:.3g}x its bound"

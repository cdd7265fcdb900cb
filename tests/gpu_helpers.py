"""Shared helpers of the GPU tests: upload a workloads.DecodeStep, run the
C-ABI path on it, and run the oracle on the same rounded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from parity import assert_scaled
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

TOL = {"f32": 1e-4, "bf16": 2e-2}     # max-abs against the fp64 oracle


def to_torch(a: np.ndarray, cache_dtype: str | None = None, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if cache_dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(device)


def from_torch(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class DeviceStep:
    """A DecodeStep resident on the GPU."""

    def __init__(self, step: wl.DecodeStep, partition_size: int = 0):
        self.step = step
        cd = step.cache_dtype
        self.q = to_torch(step.q, cd)
        self.k_new = to_torch(step.k_new, cd)
        self.v_new = to_torch(step.v_new, cd)
        self.k_cache = to_torch(step.k_cache, cd)
        self.v_cache = to_torch(step.v_cache, cd)
        self.slots = to_torch(step.slot_mapping)
        self.tables = to_torch(step.block_tables)
        self.lens = to_torch(step.context_lens)
        self.out = torch.empty_like(self.q)
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.partition_size = partition_size
        ws = pa.pa_decode_workspace_size(step.num_seqs, step.num_heads, step.head_dim,
                                         max(step.max_context_len, 0), partition_size)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device="cuda")

    def append(self):
        pa.pa_reshape_and_cache(self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache,
                                error_word=self.err)

    def decode(self, kernel="auto", max_context_len=None):
        mcl = self.step.max_context_len if max_context_len is None else max_context_len
        pa.pa_decode(self.q, self.k_cache, self.v_cache, self.tables, self.lens, self.step.scale,
                     self.out, mcl, workspace=self.workspace, error_word=self.err,
                     kernel=kernel, partition_size=self.partition_size)

    def run(self, kernel="auto"):
        self.append()
        self.decode(kernel)
        torch.cuda.synchronize()
        return self.result()

    def result(self) -> np.ndarray:
        return wl.as_f32(from_torch(self.out), self.step.cache_dtype).astype(np.float64)

    def error_word(self) -> int:
        return int(self.err.item())


def oracle_reference(step: wl.DecodeStep):
    """(appended k pool, appended v pool, fp64 output) from the oracle."""
    k = step.k_cache.copy()
    v = step.v_cache.copy()
    oracle.append(step.k_new, step.v_new, step.slot_mapping, k, v)
    out = oracle.decode(step.q, k, v, step.block_tables, step.context_lens, step.scale)
    return k, v, out


def max_abs(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def assert_parity(got: np.ndarray, want: np.ndarray, dtype: str, what="") -> None:
    """Both parity bars against the oracle: the contract's absolute max-abs
    (1e-4 for fp32 outputs, 2e-2 for bf16) and the output-scaled row bound of
    tests/parity.py (2 ulps of each output row's largest element), which
    still resolves errors where outputs are small (long contexts)."""
    err = max_abs(got, want)
    assert err <= TOL[dtype], f"{what}: max-abs {err} > {TOL[dtype]}"
    assert_scaled(got, want, dtype, str(what))

"""The decode kernel's in-kernel plan, read back from the workspace: after a
call, the work list (int4 (sequence, KV head, partition, length) per item at
byte 256 of the workspace) holds every (sequence, KV head, partition) once, in
the documented order: full partitions by sequence, partition and KV head, then
the partial last partitions from largest to smallest in 16 size classes
(ties by sequence, then KV head). Empty sequences have no item."""
import numpy as np
import pytest
import torch

from gpu_helpers import to_torch
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

BUCKETS = 16


def expected_items(lens, hkv, rows_of, base):
    """rows_of(n): rows per partition of an n-row sequence; base: the
    partition size of short sequences. Full partitions of sequences with
    larger partitions come first, then the other full partitions, then the
    partial last partitions by size bucket (relative to base; larger ones in
    bucket 0)."""
    long_full, full, partial = [], [], []
    for s, n in enumerate(lens):
        if n <= 0:
            continue
        P = rows_of(n)
        nf, r = divmod(n, P)
        for part in range(nf):
            for h in range(hkv):
                (long_full if P != base else full).append((s, h, part, n))
        if r:
            b = min(BUCKETS - 1, max(0, (base - r) * BUCKETS // base))
            partial.append((b, s, nf, n))
    partial.sort(key=lambda t: (t[0], t[1]))          # stable: by class, then sequence
    items = long_full + full
    for _, s, part, n in partial:
        for h in range(hkv):
            items.append((s, h, part, n))
    return np.array(items, dtype=np.int32).reshape(-1, 4)


@pytest.mark.parametrize("fmt,P,long_p,long_from", [
    ("bf16", 512, 0, 0), ("bf16", 64, 0, 0), ("fp8", 0, 0, 0),
    ("bf16", 512, 1024, 2048), ("bf16", 256, 2048, 5000)])
def test_work_list_order(fmt, P, long_p, long_from):
    """P = 0: the cache type's default size; long_p/long_from: larger
    partitions for sequences longer than long_from rows."""
    lens = [0, 1, 511, 512, 513, 1500, 5000, 0, 37, 1024, 2049, 300, 300, 7777, 20000, 70001]
    hq, hkv = 32, 8
    step = wl.build_step(f"wl_{fmt}", lens, hq, hkv, 128, cache_dtype=fmt, seed=61)
    q = to_torch(step.q, "bf16")
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    base = P or pa.pa_default_partition_size(fmt)
    ws_bytes = pa.pa_decode_workspace_size(step.num_seqs, hq, 128, step.max_context_len, P)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    bt, cl = to_torch(step.block_tables), to_torch(step.context_lens)
    if fmt == "fp8":
        kc = torch.from_numpy(np.ascontiguousarray(step.k_cache)).cuda()
        vc = torch.from_numpy(np.ascontiguousarray(step.v_cache)).cuda()
        pa.pa_decode_fp8(q, kc, vc, bt, cl, step.scale, out, step.max_context_len, 1.0, 1.0,
                         workspace=ws, error_word=err)
    else:
        kc, vc = to_torch(step.k_cache, "bf16"), to_torch(step.v_cache, "bf16")
        pa.pa_decode(q, kc, vc, bt, cl, step.scale, out, step.max_context_len, workspace=ws,
                     error_word=err, kernel="mma", partition_size=P,
                     long_partition_size=long_p, long_partition_from=long_from)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rule = (lambda n: long_p if long_from and n > long_from else base)
    want = expected_items(lens, hkv, rule, base)
    got = ws[256:256 + 16 * len(want)].cpu().numpy().view(np.int32).reshape(-1, 4)
    np.testing.assert_array_equal(got, want)

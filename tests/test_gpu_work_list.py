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


def expected_items(lens, hkv, P):
    full, partial = [], []
    for s, n in enumerate(lens):
        if n <= 0:
            continue
        nf, r = divmod(n, P)
        for part in range(nf):
            for h in range(hkv):
                full.append((s, h, part, n))
        if r:
            b = min(BUCKETS - 1, (P - r) * BUCKETS // P)
            partial.append((b, s, nf, n))
    partial.sort(key=lambda t: (t[0], t[1]))          # stable: by class, then sequence
    items = list(full)
    for _, s, part, n in partial:
        for h in range(hkv):
            items.append((s, h, part, n))
    return np.array(items, dtype=np.int32).reshape(-1, 4)


@pytest.mark.parametrize("fmt,P", [("bf16", 512), ("bf16", 64), ("fp8", 1024)])
def test_work_list_order(fmt, P):
    lens = [0, 1, 511, 512, 513, 1500, 5000, 0, 37, 1024, 2049, 300, 300, 7777]
    hq, hkv = 32, 8
    step = wl.build_step(f"wl_{fmt}", lens, hq, hkv, 128, cache_dtype=fmt, seed=61)
    q = to_torch(step.q, "bf16")
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_bytes = pa.pa_decode_workspace_size(step.num_seqs, hq, 128, step.max_context_len)
    if fmt == "bf16" and P != 512:
        ws_bytes = pa.lib().pa_decode_workspace_size_ex(step.num_seqs, hq, 128,
                                                         step.max_context_len, P)
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
                     error_word=err, kernel="mma", partition_size=P)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = expected_items(lens, hkv, P)
    got = ws[256:256 + 16 * len(want)].cpu().numpy().view(np.int32).reshape(-1, 4)
    np.testing.assert_array_equal(got, want)

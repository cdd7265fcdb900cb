"""The boundary used from plain C: tests/c/decode_example.c links only the
library and the CUDA runtime, appends the tiny fp32 workload's new rows and
decodes it through pa_reshape_and_cache and pa_decode; its output must match
the oracle within the fp32 tolerance."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from gpu_helpers import assert_parity, oracle_reference
from paged_kv_cache_29_gb300 import _binding as pa
from paged_kv_cache_29_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_c_program_decodes_the_tiny_workload(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not installed")
    pa.lib()                                           # built and loadable
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    lib = pa.LIB_PATH
    exe = str(tmp_path / "decode_example")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(HERE, "..", "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(HERE, "c", "decode_example.c"),
                    "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib),
                    "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.join(cuda, "lib64"),
                    "-o", exe], check=True)
    step = wl.make("tiny")
    assert step.cache_dtype == "f32"
    B, Hq, D = step.q.shape
    NB, Hkv, bs, _ = step.k_cache.shape
    MB = step.block_tables.shape[1]
    inp = tmp_path / "in.bin"
    with open(inp, "wb") as f:
        f.write(np.array([B, Hq, Hkv, D, bs, NB, MB, step.max_context_len], np.int32).tobytes())
        f.write(np.array([step.scale], np.float32).tobytes())
        for a, t in ((step.q, np.float32), (step.k_new, np.float32), (step.v_new, np.float32),
                     (step.slot_mapping, np.int64), (step.k_cache, np.float32),
                     (step.v_cache, np.float32), (step.block_tables, np.int32),
                     (step.context_lens, np.int32)):
            f.write(np.ascontiguousarray(a, dtype=t).tobytes())
    out = tmp_path / "out.bin"
    run = subprocess.run([exe, str(inp), str(out)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stderr)
    got = np.fromfile(out, dtype=np.float32).reshape(B, Hq, D).astype(np.float64)
    _, _, ref = oracle_reference(step)
    assert_parity(got, ref, "f32")

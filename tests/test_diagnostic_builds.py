"""The diagnostic builds of the CUDA library.

- The default build has no index checks and no timestamps
  (gemm_build_flags() == 0, gemm_set_stamps refused).
- The index-checked build (GEMM_DEBUG) must pass the parity tests that take
  every plain-store path of the epilogue (ragged right edges, block-scaled
  outputs, reductions, grouped row ranges, split tiles) with no check failing:
  a failed check skips the store and makes gemm_check return GEMM_ERR_BOUNDS,
  which those tests report as an error.  It runs them in a child process that
  loads that library through GEMM_SM103_LIBRARY.
- The timestamp build (GEMM_STAMPS) records, for every CTA that did work, its
  eight points in order.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import dense_gemm_epilogue_sm_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))


def _build(variant):
    sys.path.insert(0, os.path.join(ROOT, "dense_gemm_epilogue_sm_gb300"))
    import _build as b
    return b.build(variant=variant)


def test_default_build_has_no_diagnostics():
    assert g.gemm_build_flags() == 0
    assert g.lib.gemm_set_stamps(None, None) == g.ERR_UNSUPPORTED


@pytest.mark.gpu
def test_index_checked_build_passes_the_store_path_tests():
    lib = _build("debug")
    env = dict(os.environ, GEMM_SM103_LIBRARY=lib)
    files = ["test_gemm_gpu.py", "test_mx_output.py", "test_nv_output.py", "test_epilogue_variants.py",
             "test_grouped.py", "test_stream_k.py", "test_special_values.py"]
    code = ("import dense_gemm_epilogue_sm_gb300 as g, sys; "
            "sys.exit(0 if g.gemm_build_flags() & g.BUILD_DEBUG else 3)")
    assert subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT).returncode == 0
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider"] +
                       [os.path.join(HERE, f) for f in files], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.gpu
def test_timestamp_build_records_each_cta_in_order():
    lib = _build("stamps")
    code = r'''
import numpy as np, torch, sys
import dense_gemm_epilogue_sm_gb300 as g
from dense_gemm_epilogue_sm_gb300 import workloads as wl
from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec
assert g.gemm_build_flags() & g.BUILD_STAMPS
for spec in (wl.Spec("st_single", 300, 520, 256, beta=1.0, bias="col", seed=5),
             wl.Spec("st_pair", 2048, 2048, 512, seed=6)):
    inp = wl.make_inputs(spec)
    dev = torch.device("cuda", 0)
    A, B = inp.A.to(dev), inp.B.to(dev)
    C = None if inp.C is None else inp.C.to(dev)
    bias = None if inp.bias is None else inp.bias.to(dev)
    D = torch.empty(spec.matrix_elems("d"), dtype=torch.bfloat16, device=dev)
    op = GemmOp(desc_from_spec(spec))
    workers, cg = g.gemm_get_schedule(op.handle)[0], g.gemm_plan(op.desc).cta_group
    st = torch.zeros(workers * cg * 8, dtype=torch.int64, device=dev)
    g.gemm_set_stamps(op.handle, st.data_ptr())
    op(A, B, C, D, bias)
    op.check()
    t = st.cpu().numpy().reshape(-1, 8)
    for b, row in enumerate(t):
        seq = [row[0], row[1], row[2]] + ([row[3], row[4]] if b % cg == 0 else []) + [row[5], row[6], row[7]]
        assert all(x > 0 for x in seq), (spec.name, b, row)
        assert all(x <= y for x, y in zip(seq, seq[1:])), (spec.name, b, row)
        assert row[4] <= row[5] or b % cg == 1
    op.close()
print("ok")
'''
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, GEMM_SM103_LIBRARY=lib), cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]

"""Host-side helpers of bench.py (no GPU): the kernel-source hash ignores
comments only, the parity check of the timed output accepts the oracle's own
rows and rejects wrong ones in either D order, and the oracle view of
grouped and block-scaled-output workloads samples the right problem; the
reference arm runs without the CUDA library, reports the same config as
the GPU arm, and the roofline bound and the part's tensor peak follow
their definitions."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from dense_gemm_epilogue_sm_gb300 import workloads as wl  # noqa: E402
from oracle import gemm_ref  # noqa: E402


def test_code_only_drops_comments_and_keeps_code():
    a = 'int x = 1; // one\n/* two\n   lines */ int y = 2;\nconst char* s = "not // a comment";\n'
    b = 'int x = 1;\nint y = 2;   \n\nconst char* s = "not // a comment";'
    assert bench._code_only(a).split() == bench._code_only(b).split()
    assert bench._code_only(a) != bench._code_only(a.replace("y = 2", "y = 3"))
    assert "'/'" in bench._code_only("char c = '/'; // c")


def _storage_from_rows(spec, bits):
    D = torch.zeros(spec.batch * spec.matrix_elems("d"), dtype=wl.DT[spec.dtype_d])
    vals = torch.from_numpy(bits.view(np.int32 if spec.dtype_d == "f32" else np.int16)).view(wl.DT[spec.dtype_d])
    per, ld = spec.matrix_elems("d"), spec.ld("d")
    for r in range(spec.batch * spec.M):
        l, m = divmod(r, spec.M)
        n = torch.arange(spec.N)
        idx = l * per + (m * ld + n if spec.order_d == "row" else m + n * ld)
        D[idx] = vals[r]
    return D


def test_parity_on_rows_accepts_the_oracle_and_rejects_a_wrong_d():
    for spec in (wl.Spec("p_row", 200, 130, 96, alpha=0.5, beta=1.0, act="relu", bias="col", seed=3, pad=8),
                 wl.Spec("p_col", 128, 96, 64, order_a="col", order_b="col", order_c="col", order_d="col",
                         dtype_in="f16", dtype_d="f32", dist="int4", batch=2, seed=4)):
        inputs = wl.make_inputs(spec)
        bits, _ = gemm_ref.run_spec_rows(spec, inputs)
        D = _storage_from_rows(spec, bits)
        rows = np.array([0, 7, spec.batch * spec.M - 1])
        ok = bench.parity_on_rows(spec, inputs, D, rows, bits[rows])
        assert ok["pass"] and ok["max_err_over_tol"] == 0.0 and ok["elements"] == 3 * spec.N
        bad = D.clone()
        bad[:] = 1000.0
        assert not bench.parity_on_rows(spec, inputs, bad, rows, bits[rows])["pass"]


def test_oracle_view_samples_group_zero_and_quantises_block_scaled_d():
    g_spec = wl.Spec("v_grp", 600, 64, 32, groups=3, group_sizes=(100, 300, 200), seed=5)
    g_in = wl.make_inputs(g_spec)
    sub, sub_in, total, run = bench.oracle_view(g_spec, g_in)
    assert total == 100 and sub.groups == 0 and sub_in.B.numel() == g_spec.matrix_elems("b")
    bits = run(np.array([0, 99]))
    ref, _ = gemm_ref.run_spec_rows(sub, sub_in, rows=np.array([0, 99]))
    assert np.array_equal(bits, ref)
    n_spec = wl.Spec("v_nvo", 64, 64, 64, dtype_d="e2m1", scale_d=0.25, seed=6)
    n_in = wl.make_inputs(n_spec)
    f32_spec, _, total, run = bench.oracle_view(n_spec, n_in)
    assert total == 64 and f32_spec.dtype_d == "f32"
    codes, q = run(np.array([1, 2]))
    assert codes.shape == (2, 4) and q.shape == (2, 64)


def test_reference_arm_loads_no_cuda_library():
    # the workload generator is loaded by path; the package (whose __init__
    # loads libgemm_sm103.so) stays out of the reference arm's process
    code = ("import sys; sys.path.insert(0, %r); import bench; wl = bench.workloads_module(); "
            "wl.make_inputs(wl.get('tiny_exact_fp16_256')); "
            "assert 'dense_gemm_epilogue_sm_gb300' not in sys.modules, sorted(sys.modules)" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr


def test_roofline_bound_and_spec_peak():
    wl = bench.workloads_module()
    skinny, fused = wl.get("skinny_65536x256x4096"), wl.get("fused_bf16_8192")
    for spec, want in ((skinny, "hbm"), (fused, "tensor")):
        assert bench.roofline_bound(spec.flops(), spec.algorithmic_bytes(), 1861.9, 6777.6) == want
    assert bench.spec_peak_tflops("bf16", 152) == pytest.approx(152 * 8192 * 2.07e9 / 1e12)
    assert bench.spec_peak_tflops("e4m3", 152) == pytest.approx(2 * bench.spec_peak_tflops("bf16", 152))


def test_config_is_the_same_in_both_arms():
    # both arms build the config from the workload alone (no plan fields)
    wl = bench.workloads_module()
    for name in ("fused_bf16_8192", "batched_32x512", "grouped_16x_bf16"):
        spec = wl.get(name)
        cfg = bench.workload_config(spec, bench.needs_flush(spec))
        assert cfg == bench.workload_config(wl.get(name), bench.needs_flush(wl.get(name)))
        assert not {"tile", "stages", "kernel_hash"} & set(cfg)

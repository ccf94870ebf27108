"""The allocation-free entry point, gemm_run_noalloc, against gemm_run.

gemm_run_noalloc is for callers that must not call cudaMalloc (code inside a
framework memory pool that owns the device, latency-critical paths where an
allocation may synchronise the device).  It keeps the kernel's status word
in a fixed device array instead of an allocated one.  Two calls in a row,
through the C ABI, must reproduce what gemm_run computes on the same inputs,
within the parity tolerance used by the other GPU tests, and so must a call
that returns at once (wait = 0) once the caller synchronises.  This file is
collected last so a failure here cannot hide the others.
"""
import ctypes

import numpy as np
import pytest
import torch

import _harness as H
import dense_gemm_epilogue_sm_gb300 as g
from dense_gemm_epilogue_sm_gb300 import workloads as wl
from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec

pytestmark = pytest.mark.gpu

SPECS = [
    wl.Spec("noalloc_fused", 300, 520, 200, alpha=0.5, beta=1.0, act="relu", bias="col", seed=31, pad=3),
    wl.Spec("noalloc_colmajor_f32", 257, 190, 136, op_a="T", order_a="row", order_b="row", order_c="col",
            order_d="col", dtype_d="f32", beta=0.75, bias="row", seed=32),
]


def _device_inputs(spec):
    inputs = wl.make_inputs(spec)
    dev = torch.device("cuda", 0)
    moved = [None if t is None else t.to(dev) for t in (inputs.A, inputs.B, inputs.C, inputs.bias)]
    return inputs, moved


def _ptr(t):
    return None if t is None else t.data_ptr()


def test_two_calls_match_gemm_run():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    stream = torch.cuda.current_stream().cuda_stream
    for spec in SPECS:
        inputs, (A, B, C, bias) = _device_inputs(spec)
        desc = desc_from_spec(spec, inputs.scale_a, inputs.scale_b)

        ref_buf = H.canary_buffer(spec)
        op = GemmOp(desc)
        op(A, B, C, ref_buf, bias)
        op.check()
        op.close()

        # two calls that wait, then one that returns at once (the caller synchronises)
        for call, wait in enumerate((1, 1, 0)):
            out = H.canary_buffer(spec)
            status = g.lib.gemm_run_noalloc(ctypes.byref(desc), _ptr(A), _ptr(B), _ptr(C), _ptr(out), _ptr(bias),
                                            stream, wait)
            assert status == g.OK, g.gemm_status_str(status)
            torch.cuda.synchronize()
            got_bits = H.bits_of_tensor(out.cpu())
            ref_bits = H.bits_of_tensor(ref_buf.cpu())
            assert H.untouched_outside(spec, got_bits), f"{spec.name} call {call}: write outside D"
            got = H.from_bits(H.logical_d(spec, got_bits).reshape(-1), spec.dtype_d)
            ref = H.from_bits(H.logical_d(spec, ref_bits).reshape(-1), spec.dtype_d)
            assert np.isfinite(got).all(), f"{spec.name} call {call}: unwritten output"
            tol = H.tolerance(spec, inputs, ref)
            assert np.all(np.abs(got - ref) <= tol), f"{spec.name} call {call}: differs from gemm_run"


def test_rejects_bad_arguments_without_launching():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    spec = SPECS[0]
    desc = desc_from_spec(spec)
    bad = desc_from_spec(spec)
    bad.M = -1
    assert g.lib.gemm_run_noalloc(ctypes.byref(bad), None, None, None, None, None, None, 1) == g.ERR_INVALID_ARG
    assert g.lib.gemm_run_noalloc(ctypes.byref(desc), None, None, None, None, None, None, 2) == g.ERR_INVALID_ARG


def test_empty_problem_after_a_launch_reports_ok():
    # an empty problem queues no kernel: waiting must not read the status
    # word the previous call left
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    stream = torch.cuda.current_stream().cuda_stream
    spec = SPECS[0]
    inputs, (A, B, C, bias) = _device_inputs(spec)
    desc = desc_from_spec(spec, inputs.scale_a, inputs.scale_b)
    out = H.canary_buffer(spec)
    assert g.lib.gemm_run_noalloc(ctypes.byref(desc), _ptr(A), _ptr(B), _ptr(C), _ptr(out), _ptr(bias),
                                  stream, 1) == g.OK
    empty = desc_from_spec(spec, inputs.scale_a, inputs.scale_b)
    empty.M = 0
    assert g.lib.gemm_run_noalloc(ctypes.byref(empty), _ptr(A), _ptr(B), _ptr(C), _ptr(out), _ptr(bias),
                                  stream, 1) == g.OK

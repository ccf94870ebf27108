"""Dynamic schedule (gemm_set_schedule(GEMM_SCHED_DYNAMIC): cluster launch
control) on the GPU.  The launch holds one cluster per tile; clusters that
finish a tile cancel pending ones and take their tiles.  Checked: results
against the oracle on several kernels and layouts, bit-identical integer
results to the static schedule, repeated launches with new inputs, a
concurrent kernel holding SMs, and a timed-out launch that ends promptly and
leaves the handle usable."""
import dataclasses
import time

import numpy as np
import pytest
import torch

import _harness as H
import dense_gemm_epilogue_sm_gb300 as g
from dense_gemm_epilogue_sm_gb300 import workloads as wl
from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec

pytestmark = pytest.mark.gpu

SPECS = [
    wl.Spec("dyn_pair_fused", 2300, 2310, 1000, alpha=0.5, beta=1.0, act="relu", bias="col", seed=71, pad=3),
    wl.Spec("dyn_pair_f32_colmajor", 2200, 2600, 768, op_a="T", order_a="col", order_c="col", order_d="col",
            dtype_d="f32", beta=0.75, bias="row", seed=72),
    wl.Spec("dyn_pair_e4m3", 2560, 2560, 2048, dtype_in="e4m3", dist="uniform1", seed=73),
    wl.Spec("dyn_pair_batched", 512, 1024, 1024, batch=12, beta=1.0, seed=74),
    wl.Spec("dyn_single_n128", 20000, 128, 520, bias="col", act="gelu", seed=75),
    wl.Spec("dyn_single_small", 300, 520, 200, alpha=0.5, beta=1.0, bias="row", seed=76),
]


def _op(spec, inputs, mode=g.SCHED_DYNAMIC):
    op = GemmOp(desc_from_spec(spec, inputs.scale_a, inputs.scale_b))
    op.set_schedule(mode)
    return op


def _check(spec, inputs, bits):
    assert H.untouched_outside(spec, bits), "write outside the logical D"
    d = H.logical_d(spec, bits)
    rows = H.sample_rows(spec)
    H.compare(spec, inputs, d, H.oracle_rows(spec, inputs, rows), rows=rows)


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_dynamic_matches_oracle(spec):
    inputs = wl.make_inputs(spec)
    op = _op(spec, inputs)
    bits, _ = H.run_gpu(spec, inputs, op=op)
    _check(spec, inputs, bits)
    op.close()


def test_dynamic_equals_static_bit_for_bit_on_integers():
    spec = wl.Spec("dyn_int", 2304, 2304, 1024, dtype_in="f16", dtype_d="f32", dist="int4", seed=77)
    inputs = wl.make_inputs(spec)
    dyn = H.logical_d(spec, H.run_gpu(spec, inputs, op=_op(spec, inputs))[0])
    dp = H.logical_d(spec, H.run_gpu(spec, inputs, op=_op(spec, inputs, g.SCHED_DATA_PARALLEL))[0])
    assert np.array_equal(dyn, dp)
    H.compare(spec, inputs, dyn, H.oracle_rows(spec, inputs), exact=True)


def test_dynamic_repeat_launches_with_new_inputs():
    op = None
    for seed in (81, 82):
        spec = dataclasses.replace(SPECS[0], seed=seed)
        inputs = wl.make_inputs(spec)
        op = op or _op(spec, inputs)
        bits, _ = H.run_gpu(spec, inputs, op=op, repeat=3)
        _check(spec, inputs, bits)
    op.close()


def test_dynamic_beside_a_concurrent_kernel():
    spec = SPECS[0]
    inputs = wl.make_inputs(spec)
    op = _op(spec, inputs)
    other = torch.cuda.Stream()
    x = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    torch.cuda.synchronize()
    with torch.cuda.stream(other):
        for _ in range(4):
            y = x @ x                               # holds SMs while the GEMM starts
    bits, _ = H.run_gpu(spec, inputs, op=op)
    torch.cuda.synchronize()
    del y
    _check(spec, inputs, bits)
    op.close()


def test_dynamic_timeout_ends_promptly_and_recovers():
    spec = wl.get("bf16_4096")
    inputs = wl.make_inputs(spec)
    op = _op(spec, inputs)
    g.gemm_set_debug(op.handle, 1, 100)
    dev = torch.device("cuda", 0)
    A, B = inputs.A.to(dev), inputs.B.to(dev)
    D = H.canary_buffer(spec)
    torch.cuda.synchronize()
    t0 = time.time()
    op(A, B, None, D)
    with pytest.raises(g.GemmError) as e:
        op.check()
    assert e.value.status == g.ERR_TIMEOUT
    # clusters started after the failure do no work: far less than one
    # timeout per tile (256 tiles x 100 ms)
    assert time.time() - t0 < 5.0
    g.gemm_set_debug(op.handle, 0, 2000)
    bits, _ = H.run_gpu(spec, inputs, op=op)
    _check(spec, inputs, bits)
    op.close()

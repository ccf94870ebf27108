"""The staged epilogue's compile-time forms on the GPU.

Staged subtiles outside the extended epilogue are written by one of twelve
compile-time forms: C or not (beta = 0 / 1), no / column / row bias, ReLU or
not.  Each form, for a 16-bit and an fp32 output, is compared with the oracle
on rows sampled from every 128-row tile.  M = 2304, N = 2200 gives 81 CTA-pair
tiles (the pair kernel) and a ragged right edge (N is not a multiple of the
64-column subtile), so the plain-store subtile sits beside staged ones in the
last tile column; nothing outside D may be written.
"""
import pytest

import _harness as H
import dense_gemm_epilogue_sm_gb300 as g
from dense_gemm_epilogue_sm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FORMS = [(beta, bias, act) for beta in (0.0, 1.0) for bias in ("none", "col", "row") for act in ("none", "relu")]


@pytest.mark.parametrize("dtype_d", ["bf16", "f32"])
@pytest.mark.parametrize("beta,bias,act", FORMS, ids=lambda v: str(v))
def test_every_epilogue_form_matches_oracle(dtype_d, beta, bias, act):
    spec = wl.Spec(f"form_{dtype_d}_{beta}_{bias}_{act}", 2304, 2200, 256, order_a="row", order_b="col",
                   dtype_d=dtype_d, alpha=0.5, beta=beta, bias=bias, act=act, seed=301)
    inputs = wl.make_inputs(spec)
    bits, op = H.run_gpu(spec, inputs)
    assert g.gemm_plan(op.desc).cta_group == 2, "the case should take the CTA-pair kernel"
    assert H.untouched_outside(spec, bits), "write outside the logical D"
    rows = H.sample_rows(spec)
    H.compare(spec, inputs, H.logical_d(spec, bits), H.oracle_rows(spec, inputs, rows), rows=rows)
    op.close()

"""Epilogue variants on the GPU: the GELU activation and the row-sum,
column-sum and abs-max reductions of the epilogue value t (gemm_run_ex),
against the oracle's t and its reductions.

Tolerances (derived from the arithmetic, with u = 2^-24):
  t, per element   e = slope * tau * sqrt(K) * max|A| * max|B| + 4u|t|
  row sum over N   N e + (N + tiles) u sum|t|   (fp32 sums in the epilogue
  column sum       M e + (M + 5) u sum|t|        and the finishing pass)
  abs-max          e + u |t|max
Integer-valued inputs make every t and every sum exact in fp32: compared bit
for bit.
"""
import dataclasses

import numpy as np
import pytest
import torch

import _harness as H
from _dtypes import from_bits, to_bits
import dense_gemm_epilogue_sm_gb300 as g
from dense_gemm_epilogue_sm_gb300 import workloads as wl
from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec
from oracle import gemm_ref

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


def _oracle_t(spec, inputs):
    _, t = gemm_ref.run_spec_rows(spec, inputs, want_t=True)
    return t.reshape(spec.batch, spec.M, spec.N)


def _run_ex(spec, inputs, mode=None, repeat=1):
    op = GemmOp(desc_from_spec(spec, inputs.scale_a, inputs.scale_b))
    if mode is not None:
        op.set_schedule(mode)
    dev = torch.device("cuda", 0)
    A, B = inputs.A.to(dev), inputs.B.to(dev)
    C = inputs.C.to(dev) if inputs.C is not None else None
    bias = inputs.bias.to(dev) if inputs.bias is not None else None
    D = H.canary_buffer(spec)
    L, red = spec.batch, spec.reduce.split("+")
    nan = lambda n: torch.full((n,), float("nan"), dtype=torch.float32, device=dev)
    rs = nan(L * spec.M) if "row" in red else None
    cs = nan(L * spec.N) if "col" in red else None
    am = nan(L) if "amax" in red else None
    for _ in range(repeat):
        op.run_ex(A, B, C, D, bias, rs, cs, am)
    op.check()
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy().astype(np.float64).reshape(L, -1)
           for k, v in (("row", rs), ("col", cs), ("amax", am)) if v is not None}
    bits = H.bits_of_tensor(D.cpu())
    info = g.gemm_plan(op.desc)
    op.close()
    return bits, out, info


def _check_reductions(spec, inputs, out, t, info):
    e = H.accumulation_bound(spec, inputs) + 4 * U * np.abs(t)
    at = np.abs(t)
    tiles = max(info.tiles_m, info.tiles_n)
    if "row" in out:
        tol = e.sum(axis=2) + (spec.N + tiles) * U * at.sum(axis=2)
        err = np.abs(out["row"] - gemm_ref.row_sums(t))
        assert np.all(err <= tol), f"row sums: worst {np.max(err - tol)} over"
    if "col" in out:
        tol = e.sum(axis=1) + (spec.M + 5) * U * at.sum(axis=1)
        err = np.abs(out["col"] - gemm_ref.col_sums(t))
        assert np.all(err <= tol), f"column sums: worst {np.max(err - tol)} over"
    if "amax" in out:
        want = gemm_ref.abs_max(t)
        tol = e.max(axis=(1, 2)) + U * want
        assert np.all(np.abs(out["amax"].reshape(-1) - want) <= tol)


GELU_CASES = [("bf16", "bf16"), ("f16", "f16"), ("bf16", "f32"), ("e4m3", "bf16")]


@pytest.mark.parametrize("order_d", ["row", "col"])
@pytest.mark.parametrize("dtype_in,dtype_d", GELU_CASES)
def test_gelu_matches_oracle(dtype_in, dtype_d, order_d):
    spec = wl.Spec("gelu", 300, 528, 208, dtype_in=dtype_in, dtype_d=dtype_d, order_c=order_d, order_d=order_d,
                   alpha=0.75, beta=0.5, act="gelu", bias="col", seed=61,
                   dist="uniform1" if dtype_in == "e4m3" else "normal")
    inputs = wl.make_inputs(spec)
    bits, _ = H.run_gpu(spec, inputs)
    assert H.untouched_outside(spec, bits)
    H.compare(spec, inputs, H.logical_d(spec, bits), H.oracle_rows(spec, inputs))


RED_SPECS = [
    wl.Spec("red_single", 600, 520, 256, alpha=0.5, beta=1.0, act="gelu", bias="col", reduce="row+col+amax",
            seed=62, pad=5),
    wl.Spec("red_pair_f32_colmajor", 2048, 2176, 256, op_a="T", order_a="col", order_c="col", order_d="col",
            dtype_d="f32", beta=0.75, act="relu", bias="row", reduce="row+col+amax", seed=63),
    wl.Spec("red_batched", 300, 400, 128, batch=3, act="gelu", bias="col", reduce="row+col+amax", seed=64),
    wl.Spec("red_e4m3", 640, 512, 512, dtype_in="e4m3", dist="uniform1", act="gelu", reduce="amax+col", seed=65),
    wl.Spec("red_rows_only", 1000, 1000, 320, beta=1.0, reduce="row", seed=66),
]


@pytest.mark.parametrize("spec", RED_SPECS, ids=lambda s: s.name)
def test_reductions_match_oracle(spec):
    inputs = wl.make_inputs(spec)
    bits, out, info = _run_ex(spec, inputs)
    assert H.untouched_outside(spec, bits)
    H.compare(spec, inputs, H.logical_d(spec, bits), H.oracle_rows(spec, inputs))
    _check_reductions(spec, inputs, out, _oracle_t(spec, inputs), info)


def test_reductions_with_split_tiles():
    # 81 pair tiles on 76 workers: the split cuts the last tiles between
    # workers, so owners reduce after adding partial sums
    spec = wl.Spec("red_split", 2304, 2304, 512, alpha=0.5, beta=1.0, act="gelu", bias="col",
                   reduce="row+col+amax", seed=67)
    inputs = wl.make_inputs(spec)
    t = _oracle_t(spec, inputs)
    for mode in (g.SCHED_SPLIT_TAIL, g.SCHED_STREAM_K):
        bits, out, info = _run_ex(spec, inputs, mode=mode)
        H.compare(spec, inputs, H.logical_d(spec, bits), H.oracle_rows(spec, inputs))
        _check_reductions(spec, inputs, out, t, info)


def test_reductions_exact_on_integers_and_repeatable():
    spec = wl.Spec("red_int", 512, 768, 256, dtype_in="f16", dtype_d="f32", dist="int4", beta=1.0, bias="col",
                   reduce="row+col+amax", seed=68)
    inputs = wl.make_inputs(spec)
    # integer bias keeps t integral
    inputs = dataclasses.replace(inputs, bias=torch.round(inputs.bias * 20))
    t = _oracle_t(spec, inputs)
    bits, out, _ = _run_ex(spec, inputs, repeat=2)
    assert np.array_equal(out["row"], gemm_ref.row_sums(t))
    assert np.array_equal(out["col"], gemm_ref.col_sums(t))
    assert np.array_equal(out["amax"].reshape(-1), gemm_ref.abs_max(t))
    _, out2, _ = _run_ex(spec, inputs)
    for k in out:
        assert np.array_equal(out[k], out2[k])


def test_full_size_fused_reductions():
    spec = dataclasses.replace(wl.get("fused_bf16_8192"), reduce="row+col+amax")
    inputs = wl.make_inputs(spec)
    bits, out, info = _run_ex(spec, inputs)
    d = from_bits(H.logical_d(spec, bits).reshape(-1), "bf16")
    # both come from the same fp32 t: rounding is monotonic, so the largest
    # |D| is the rounded abs-max
    amax_bf16 = from_bits(to_bits(np.array([out["amax"][0, 0]]), "bf16"), "bf16")[0]
    assert amax_bf16 == np.max(np.abs(d))
    # sampled rows: row sums against the oracle's t of those rows
    rows = H.sample_rows(spec, per_tile=1)
    _, t_rows = gemm_ref.run_spec_rows(spec, inputs, rows=rows, want_t=True)
    e = H.accumulation_bound(spec, inputs) + 4 * U * np.abs(t_rows)
    tol = e.sum(axis=1) + (spec.N + info.tiles_n) * U * np.abs(t_rows).sum(axis=1)
    assert np.all(np.abs(out["row"][0, rows] - t_rows.sum(axis=1)) <= tol)
    # every column sum and every row sum add up to the same total
    tot_r, tot_c = out["row"].sum(), out["col"].sum()
    assert abs(tot_r - tot_c) <= 2 * (spec.M + spec.N) * U * np.abs(out["row"]).sum()


def test_reduction_argument_errors():
    spec = dataclasses.replace(RED_SPECS[0])
    desc = desc_from_spec(spec)
    op = GemmOp(desc)
    dev = torch.device("cuda", 0)
    x = torch.zeros(1 << 20, device=dev)
    with pytest.raises(g.GemmError) as e:
        op(x, x, x, x, x)                                  # plain gemm_run: outputs missing
    assert e.value.status == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        op.run_ex(x, x, x, x, x, row_sum=x, col_sum=x)    # abs-max output missing
    assert e.value.status == g.ERR_INVALID_ARG
    op.close()
    with pytest.raises(g.GemmError) as e:
        g.gemm_run_noalloc(desc, x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), None)
    assert e.value.status == g.ERR_UNSUPPORTED

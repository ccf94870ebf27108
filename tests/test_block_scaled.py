"""Block-scaled GEMM on the GPU, through gemm_run_args, against the oracle:
MXFP8 (e4m3 operands, one ue8m0 scale factor per 32 elements of K) and
NVFP4 (e2m1 operands two per byte, one ue4m3 factor per 16, fp32 global
scales in scale_a / scale_b).

Both sides read the same operand bytes and scale-factor bytes, so the only
difference is fp32 accumulation order: per element
    |D - D_ref| <= 2 K u |alpha| sum_k |a_k b_k| + 4 u |t| + ulp_D(|D_ref|)
with u = 2^-24 and sum_k |a_k b_k| (scale factors included) taken from the
oracle run on the operands with their sign bits cleared.  Integer data
(MXFP8) or any e2m1 code (NVFP4) with factors 2^-1..2^1 makes every sum
exact in fp32: compared bit for bit.  The exact case catches any misplaced
scale factor, since factors differ by powers of two from block to block."""
import dataclasses

import numpy as np
import pytest
import torch

import _harness as H
from _dtypes import from_bits
import dense_gemm_epilogue_sm_gb300 as g
from dense_gemm_epilogue_sm_gb300 import workloads as wl
from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec
from oracle import gemm_ref

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


def _dev(t):
    return None if t is None else t.to("cuda")


def _run(spec, inputs, op=None, repeat=1):
    op = op or GemmOp(desc_from_spec(spec, inputs.scale_a, inputs.scale_b))
    A, B, C, bias = (_dev(t) for t in (inputs.A, inputs.B, inputs.C, inputs.bias))
    sfa, sfb = _dev(inputs.extras["sfa"]), _dev(inputs.extras["sfb"])
    D = H.canary_buffer(spec)
    for _ in range(repeat):
        op.run_args(A, B, C, D, bias, sfa=sfa, sfb=sfb)
    op.check()
    torch.cuda.synchronize()
    return H.bits_of_tensor(D.cpu()), op


def _clear_sign(t):
    if t.dtype == torch.uint8:                  # two e2m1 codes per byte, sign in bit 3 of each
        return t & 0x77
    return (t.view(torch.uint8) & 0x7F).view(torch.float8_e4m3fn)


def _check(spec, inputs, bits, rows=None, exact=False):
    assert H.untouched_outside(spec, bits), "write outside the logical D"
    d = H.logical_d(spec, bits)
    ref_bits, t = gemm_ref.run_spec_rows(spec, inputs, rows=rows, want_t=True)
    if exact:
        H.compare(spec, inputs, d, ref_bits, rows=rows, exact=True)
        return
    abs_spec = dataclasses.replace(spec, alpha=1.0, beta=0.0, bias="none", act="none", dtype_d="f32",
                                   order_c="row", order_d="row", pad=0, ldc=0, ldd=0)
    abs_inputs = wl.Inputs(abs_spec, _clear_sign(inputs.A), _clear_sign(inputs.B), None, None, inputs.scale_a,
                           inputs.scale_b, extras=inputs.extras)
    _, tabs = gemm_ref.run_spec_rows(abs_spec, abs_inputs, rows=rows, want_t=True)
    got = d.reshape(spec.batch * spec.M, spec.N)
    if rows is not None:
        got = got[np.asarray(rows)]
    got = from_bits(got, spec.dtype_d).reshape(got.shape)
    ref = from_bits(ref_bits, spec.dtype_d).reshape(ref_bits.shape)
    slope = H.SLOPE[spec.act]
    tol = slope * (2 * spec.K * U * abs(spec.alpha) * tabs + 4 * U * np.abs(t)) + H.ulp(ref, spec.dtype_d)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), "non-finite output"
    assert np.all(err <= tol), f"{int((err > tol).sum())} elements out of tolerance, worst {np.max(err - tol)}"


SPECS = [
    wl.Spec("mx_one_tile", 128, 128, 128, dtype_in="e4m3", block_scale="mx", seed=91),
    wl.Spec("mx_ragged_fused", 300, 520, 256, dtype_in="e4m3", block_scale="mx", alpha=0.5, beta=1.0, act="relu",
            bias="col", seed=92, pad=16),
    wl.Spec("mx_partial_k_colmajor_f32", 257, 190, 1008, dtype_in="e4m3", dtype_d="f32", block_scale="mx",
            order_c="col", order_d="col", beta=0.75, bias="row", seed=93),
    wl.Spec("mx_mn_major", 384, 256, 512, order_a="col", order_b="row", dtype_in="e4m3", block_scale="mx",
            act="gelu", seed=94),
    wl.Spec("mx_transposed", 200, 272, 384, op_a="T", op_b="T", order_a="row", order_b="row", dtype_in="e4m3",
            block_scale="mx", seed=95),
    wl.Spec("mx_batched", 256, 384, 320, batch=3, dtype_in="e4m3", block_scale="mx", beta=1.0, seed=96),
]


# big enough for the CTA-pair variants: 256 x 256 tiles (one accumulator)
# where at least 64 of them exist, else 256 x 128
PAIR256_SPECS = [
    wl.Spec("mx_pair256_ragged_fused", 2300, 2100, 1024, dtype_in="e4m3", block_scale="mx", alpha=0.5, beta=1.0,
            act="gelu", bias="col", seed=105, pad=16),
    wl.Spec("mx_pair256_b_mn_major", 2048, 2048, 640, order_b="row", dtype_in="e4m3", block_scale="mx", seed=106),
]
PAIR_SPECS = [
    wl.Spec("mx_pair_ragged_fused", 2100, 1300, 1024, dtype_in="e4m3", block_scale="mx", alpha=0.5, beta=1.0,
            act="relu", bias="col", seed=101, pad=16),
    wl.Spec("mx_pair_colmajor_f32", 1500, 2400, 768, dtype_in="e4m3", dtype_d="f32", block_scale="mx",
            order_c="col", order_d="col", bias="row", seed=102),
    wl.Spec("mx_pair_a_mn_major_batched", 1024, 1024, 512, batch=3, order_a="col", order_b="col", dtype_in="e4m3",
            block_scale="mx", beta=1.0, seed=103),
]


def test_mn_major_b_stays_on_one_cta():
    # too few 256 x 256 tiles; each CTA of a 256 x 128 pair would hold 64 rows
    # of B, narrower than one MN-major e4m3 box
    spec = wl.Spec("mx_b_mn", 2048, 1024, 512, order_b="row", dtype_in="e4m3", block_scale="mx", seed=104)
    info = g.gemm_plan(desc_from_spec(spec))
    assert not info.b_k_major and info.cta_group == 1
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs)
    _check(spec, inputs, bits, rows=H.sample_rows(spec))
    op.close()


@pytest.mark.parametrize("spec", SPECS + PAIR_SPECS + PAIR256_SPECS, ids=lambda s: s.name)
def test_block_scaled_matches_oracle(spec):
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs)
    info = g.gemm_plan(op.desc)
    want_cg = 1 if spec in SPECS else 2
    want_n = 256 if spec in PAIR256_SPECS else 128
    assert (info.cta_group, info.tile_m, info.tile_n, info.tile_k) == (want_cg, 128 * want_cg, want_n, 128)
    rows = H.sample_rows(spec) if want_cg == 2 else None
    _check(spec, inputs, bits, rows=rows)
    op.close()


@pytest.mark.parametrize("M,N", [(512, 384), (2304, 1152), (2304, 2176)])   # one CTA, pairs 256x128, 256x256
@pytest.mark.parametrize("order_d", ["row", "col"])
def test_block_scaled_integer_sums_bit_exact(order_d, M, N):
    spec = wl.Spec("mx_int", M, N, 1024, dtype_in="e4m3", dtype_d="f32", dist="int4", block_scale="mx",
                   order_c=order_d, order_d=order_d, seed=97)
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs, repeat=2)
    _check(spec, inputs, bits, exact=True)
    op.close()


def test_block_scaled_full_size_sampled_rows():
    spec = wl.get("mxfp8_8192")
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs)
    _check(spec, inputs, bits, rows=H.sample_rows(spec, per_tile=1))
    op.close()


def test_block_scaled_argument_errors():
    spec = SPECS[0]
    inputs = wl.make_inputs(spec)
    op = GemmOp(desc_from_spec(spec))
    A, B = _dev(inputs.A), _dev(inputs.B)
    sf = _dev(inputs.extras["sfa"])
    D = H.canary_buffer(spec)
    with pytest.raises(g.GemmError) as e:
        op(A, B, None, D)                                   # gemm_run has no scale factors
    assert e.value.status == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        op.run_args(A, B, None, D, sfa=sf)                  # sfb missing
    assert e.value.status == g.ERR_INVALID_ARG
    raw = torch.zeros(sf.numel() + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.GemmError) as e:
        op.run_args(A, B, None, D, sfa=raw[1:], sfb=sf)      # not 16-byte aligned
    assert e.value.status == g.ERR_MISALIGNED
    op.close()
    desc = desc_from_spec(spec)
    with pytest.raises(g.GemmError) as e:
        g.gemm_run_noalloc(desc, A.data_ptr(), B.data_ptr(), None, D.data_ptr(), None, None)
    assert e.value.status == g.ERR_UNSUPPORTED


# ----------------------------------------------------------------- NVFP4 --
NV_SPECS = [
    wl.Spec("nv_one_tile", 128, 128, 256, dtype_in="e2m1", block_scale="nv", seed=111),
    wl.Spec("nv_ragged_fused", 300, 520, 1000, dtype_in="e2m1", block_scale="nv", alpha=0.5, beta=1.0, act="relu",
            bias="col", seed=112, pad=32),
    wl.Spec("nv_short_k_colmajor_f32", 257, 190, 176, dtype_in="e2m1", dtype_d="f32", block_scale="nv",
            order_c="col", order_d="col", beta=0.75, bias="row", seed=113),
    wl.Spec("nv_transposed_gelu", 200, 272, 512, op_a="T", op_b="T", order_a="col", order_b="row",
            dtype_in="e2m1", block_scale="nv", act="gelu", seed=114),
    wl.Spec("nv_batched", 256, 384, 320, batch=3, dtype_in="e2m1", block_scale="nv", beta=1.0, seed=115),
]
NV_PAIR_SPECS = [
    wl.Spec("nv_pair_ragged_fused", 2100, 1300, 1024, dtype_in="e2m1", block_scale="nv", alpha=0.5, beta=1.0,
            act="relu", bias="col", seed=116, pad=32),
    wl.Spec("nv_pair_batched_f32", 1024, 1024, 768, batch=3, dtype_in="e2m1", dtype_d="f32", block_scale="nv",
            beta=1.0, seed=117),
]
NV_PAIR256_SPECS = [
    wl.Spec("nv_pair256_ragged_fused", 2300, 2100, 1056, dtype_in="e2m1", block_scale="nv", alpha=0.5, beta=1.0,
            act="gelu", bias="col", seed=118, pad=32),
    wl.Spec("nv_pair256_colmajor", 2048, 2304, 2048, dtype_in="e2m1", block_scale="nv", order_c="col",
            order_d="col", beta=1.0, bias="row", seed=119),
]


@pytest.mark.parametrize("spec", NV_SPECS + NV_PAIR_SPECS + NV_PAIR256_SPECS, ids=lambda s: s.name)
def test_nvfp4_matches_oracle(spec):
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs)
    info = g.gemm_plan(op.desc)
    want_cg = 1 if spec in NV_SPECS else 2
    want_n = 256 if spec in NV_PAIR256_SPECS else 128
    assert (info.cta_group, info.tile_m, info.tile_n, info.tile_k) == (want_cg, 128 * want_cg, want_n, 256)
    rows = H.sample_rows(spec) if want_cg == 2 else None
    _check(spec, inputs, bits, rows=rows)
    op.close()


@pytest.mark.parametrize("M,N", [(512, 384), (2304, 1152), (2304, 2176)])   # one CTA, pairs 256x128, 256x256
@pytest.mark.parametrize("order_d", ["row", "col"])
def test_nvfp4_exact_sums_bit_exact(order_d, M, N):
    spec = wl.Spec("nv_int", M, N, 1024, dtype_in="e2m1", dtype_d="f32", dist="int4", block_scale="nv",
                   order_c=order_d, order_d=order_d, seed=120)
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs, repeat=2)
    _check(spec, inputs, bits, exact=True)
    op.close()


def test_nvfp4_full_size_sampled_rows():
    spec = wl.get("nvfp4_8192")
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs)
    _check(spec, inputs, bits, rows=H.sample_rows(spec, per_tile=1))
    op.close()


# ------------------------------------------------------ work splits ----
@pytest.mark.parametrize("mode", ["stream_k", "split_tail", "dynamic"])
@pytest.mark.parametrize("fmt", ["mx", "nv"])
def test_block_scaled_under_every_work_split_bit_exact(fmt, mode):
    # 81 pair tiles of 256 x 256 on 76 pairs: the last wave is cut (split
    # forms) or scheduled on the fly (dynamic); exact sums make every form
    # equal to the data-parallel result bit for bit
    dtype = "e4m3" if fmt == "mx" else "e2m1"
    spec = wl.Spec(f"bs_{fmt}_{mode}", 2304, 2304, 2048, dtype_in=dtype, dtype_d="f32", dist="int4",
                   block_scale=fmt, seed=150)
    inputs = wl.make_inputs(spec)
    modes = {"stream_k": g.SCHED_STREAM_K, "split_tail": g.SCHED_SPLIT_TAIL, "dynamic": g.SCHED_DYNAMIC}
    op = GemmOp(desc_from_spec(spec, inputs.scale_a, inputs.scale_b))
    op.set_schedule(modes[mode])
    if mode != "dynamic":
        assert op.schedule[2] > 0, "the split cuts no tile: the case tests nothing"
    bits, _ = _run(spec, inputs, op=op, repeat=2)
    dp = GemmOp(desc_from_spec(spec, inputs.scale_a, inputs.scale_b))
    dp.set_schedule(g.SCHED_DATA_PARALLEL)
    dp_bits, _ = _run(spec, inputs, op=dp)
    assert np.array_equal(H.logical_d(spec, bits), H.logical_d(spec, dp_bits))
    _check(spec, inputs, bits, exact=True)
    op.close()
    dp.close()

"""Special values through the C ABI, element by element against the oracle.

Every case is built from small-integer operands so that all finite sums are
exact in fp32 and fp64 alike; the GPU result must then equal the oracle's bit
for bit, NaN included (any NaN matches any NaN):
- beta = 0 with a C buffer full of NaN: C is not read, D stays finite (the
  BLAS rule of "CUTLASS", opening section: C enters only through beta * C);
- NaN in A (and the e4m3 NaN code), +Inf and -Inf in B: IEEE products and sums,
  so NaN rows, Inf * 0 = NaN, Inf - Inf = NaN and +-Inf columns, and ReLU
  sending NaN to 0 (t > 0 ? t : 0);
- results past the largest f16, bf16 and fp32 values become +-Inf;
- results in the subnormal range of f16, bf16 and fp32 are rounded to nearest
  even among the subnormals, not flushed, and fp32-subnormal products are
  kept by the tensor core's accumulation;
- -0 results (alpha < 0 times a zero sum) keep their sign.
ReLU results are compared by value (its zero may be either sign).
"""
import dataclasses

import numpy as np
import pytest
import torch

import _harness as H
from _dtypes import from_bits
from dense_gemm_epilogue_sm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SHAPES = [(300, 520, 256), (2048, 2048, 128)]          # one CTA per tile / CTA pairs


def _run_and_compare(spec, inputs, by_value=False):
    bits, op = H.run_gpu(spec, inputs)
    op.close()
    assert H.untouched_outside(spec, bits), "write outside the logical D"
    got = H.logical_d(spec, bits).reshape(spec.batch * spec.M, spec.N)
    ref = H.oracle_rows(spec, inputs)
    g = from_bits(got, spec.dtype_d).reshape(got.shape)
    r = from_bits(ref, spec.dtype_d).reshape(ref.shape)
    both_nan = np.isnan(g) & np.isnan(r)
    same = (g == r) if by_value else (got.astype(np.uint64) == ref.astype(np.uint64))
    bad = ~(both_nan | same)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{int(bad.sum())} elements differ; first at {i}: got {g[i]!r} "
                             f"({int(got[i]):#x}), want {r[i]!r} ({int(ref[i]):#x})")
    return g, r


def _int_spec(name, M, N, K, **kw):
    kw.setdefault("dist", "int4")
    return wl.Spec(name, M, N, K, seed=kw.pop("seed", 900), **kw)


def _a_index(spec, m, k):
    assert spec.op_a == "N" and spec.order_a == "row"
    return m * spec.ld("a") + k


def _b_index(spec, k, n):
    assert spec.op_b == "N" and spec.order_b == "col"
    return n * spec.ld("b") + k


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_nan_c_is_not_read_when_beta_is_zero(M, N, K):
    spec = _int_spec("nan_c_beta0", M, N, K, bias="col")
    inputs = wl.make_inputs(spec)
    nan_c = torch.full((spec.batch * spec.matrix_elems("c"),), float("nan"), dtype=torch.bfloat16)
    inputs = dataclasses.replace(inputs, C=nan_c, bias=torch.round(inputs.bias * 40))
    g, _ = _run_and_compare(spec, inputs)
    assert np.isfinite(g).all()


def _plant_specials(spec, inputs, nan_code=None):
    """NaN in A (row 3 at k 5), +Inf and -Inf in B (column 11 at k 9 and
    column 12 at k 10, both at k 9 and 10 in column 13), and zeros beside
    them in A so that Inf * 0 appears (row 20 at k 9)."""
    A = inputs.A.clone()
    B = inputs.B.clone()
    if nan_code is None:
        A[_a_index(spec, 3, 5)] = float("nan")
        B[_b_index(spec, 9, 11)] = float("inf")
        B[_b_index(spec, 10, 12)] = float("-inf")
        B[_b_index(spec, 9, 13)] = float("inf")
        B[_b_index(spec, 10, 13)] = float("-inf")
    else:                                   # e4m3 has a NaN code and no infinities
        A.view(torch.uint8)[_a_index(spec, 3, 5)] = nan_code
        B.view(torch.uint8)[_b_index(spec, 9, 11)] = nan_code
    A[_a_index(spec, 20, 9)] = 0.0
    return dataclasses.replace(inputs, A=A, B=B)


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("act", ["none", "relu"])
def test_nan_and_inf_operands_propagate_as_ieee(M, N, K, act):
    spec = _int_spec("nan_inf_ops", M, N, K, act=act)
    inputs = _plant_specials(spec, wl.make_inputs(spec))
    g, r = _run_and_compare(spec, inputs, by_value=(act == "relu"))
    if act == "none":
        assert np.isnan(r[3]).all()                          # a NaN in row 3 of A
        assert np.isnan(r[20, 11]) and np.isnan(r[20, 13])  # Inf * 0
        assert np.isinf(r[:, 11]).sum() > M // 2            # Inf in B column 11
        assert np.isnan(r[:, 13]).any() and np.isinf(r[:, 13]).any()   # Inf - Inf, and Inf + Inf
    else:
        assert (r[3] == 0).all() and not np.isnan(r).any()   # ReLU sends NaN to 0


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_e4m3_nan_code_propagates(M, N, K):
    spec = _int_spec("nan_e4m3", M, N, K, dtype_in="e4m3")
    # integers in [-4, 4] are e4m3 values: take them as codes with unit scales
    twin = wl.make_inputs(dataclasses.replace(spec, dtype_in="bf16"))
    assert spec.ld("a") == twin.spec.ld("a") and spec.ld("b") == twin.spec.ld("b")
    inputs = wl.Inputs(spec, twin.A.float().to(torch.float8_e4m3fn), twin.B.float().to(torch.float8_e4m3fn))
    inputs = _plant_specials(spec, inputs, nan_code=0x7F)
    _, r = _run_and_compare(spec, inputs)
    assert np.isnan(r[3]).all() and np.isnan(r[:, 11]).all()


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("dtype_d,alpha", [("f16", 1024.0), ("bf16", 2.0 ** 124), ("f32", 2.0 ** 124)])
def test_results_past_the_largest_value_become_infinite(M, N, K, dtype_d, alpha):
    # int4 sums spread over about +-100; alpha pushes those past 64 (f16:
    # 65504) or 16 (bf16 and fp32: 2^128, where the fp32 product itself
    # overflows) beyond the output type's largest finite value
    spec = _int_spec("overflow", M, N, K, dtype_in="f16" if dtype_d == "f16" else "bf16", dtype_d=dtype_d,
                     alpha=alpha)
    inputs = wl.make_inputs(spec)
    _, r = _run_and_compare(spec, inputs)
    assert (r == np.inf).any() and (r == -np.inf).any() and np.isfinite(r).any()


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("dtype_d,alpha,tiny", [("f16", 2.0 ** -30, 2.0 ** -14), ("bf16", 2.0 ** -134, 2.0 ** -126),
                                                ("f32", 2.0 ** -140, 2.0 ** -126)])
def test_subnormal_results_round_to_nearest_even(M, N, K, dtype_d, alpha, tiny):
    # alpha times an integer sum lands below the type's smallest normal value
    # (and for bf16 / fp32 alpha itself is an fp32 subnormal)
    spec = _int_spec("subnormal", M, N, K, dtype_in="f16" if dtype_d == "f16" else "bf16", dtype_d=dtype_d,
                     alpha=alpha)
    inputs = wl.make_inputs(spec)
    _, r = _run_and_compare(spec, inputs)
    sub = (r != 0) & (np.abs(r) < tiny)
    assert sub.mean() > 0.5, "the case does not reach the subnormal range"


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_subnormal_products_are_kept_by_the_tensor_core(M, N, K):
    # bf16 operands 2^-70 * (integers in [-4, 4]): every product is an fp32
    # subnormal, every sum a multiple of 2^-140; fp32 D holds them exactly
    spec = _int_spec("subnormal_products", M, N, K, dtype_d="f32")
    inputs = wl.make_inputs(spec)
    tiny = lambda x: (x.float() * 2.0 ** -70).to(torch.bfloat16)
    inputs = dataclasses.replace(inputs, A=tiny(inputs.A), B=tiny(inputs.B))
    _, r = _run_and_compare(spec, inputs)
    assert ((r != 0) & (np.abs(r) < 2.0 ** -126)).mean() > 0.9


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("dtype_d", ["bf16", "f32"])
def test_negative_zero_results_keep_their_sign(M, N, K, dtype_d):
    spec = _int_spec("neg_zero", M, N, K, dtype_d=dtype_d, alpha=-1.0)
    inputs = wl.make_inputs(spec)
    A = inputs.A.clone()
    for m in range(10):                      # rows 0..9 of A are +0: a zero sum, times -1
        A[m * spec.ld("a"): m * spec.ld("a") + K] = 0.0
    inputs = dataclasses.replace(inputs, A=A)
    g, r = _run_and_compare(spec, inputs)
    assert np.all(np.signbit(r[:10])) and np.all(r[:10] == 0)

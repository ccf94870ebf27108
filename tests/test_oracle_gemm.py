"""Pins the C GEMM oracle to things other than itself (no GPU needed):
exact rational arithmetic on tiny inputs, closed forms, independent codecs
(numpy / torch conversions), an exact integer product, and the fp64 error
bound against a library matmul."""
import itertools
from fractions import Fraction

import numpy as np
import pytest
import torch

from _dtypes import from_bits, to_bits
from _storage import to_storage
from oracle import gemm_ref as g


# ---------------------------------------------------------------- codecs ----
def test_decode_f16_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32)
    want = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([g.decode("f16", int(b)) for b in bits])
    assert np.array_equal(got, want, equal_nan=True)


def test_decode_bf16_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):                    # NaN patterns are part of the sweep
        want = (bits << 16).view(np.float32).astype(np.float64)
    got = np.array([g.decode("bf16", int(b)) for b in bits])
    assert np.array_equal(got, want, equal_nan=True)


def test_decode_e4m3_all_patterns():
    # Torch's float8_e4m3fn is the OCP E4M3 type named by the narrow-precision
    # table on "Technical Documentation: NVIDIA/cutlass".
    bits = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([g.decode("e4m3", int(b)) for b in bits])
    assert np.array_equal(got, want, equal_nan=True)
    assert g.decode("e4m3", 0x7E) == 448.0 and np.isnan(g.decode("e4m3", 0x7F))


def test_decode_f32_random_patterns():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    with np.errstate(invalid="ignore"):                    # NaN patterns are part of the sample
        want = bits.view(np.float32).astype(np.float64)
    got = np.array([g.decode("f32", int(b)) for b in bits])
    assert np.array_equal(got, want, equal_nan=True)


def _hard_doubles(rng, n):
    """Doubles around rounding boundaries of the 16-bit types, plus spread values."""
    base = rng.standard_normal(n) * np.exp2(rng.integers(-30, 20, n))
    # exact midpoints between neighbouring f16 values
    h = rng.integers(0, 0x7BFF, n // 4).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    return np.concatenate([base, (lo + hi) / 2, -(lo + hi) / 2, [65504.0, 65519.99, 65520.0, 1e6, 0.0, -0.0,
                                                                 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]])


def test_encode_f16_matches_numpy():
    rng = np.random.default_rng(1)
    vals = _hard_doubles(rng, 20000)
    with np.errstate(over="ignore"):                   # values past the f16 range are part of the sample
        want = vals.astype(np.float16).view(np.uint16)   # numpy rounds double->half directly (RNE)
    got = np.array([g.encode("f16", float(v)) for v in vals], dtype=np.uint32).astype(np.uint16)
    assert np.array_equal(got, want)


def test_encode_f32_matches_hardware_cast():
    rng = np.random.default_rng(2)
    vals = rng.standard_normal(20000) * np.exp2(rng.integers(-140, 120, 20000))
    want = vals.astype(np.float32).view(np.uint32)
    got = np.array([g.encode("f32", float(v)) for v in vals], dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(got, want)


def test_encode_bf16_matches_torch_on_fp32_values():
    # Values that are exact in fp32, so torch's fp32->bf16 RNE is a single rounding.
    rng = np.random.default_rng(3)
    f = (rng.standard_normal(20000) * np.exp2(rng.integers(-120, 120, 20000))).astype(np.float32)
    hb = rng.integers(0, 0x7F7F, 5000).astype(np.uint32)
    mids = (((hb << 16) | 0x8000).view(np.float32))          # exact bf16 midpoints
    f = np.concatenate([f, mids, -mids])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([g.encode("bf16", float(v)) for v in f.astype(np.float64)], dtype=np.uint32).astype(np.uint16)
    assert np.array_equal(got, want)


def test_encode_roundtrip_and_ties_to_even():
    for dt in ("f16", "bf16"):
        for b in range(0, 1 << 16, 7):
            v = g.decode(dt, b)
            if np.isfinite(v):
                assert g.encode(dt, v) == b or (v == 0 and g.encode(dt, v) in (0, 0x8000))
    # 1 + half an ulp rounds to 1 (even); 1 + 3 half-ulps rounds up to 1 + 2 ulps
    assert g.encode("bf16", 1.0 + 2 ** -8) == 0x3F80
    assert g.encode("bf16", 1.0 + 3 * 2 ** -8) == 0x3F82
    assert g.encode("f16", 2049.0) == 0x6800       # 2048 (even)
    assert g.encode("f16", 2051.0) == 0x6802       # 2052 (even)


# ------------------------------------------------------- brute force -------
def _exact_expected(a, b, c, bias, alpha, beta, scale_a, scale_b, act, bias_per_row):
    """Exact rational D before rounding, from logical matrices (L, M, K) etc."""
    L, M, K = a.shape
    N = b.shape[2]
    out = np.empty((L, M, N), dtype=object)
    s = Fraction(alpha) * Fraction(scale_a) * Fraction(scale_b)
    for l in range(L):
        for m in range(M):
            for n in range(N):
                acc = sum((Fraction(a[l, m, k]) * Fraction(b[l, k, n]) for k in range(K)), Fraction(0))
                t = s * acc
                if beta != 0:
                    t += Fraction(beta) * Fraction(c[l, m, n])
                if bias is not None:
                    t += Fraction(float(bias[l, m if bias_per_row else n]))
                if act == "relu" and t < 0:
                    t = Fraction(0)
                out[l, m, n] = t
    return out


def _round_exact(t, dtype):
    """Reference rounding of exact values that are representable in fp32."""
    f = np.array([float(x) for x in t.reshape(-1)], dtype=np.float64)
    assert np.array_equal(f.astype(np.float32).astype(np.float64), f), "test values must be fp32-exact"
    if dtype == "f32":
        return f.astype(np.float32).view(np.uint32).reshape(t.shape)
    if dtype == "f16":
        return f.astype(np.float16).view(np.uint16).reshape(t.shape)
    return to_bits(f, "bf16").reshape(t.shape)


def _run_oracle(a, b, c, bias, *, op_a, op_b, order_a, order_b, order_cd, dt_in, dt_out,
                alpha=1.0, beta=0.0, scale_a=1.0, scale_b=1.0, act="none", bias_per_row=False, pad=3):
    L, M, K = a.shape
    N = b.shape[2]
    sa, sb = (M, K) if op_a == "N" else (K, M), (K, N) if op_b == "N" else (N, K)
    lda = (sa[1] if order_a == "row" else sa[0]) + pad
    ldb = (sb[1] if order_b == "row" else sb[0]) + pad
    ldc = (N if order_cd == "row" else M) + pad
    abuf, lda, bsa = to_storage(to_bits(a, dt_in).reshape(a.shape), op_a, order_a, lda)
    bbuf, ldb, bsb = to_storage(to_bits(b, dt_in).reshape(b.shape), op_b, order_b, ldb)
    cbuf, bsc = None, 0
    if c is not None:
        cbuf, ldc, bsc = to_storage(to_bits(c, dt_out).reshape(c.shape), "N", order_cd, ldc)
    p = g.make_problem(M, N, K, L, op_a, op_b, order_a, order_b, order_cd, order_cd, lda, ldb, ldc, ldc,
                       bsa, bsb, bsc, bsc, bias.shape[1] if bias is not None else 0,
                       dt_in, dt_in, dt_out, dt_out, alpha, beta, scale_a, scale_b,
                       bias is not None, bias_per_row, act)
    bias_buf = None if bias is None else np.ascontiguousarray(bias.reshape(-1), dtype=np.float32)
    bits, t = g.gemm_rows(p, abuf, bbuf, cbuf, bias_buf, want_t=True)
    return bits.reshape(L, M, N), t.reshape(L, M, N)


LAYOUTS = list(itertools.product("NT", "NT", ("row", "col"), ("row", "col")))


@pytest.mark.parametrize("op_a,op_b,order_a,order_b", LAYOUTS)
def test_bruteforce_layouts_exact(op_a, op_b, order_a, order_b):
    rng = np.random.default_rng(LAYOUTS.index((op_a, op_b, order_a, order_b)))
    for (L, M, N, K) in [(1, 1, 1, 1), (1, 3, 5, 2), (2, 7, 4, 6), (1, 5, 8, 8)]:
        a = rng.integers(-8, 9, (L, M, K)) / 4.0
        b = rng.integers(-8, 9, (L, K, N)) / 4.0
        c = rng.integers(-8, 9, (L, M, N)) / 8.0
        bias = (rng.integers(-16, 17, (L, N)) / 16.0).astype(np.float32)
        for order_cd, dt_in, dt_out, act in [("row", "bf16", "bf16", "relu"), ("col", "f16", "f32", "none"),
                                             ("row", "e4m3", "f16", "none"), ("col", "bf16", "bf16", "none")]:
            alpha, beta = 0.75, -1.5
            bits, t = _run_oracle(a, b, c, bias, op_a=op_a, op_b=op_b, order_a=order_a, order_b=order_b,
                                  order_cd=order_cd, dt_in=dt_in, dt_out=dt_out, alpha=alpha, beta=beta,
                                  act=act)
            exact = _exact_expected(a, b, c, bias, alpha, beta, 1.0, 1.0, act, False)
            assert np.array_equal(t, np.array([float(x) for x in exact.reshape(-1)]).reshape(t.shape))
            assert np.array_equal(bits, _round_exact(exact, dt_out))


def test_bruteforce_scales_and_row_bias():
    rng = np.random.default_rng(5)
    L, M, N, K = 2, 6, 5, 7
    a = rng.integers(-8, 9, (L, M, K)) / 4.0
    b = rng.integers(-8, 9, (L, K, N)) / 4.0
    bias = (rng.integers(-16, 17, (L, M)) / 16.0).astype(np.float32)
    bits, t = _run_oracle(a, b, None, bias, op_a="N", op_b="T", order_a="row", order_b="row", order_cd="row",
                          dt_in="e4m3", dt_out="f32", alpha=2.0, scale_a=0.5, scale_b=0.25,
                          bias_per_row=True)
    exact = _exact_expected(a, b, None, bias, 2.0, 0.0, 0.5, 0.25, "none", True)
    assert np.array_equal(bits, _round_exact(exact, "f32"))


# ------------------------------------------------------- closed forms ------
def _normal_bf16(rng, shape):
    return from_bits(to_bits(rng.standard_normal(shape), "bf16"), "bf16").reshape(shape)


def test_identity_operand_returns_b_exactly():
    rng = np.random.default_rng(6)
    K, N = 40, 24
    a = np.eye(K)[None]
    b = _normal_bf16(rng, (1, K, N))
    bits, _ = _run_oracle(a, b, None, None, op_a="N", op_b="N", order_a="col", order_b="row", order_cd="row",
                          dt_in="bf16", dt_out="bf16")
    assert np.array_equal(bits, to_bits(b, "bf16").reshape(bits.shape))


def test_permutation_reorders_rows_exactly():
    rng = np.random.default_rng(7)
    K, N = 16, 9
    perm = rng.permutation(K)
    a = np.eye(K)[perm][None]
    b = _normal_bf16(rng, (1, K, N))
    bits, _ = _run_oracle(a, b, None, None, op_a="T", op_b="N", order_a="row", order_b="col", order_cd="col",
                          dt_in="bf16", dt_out="f32")
    assert np.array_equal(from_bits(bits, "f32").reshape(bits.shape), b[:, perm, :])


def test_rank_one_k1():
    rng = np.random.default_rng(8)
    M, N = 13, 11
    u, v = _normal_bf16(rng, (1, M, 1)), _normal_bf16(rng, (1, 1, N))
    bits, _ = _run_oracle(u, v, None, None, op_a="N", op_b="N", order_a="row", order_b="row", order_cd="row",
                          dt_in="bf16", dt_out="f32")
    want = (u[0] * v[0]).astype(np.float32)   # exact product in fp64, then one rounding
    assert np.array_equal(from_bits(bits, "f32").reshape(M, N), want.astype(np.float64))


def test_all_ones_gives_k():
    for K in (1, 17, 256, 1000):
        a, b = np.ones((1, 3, K)), np.ones((1, K, 5))
        bits, _ = _run_oracle(a, b, None, None, op_a="N", op_b="T", order_a="row", order_b="col", order_cd="row",
                              dt_in="f16", dt_out="f32")
        assert np.all(from_bits(bits, "f32") == K)


def test_alpha0_beta1_copies_c_and_bias_broadcasts():
    rng = np.random.default_rng(9)
    L, M, N, K = 2, 5, 6, 3
    a, b = _normal_bf16(rng, (L, M, K)), _normal_bf16(rng, (L, K, N))
    c = _normal_bf16(rng, (L, M, N))
    bits, _ = _run_oracle(a, b, c, None, op_a="N", op_b="N", order_a="row", order_b="row", order_cd="col",
                          dt_in="bf16", dt_out="bf16", alpha=0.0, beta=1.0)
    assert np.array_equal(bits, to_bits(c, "bf16").reshape(bits.shape))
    bias = (rng.standard_normal((L, N)) * 0.1).astype(np.float32)
    bits, _ = _run_oracle(a, b, None, bias, op_a="N", op_b="N", order_a="row", order_b="row", order_cd="row",
                          dt_in="bf16", dt_out="bf16", alpha=0.0)
    want = to_bits(np.broadcast_to(bias[:, None, :].astype(np.float64), (L, M, N)), "bf16").reshape(L, M, N)
    assert np.array_equal(bits, want)


def test_relu_masks_exactly_the_negatives():
    rng = np.random.default_rng(10)
    L, M, N, K = 1, 9, 10, 12
    a, b = _normal_bf16(rng, (L, M, K)), _normal_bf16(rng, (L, K, N))
    kw = dict(op_a="N", op_b="T", order_a="row", order_b="row", order_cd="row", dt_in="bf16", dt_out="f32")
    plain, tp = _run_oracle(a, b, None, None, **kw)
    relu, _ = _run_oracle(a, b, None, None, act="relu", **kw)
    vals = from_bits(plain, "f32").reshape(plain.shape)
    want = np.where(tp > 0, vals, 0.0)
    assert np.array_equal(from_bits(relu, "f32").reshape(relu.shape), want)
    assert (tp < 0).any() and (tp > 0).any()


def test_batches_are_independent_slices():
    rng = np.random.default_rng(11)
    L, M, N, K = 3, 7, 5, 9
    a, b = _normal_bf16(rng, (L, M, K)), _normal_bf16(rng, (L, K, N))
    c = _normal_bf16(rng, (L, M, N))
    bias = (rng.standard_normal((L, N)) * 0.1).astype(np.float32)
    kw = dict(op_a="T", op_b="N", order_a="col", order_b="row", order_cd="row", dt_in="bf16", dt_out="bf16",
              alpha=0.5, beta=1.0, act="relu")
    full, _ = _run_oracle(a, b, c, bias, **kw)
    for l in range(L):
        one, _ = _run_oracle(a[l:l + 1], b[l:l + 1], c[l:l + 1], bias[l:l + 1], **kw)
        assert np.array_equal(full[l], one[0])


# ------------------------------------------- exact integer product (C1) ----
def test_tiny_exact_config_matches_integer_matmul():
    # M=N=K=256, fp16 integers in [-4,4], A and B column-major, no transpose,
    # D fp32 column-major: every sum is an integer below 2^24, so the result
    # is exactly the integer matrix product.
    rng = np.random.default_rng(0)
    M = N = K = 256
    a = rng.integers(-4, 5, (1, M, K))
    b = rng.integers(-4, 5, (1, K, N))
    bits, _ = _run_oracle(a.astype(np.float64), b.astype(np.float64), None, None, op_a="N", op_b="N",
                          order_a="col", order_b="col", order_cd="col", dt_in="f16", dt_out="f32", pad=0)
    assert np.array_equal(from_bits(bits, "f32").reshape(M, N), (a[0] @ b[0]).astype(np.float64))


# ------------------------------------------------ fp64 error bound ----------
@pytest.mark.parametrize("op_a,op_b,order_a,order_b", LAYOUTS[::3])
def test_within_fp64_bound_of_library_matmul(op_a, op_b, order_a, order_b):
    rng = np.random.default_rng(12)
    L, M, N, K = 1, 37, 29, 300
    a, b = _normal_bf16(rng, (L, M, K)), _normal_bf16(rng, (L, K, N))
    c = _normal_bf16(rng, (L, M, N))
    bias = (rng.standard_normal((L, N)) * 0.1).astype(np.float32)
    _, t = _run_oracle(a, b, c, bias, op_a=op_a, op_b=op_b, order_a=order_a, order_b=order_b,
                       order_cd="row", dt_in="bf16", dt_out="bf16", alpha=0.5, beta=1.0)
    ref = 0.5 * (a[0] @ b[0]) + c[0] + bias[0].astype(np.float64)[None, :]
    bound = 4 * K * np.finfo(np.float64).eps * (np.abs(a[0]) @ np.abs(b[0]) + np.abs(c[0]) + 1)
    assert np.all(np.abs(t[0] - ref) <= bound)


def test_sampled_rows_equal_full_rows():
    rng = np.random.default_rng(13)
    L, M, N, K = 2, 50, 20, 33
    a, b = _normal_bf16(rng, (L, M, K)), _normal_bf16(rng, (L, K, N))
    kw = dict(op_a="N", op_b="T", order_a="row", order_b="row", order_cd="row", dt_in="bf16", dt_out="bf16")
    full, _ = _run_oracle(a, b, None, None, **kw)
    abuf, lda, bsa = to_storage(to_bits(a, "bf16").reshape(a.shape), "N", "row")
    bbuf, ldb, bsb = to_storage(to_bits(b, "bf16").reshape(b.shape), "T", "row")
    p = g.make_problem(M, N, K, L, "N", "T", "row", "row", "row", "row", lda, ldb, None, None, bsa, bsb)
    rows = np.array([0, 7, M - 1, M + 3, 2 * M - 1])
    part, _ = g.gemm_rows(p, abuf, bbuf, rows=rows)
    assert np.array_equal(part, full.reshape(L * M, N)[rows])


def test_panel_reuse_sees_changed_operand_bytes():
    # The oracle keeps its last decoded B panel; a B rewritten in place (same
    # address, new bytes) must not be served from it.
    rng = np.random.default_rng(14)
    M, N, K = 4, 6, 5
    a, b = _normal_bf16(rng, (1, M, K)), _normal_bf16(rng, (1, K, N))
    abuf, lda, _ = to_storage(to_bits(a, "bf16").reshape(a.shape), "N", "row")
    bbuf, ldb, _ = to_storage(to_bits(b, "bf16").reshape(b.shape), "N", "row")
    p = g.make_problem(M, N, K, 1, "N", "N", "row", "row", "row", "row", lda, ldb, dtype_d="f32")
    first, _ = g.gemm_rows(p, abuf, bbuf)
    again, _ = g.gemm_rows(p, abuf, bbuf)
    assert np.array_equal(first, again)
    bbuf[:] = to_bits(2.0 * b, "bf16").reshape(-1)          # exact doubling, same buffer
    doubled, _ = g.gemm_rows(p, abuf, bbuf)
    assert np.array_equal(from_bits(doubled, "f32"), 2.0 * from_bits(first, "f32"))


# ------------------------------------------------------------------ GELU ----
def _t_of(values, act, dt_out="f32"):
    """Oracle t for a K = 1 problem whose products are exactly `values`."""
    x = np.asarray(values, dtype=np.float64)
    n = x.size
    a = x.reshape(1, 1, n).transpose(0, 2, 1)          # (L=1, M=n, K=1)
    b = np.ones((1, 1, 1))
    _, t = _run_oracle(a, b, None, None, op_a="N", op_b="N", order_a="row", order_b="row", order_cd="row",
                       dt_in="bf16", dt_out=dt_out, act=act)
    return t.reshape(-1)


# Standard normal CDF values as printed in statistical tables (to 16 digits).
PHI = {0.5: 0.6914624612740131, 1.0: 0.8413447460685429, 2.0: 0.9772498680518208,
       3.0: 0.9986501019683699}


def test_gelu_equals_x_times_the_normal_cdf_table():
    xs = sorted(PHI) + [-x for x in sorted(PHI)] + [0.0]
    got = _t_of(xs, "gelu")
    for x, gx in zip(xs, got):
        want = x * PHI[x] if x > 0 else (x * (1.0 - PHI[-x]) if x < 0 else 0.0)
        assert abs(gx - want) <= 2e-15 * max(1.0, abs(x)), (x, gx, want)


def test_gelu_odd_part_and_limits():
    rng = np.random.default_rng(21)
    x = from_bits(to_bits(rng.uniform(0.0, 6.0, 64), "bf16"), "bf16")
    gp, gm = _t_of(x, "gelu"), _t_of(-x, "gelu")
    # x*Phi(x) - (-x)*Phi(-x) = x, since Phi(-x) = 1 - Phi(x)
    assert np.allclose(gp - gm, x, rtol=0, atol=1e-14)
    big = _t_of([8.0, -8.0, 16.0, -16.0], "gelu")
    assert abs(big[0] - 8.0) < 1e-13 and abs(big[1]) < 1e-13
    assert big[2] == 16.0 and abs(big[3]) < 1e-50


def test_gelu_rounds_once_to_the_output_type():
    rng = np.random.default_rng(22)
    x = from_bits(to_bits(rng.standard_normal(40), "bf16"), "bf16")
    a = x.reshape(1, 40, 1)
    bits, t = _run_oracle(a, np.ones((1, 1, 1)), None, None, op_a="N", op_b="N", order_a="row",
                          order_b="row", order_cd="row", dt_in="bf16", dt_out="bf16", act="gelu")
    assert np.array_equal(bits.reshape(-1), to_bits(t.reshape(-1), "bf16"))


# ------------------------------------------------------------ reductions --
def test_reductions_exact_on_integers():
    rng = np.random.default_rng(23)
    L, M, N, K = 2, 5, 7, 6
    a = rng.integers(-4, 5, (L, M, K)).astype(np.float64)
    b = rng.integers(-4, 5, (L, K, N)).astype(np.float64)
    c = rng.integers(-4, 5, (L, M, N)).astype(np.float64)
    bias = rng.integers(-3, 4, (L, N)).astype(np.float32)
    for act in ("none", "relu"):
        _, t = _run_oracle(a, b, c, bias, op_a="N", op_b="T", order_a="col", order_b="row", order_cd="row",
                           dt_in="f16", dt_out="f32", alpha=1.0, beta=1.0, act=act)
        exact = _exact_expected(a, b, c, bias, 1.0, 1.0, 1.0, 1.0, act, False)
        rows = [[sum(exact[l, m, n] for n in range(N)) for m in range(M)] for l in range(L)]
        cols = [[sum(exact[l, m, n] for m in range(M)) for n in range(N)] for l in range(L)]
        amax = [max(abs(exact[l, m, n]) for m in range(M) for n in range(N)) for l in range(L)]
        assert np.array_equal(g.row_sums(t), np.array(rows, dtype=np.float64))
        assert np.array_equal(g.col_sums(t), np.array(cols, dtype=np.float64))
        assert np.array_equal(g.abs_max(t), np.array(amax, dtype=np.float64))


def test_row_and_column_sums_share_the_total():
    rng = np.random.default_rng(24)
    L, M, N, K = 3, 11, 13, 17
    a, b = _normal_bf16(rng, (L, M, K)), _normal_bf16(rng, (L, K, N))
    _, t = _run_oracle(a, b, None, None, op_a="N", op_b="N", order_a="row", order_b="col", order_cd="row",
                       dt_in="bf16", dt_out="f32", act="gelu")
    assert g.row_sums(t).shape == (L, M) and g.col_sums(t).shape == (L, N)
    assert np.allclose(g.row_sums(t).sum(axis=1), g.col_sums(t).sum(axis=1), rtol=1e-13, atol=1e-12)
    assert np.all(g.abs_max(t) >= np.abs(t).reshape(L, -1).max(axis=1))

"""Pins the oracle's NVFP4 path (no GPU): the e2m1 and ue4m3 codecs against
the values the format definitions fix, the nibble order of packed e2m1
storage, exact rational brute force of D = sum_k (A x SFA)(B x SFB) with
16-element scale vectors ("Technical Documentation: NVIDIA/cutlass", "Block
Scaled GEMMs" and "Blackwell Narrow Precision Data Types"), and the special
case that reduces to an e4m3 product.  Also checks the input generator's
e2m1 rounding, which both sides consume."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import gemm_ref as g

# E2M1 values by code, as tabulated by the OCP microscaling specification the
# page's narrow-precision table points to (sign in bit 3)
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decodes_every_code():
    for c in range(16):
        want = E2M1[c & 7] * (-1.0 if c & 8 else 1.0)
        got = g.decode("e2m1", c)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want)


def test_ue4m3_is_e4m3_without_a_sign():
    assert [g.decode("ue4m3", c) for c in (0x38, 0x30, 0x40, 0x7E, 0x01, 0x08, 0x00)] == \
        [1.0, 0.5, 2.0, 448.0, 2.0 ** -9, 2.0 ** -6, 0.0]
    assert math.isnan(g.decode("ue4m3", 0x7F))
    for c in range(0x80):
        x, y = g.decode("ue4m3", c), g.decode("e4m3", c)
        assert (math.isnan(x) and math.isnan(y)) or x == y


def _pack(codes):
    """Flat nibble codes -> bytes, the element of lower index in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1, 2)
    return (c[:, 0] | (c[:, 1] << 4)).astype(np.uint8)


def _pack_sf(codes, pad=0x38):
    L, rows, sfk = codes.shape
    size = ((rows + 127) // 128) * ((sfk + 3) // 4) * 512
    out = np.full(L * size, pad, dtype=np.uint8)
    for l in range(L):
        for r in range(rows):
            for k in range(sfk):
                out[g.sf_index(l, r, k, rows, sfk)] = codes[l, r, k]
    return out


def _ue4m3_fraction(c):
    e, m = (c >> 3) & 15, c & 7
    return Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def _run(ca, cb, sfa, sfb, L, M, N, K, kmajor_a=("N", "row"), kmajor_b=("N", "col"), sf_vec=16, dt="e2m1",
         pad=0x38):
    """ca: (L, M, K), cb: (L, N, K) element codes; A and B K-contiguous."""
    op_a, order_a = kmajor_a
    op_b, order_b = kmajor_b
    lda = ldb = K
    # K-contiguous storage of rows of op(A) and columns of op(B)
    a_store = np.asarray(ca).reshape(-1)
    b_store = np.asarray(cb).reshape(-1)
    if dt == "e2m1":
        a_store, b_store = _pack(a_store), _pack(b_store)
    p = g.make_problem(M, N, K, L, op_a, op_b, order_a, order_b, "row", "row", lda, ldb, N, N,
                       M * K if L > 1 else 0, N * K if L > 1 else 0, 0, M * N if L > 1 else 0, 0,
                       dt, dt, "f32", "f32", sf_vec=sf_vec)
    sa = _pack_sf(sfa, pad) if sf_vec else None
    sb = _pack_sf(sfb, pad) if sf_vec else None
    bits, t = g.gemm_rows(p, a_store, b_store, want_t=True, sfa=sa, sfb=sb)
    return t.reshape(L, M, N)


@pytest.mark.parametrize("layout", ["NN_row_col", "TT_col_row"])
@pytest.mark.parametrize("K", [48, 40])          # three full factor blocks; a last block of 8 elements
def test_nvfp4_bruteforce_exact(layout, K):
    rng = np.random.default_rng(41)
    L, M, N = 2, 5, 6
    ca = rng.integers(0, 16, (L, M, K))
    cb = rng.integers(0, 16, (L, N, K))
    sfk = (K + 15) // 16
    sfa = rng.integers(0x20, 0x50, (L, M, sfk))
    sfb = rng.integers(0x20, 0x50, (L, N, sfk))
    kw = {} if layout == "NN_row_col" else {"kmajor_a": ("T", "col"), "kmajor_b": ("T", "row")}
    t = _run(ca, cb, sfa, sfb, L, M, N, K, **kw)
    e2m1 = lambda c: Fraction(E2M1[c & 7]) * (-1 if c & 8 else 1)
    for l in range(L):
        for m in range(M):
            for n in range(N):
                want = sum(e2m1(int(ca[l, m, k])) * _ue4m3_fraction(int(sfa[l, m, k // 16])) *
                           e2m1(int(cb[l, n, k])) * _ue4m3_fraction(int(sfb[l, n, k // 16])) for k in range(K))
                assert Fraction(t[l, m, n]) == want


def test_swapped_nibbles_change_the_result():
    # a reader of the high nibble first would see a different product
    rng = np.random.default_rng(42)
    L, M, N, K = 1, 3, 3, 32
    ca, cb = rng.integers(1, 8, (L, M, K)), rng.integers(1, 8, (L, N, K))
    ones = lambda R: np.full((L, R, 2), 0x38)
    t = _run(ca, cb, ones(M), ones(N), L, M, N, K)
    swapped = ca.reshape(L, M, K // 2, 2)[..., ::-1].reshape(L, M, K)
    t_sw = _run(swapped, cb, ones(M), ones(N), L, M, N, K)
    assert not np.array_equal(t, t_sw)


def test_unit_factors_reduce_to_the_e4m3_product_of_the_same_values():
    # every e2m1 value is exact in e4m3; with factors 1.0 the block-scaled
    # e2m1 GEMM equals the plain e4m3 GEMM of the same numbers
    rng = np.random.default_rng(43)
    L, M, N, K = 1, 20, 24, 96
    ca, cb = rng.integers(0, 16, (L, M, K)), rng.integers(0, 16, (L, N, K))
    t = _run(ca, cb, np.full((L, M, 6), 0x38), np.full((L, N, 6), 0x38), L, M, N, K)
    e4 = {}
    for c in range(16):
        v = E2M1[c & 7] * (-1.0 if c & 8 else 1.0)
        code = [x for x in range(256) if g.decode("e4m3", x) == v and math.copysign(1, g.decode("e4m3", x)) ==
                math.copysign(1, v)][0]
        e4[c] = code
    ea = np.vectorize(e4.get)(ca).astype(np.uint8)
    eb = np.vectorize(e4.get)(cb).astype(np.uint8)
    t_e4 = _run(ea, eb, None, None, L, M, N, K, sf_vec=0, dt="e4m3")
    assert np.array_equal(t, t_e4)


def test_padding_factors_past_k_are_not_read():
    rng = np.random.default_rng(44)
    L, M, N, K = 1, 4, 4, 36                       # factors 0..2 real, the fourth slot is padding
    ca, cb = rng.integers(0, 16, (L, M, K)), rng.integers(0, 16, (L, N, K))
    sfa, sfb = rng.integers(0x30, 0x41, (L, M, 3)), rng.integers(0x30, 0x41, (L, N, 3))
    t = _run(ca, cb, sfa, sfb, L, M, N, K, pad=0x7F)     # NaN padding
    assert np.all(np.isfinite(t))


def test_generator_e2m1_rounding_ties_to_even_and_saturates():
    from dense_gemm_epilogue_sm_gb300 import workloads as wl
    v = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.3, -5.1, 0.0, 6.0, 1e9])
    codes = wl._encode_e2m1(v).tolist()
    got = [g.decode("e2m1", c) for c in codes]
    assert got == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, -0.5, -6.0, 0.0, 6.0, 6.0]
    grid = torch.tensor([E2M1[c & 7] * (-1.0 if c & 8 else 1.0) for c in range(16)])
    back = wl._encode_e2m1(grid).tolist()
    assert [c if c != 8 else 0 for c in back] == [c if c != 8 else 0 for c in range(16)]


def test_generated_nvfp4_inputs_dequantise_close_to_their_source():
    from dense_gemm_epilogue_sm_gb300 import workloads as wl
    gen = torch.Generator().manual_seed(5)
    x = torch.randn(1, 8, 64, generator=gen)
    q, sf, gs = wl._nv_quantise(x)
    deq = torch.tensor([[g.decode("e2m1", int(c)) for c in row] for row in q[0]])
    scale = torch.tensor([[g.decode("ue4m3", int(c)) for c in row] for row in sf[0]]).repeat_interleave(16, dim=1)
    deq = deq * scale * gs
    blk_amax = x[0].abs().view(8, 4, 16).amax(dim=2).repeat_interleave(16, dim=1)
    # half the widest e2m1 step (2 of 6) of the block's range, plus the factor's own rounding
    assert torch.all((deq - x[0]).abs() <= blk_amax * (1.0 / 6.0 + 1.0 / 16.0) + 1e-6)


# ------------------------------------------------------- NVFP4 output ----
def test_e2m1_encoder_round_trips_ties_to_even_and_saturates():
    vals = np.array([g.decode("e2m1", c) for c in range(16)])
    assert g.encode_e2m1(vals).tolist() == list(range(16))          # -0 included (code 8)
    # halfway points go to the even code; 6 and beyond saturate
    got = g.encode_e2m1(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.5, 7.0, 1e9, -1e9])).tolist()
    assert got == [0, 2, 2, 4, 4, 6, 6, 7, 7, 7, 15]
    assert g.encode_e2m1(np.array([0.2, 0.3, 2.9, 3.1])).tolist() == [0, 1, 5, 5]


def test_nv_output_factor_and_elements_follow_the_rule():
    t = np.zeros((3, 40))
    t[0, :16] = np.linspace(-6.0, 6.0, 16)          # amax 6, g = 1: factor 1.0 (0x38), elements e2m1(t)
    t[0, 16:32] = 6.0 * 448 * 3                     # amax/6 = 1344 saturates to 448 (0x7E); elements 18 -> 6
    t[0, 32:] = 0.0                                 # zeros: factor 0, elements 0
    t[1, 3] = np.nan                                # a NaN: factor 0x7F, elements 0
    t[2, :] = 0.75                                  # amax/6 = 0.125 = 2^-3 exactly (0x20); elements 6.0
    codes, q = g.nv_quantise_rows(t, 1.0)
    assert codes.shape == (3, 3) and q.shape == (3, 40)
    assert codes[0].tolist() == [0x38, 0x7E, 0x00]
    assert q[0, :16].tolist() == g.encode_e2m1(t[0, :16]).tolist()
    assert np.all(q[0, 16:32] == 7) and np.all(q[0, 32:] == 0)
    assert codes[1, 0] == 0x7F and np.all(q[1, :16] == 0) and codes[1, 1] == 0
    assert codes[2].tolist() == [0x20, 0x20, 0x20] and np.all(q[2] == 7)


def _rne_brute(num, den, grid):
    """Nearest grid value to the exact rational num / den, ties to the even
    index, saturating: a scan over the whole grid in exact arithmetic."""
    x = Fraction(num) / Fraction(den)
    best, best_d = 0, None
    for i, v in enumerate(grid):
        d = abs(x - Fraction(v))
        if best_d is None or d < best_d or (d == best_d and i % 2 == 0):
            best, best_d = i, d
    return best


def test_rne_quotient_equals_exact_rational_rounding():
    rng = np.random.default_rng(47)
    e2m1 = np.array([g.decode("e2m1", c) for c in range(8)])
    e4m3 = np.array([g.decode("e4m3", c) for c in range(0x7F)])
    cases = []
    for _ in range(400):
        gs = float(np.float32(rng.uniform(0.01, 3.0)))
        f = e4m3[rng.integers(1, 0x7F)]
        den = f * gs
        mid = rng.choice((e2m1[:-1] + e2m1[1:]) / 2)
        # exact ties, the nearest doubles on either side of them, and random quotients
        tie = mid * den
        for num in (tie, np.nextafter(tie, 0), np.nextafter(tie, np.inf), rng.uniform(0, 8) * den):
            cases.append((num, den, e2m1))
        den6 = 6.0 * gs
        mid4 = rng.choice((e4m3[:-1] + e4m3[1:]) / 2)
        for num in (mid4 * den6, np.nextafter(mid4 * den6, np.inf), rng.uniform(0, 500) * den6):
            cases.append((num, den6, e4m3))
    for num, den, grid in cases:
        got = int(g.rne_quotient(np.array([num]), np.array([den]), grid)[0])
        assert got == _rne_brute(num, den, grid), (num, den)


def test_nv_output_rounds_the_exact_quotient_at_ties():
    # g = 0.25, factor 144 (0x6E... e4m3 144 = 1.125 * 2^7): factor * g = 36, and t = 9
    # gives the quotient 0.25 exactly, halfway between 0 and 0.5: the even code 0.
    # t = 27 gives 0.75 exactly: halfway between 0.5 (code 1) and 1.0 (code 2) -> 2.
    amax = 144 * 6 * 0.25                           # the block's factor is exactly 144
    t = np.zeros((1, 16))
    t[0, :4] = [amax, 9.0, 27.0, -9.0]
    codes, q = g.nv_quantise_rows(t, 0.25)
    assert g.decode("e4m3", int(codes[0, 0])) == 144.0
    assert q[0, 1] == 0 and q[0, 2] == 2 and (q[0, 3] & 7) == 0
    # the nearest doubles past the ties round away from them
    t[0, 1] = np.nextafter(9.0, 10.0)
    t[0, 2] = np.nextafter(27.0, 0.0)
    _, q = g.nv_quantise_rows(t, 0.25)
    assert q[0, 1] == 1 and q[0, 2] == 1


def test_nv_output_global_scale_is_a_pure_rescaling():
    rng = np.random.default_rng(45)
    t = rng.normal(size=(4, 64)) * 3.0
    c1, q1 = g.nv_quantise_rows(t, 1.0)
    c2, q2 = g.nv_quantise_rows(t * 2.0 ** 7, 2.0 ** 7)   # a power of two scales every quotient exactly
    assert np.array_equal(c1, c2) and np.array_equal(q1, q2)


def test_nv_output_dequantises_within_half_a_step():
    rng = np.random.default_rng(46)
    t = rng.normal(size=(6, 96)) * np.exp2(rng.integers(-3, 4, (6, 1)))
    gs = float(np.abs(t).max()) / (448.0 * 6.0)      # the tensor's global scale: no factor saturates
    codes, q = g.nv_quantise_rows(t, gs)
    fac = np.array([[g.decode("e4m3", int(c)) for c in row] for row in codes]).repeat(16, axis=1)[:, :96]
    dq = np.array([[g.decode("e2m1", int(c)) for c in row] for row in q]) * fac * gs
    amax = np.abs(t).reshape(6, 6, 16).max(axis=2).repeat(16, axis=1)
    # one e2m1 step is at most 2 at the top of the range (4 -> 6) in units of
    # factor * g ~ amax / 6; the factor's own rounding adds at most 1/16
    assert np.all(np.abs(dq - t) <= amax * (1.0 / 6.0) * (1 + 1.0 / 16.0) + 1e-12)

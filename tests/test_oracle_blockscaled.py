"""Pins the oracle's block-scaled GEMM (no GPU): the ue8m0 scale-factor codec
against exact powers of two, the scale-factor index against the byte order
stated on "Technical Documentation: NVIDIA/cutlass", "Scale Factor Layouts",
exact rational brute force of D = sum_k (A x SFA)(B x SFB) on small inputs,
and the closed forms where all scale factors are one or constant."""
import dataclasses
import math
from fractions import Fraction

import numpy as np
import pytest

from _dtypes import from_bits, to_bits
from _storage import to_storage
from oracle import gemm_ref as g


def test_ue8m0_decodes_to_powers_of_two_and_nan():
    for e in range(255):
        assert g.decode("ue8m0", e) == math.ldexp(1.0, e - 127)
    assert math.isnan(g.decode("ue8m0", 255))


def test_scale_factor_index_follows_the_stated_byte_order():
    rows, sfk = 300, 10                     # 3 blocks of 128 rows, ceil(10/4) = 3 blocks of 4 factors
    idx = lambda l, r, k: g.sf_index(l, r, k, rows, sfk)
    # "M0SF0 to M0SF3, M32SF0 to M32SF3, M64SF0 to M64SF3, and M96SF0 to
    # M96SF3 are stored consecutively"
    order = [(0, k) for k in range(4)] + [(32, k) for k in range(4)] + [(64, k) for k in range(4)] + \
            [(96, k) for k in range(4)] + [(1, k) for k in range(4)]
    assert [idx(0, r, k) for r, k in order] == list(range(20))
    assert idx(0, 127, 3) == 511                     # the basic block is 512 bytes
    # blocks follow each other K-major: the next 4 factors of the same rows,
    # then the next 128 rows
    assert idx(0, 0, 4) == 512 and idx(0, 0, 8) == 1024 and idx(0, 128, 0) == 3 * 512
    assert idx(1, 0, 0) == 3 * 3 * 512               # one tensor per batch
    seen = {idx(0, r, k) for r in range(384) for k in range(12)}
    assert seen == set(range(3 * 3 * 512))           # a bijection onto the padded tensor


def _pack_sf(codes, pad=127):
    """(L, rows, sfk) ue8m0 codes -> byte tensor; unused bytes hold `pad`."""
    L, rows, sfk = codes.shape
    size = ((rows + 127) // 128) * ((sfk + 3) // 4) * 512
    out = np.full(L * size, pad, dtype=np.uint8)
    for l in range(L):
        for r in range(rows):
            for k in range(sfk):
                out[g.sf_index(l, r, k, rows, sfk)] = codes[l, r, k]
    return out


def _e4m3(rng, shape, scale=1.0):
    return from_bits(to_bits(rng.uniform(-scale, scale, shape), "e4m3"), "e4m3").reshape(shape)


def _run(a, b, sfa_codes, sfb_codes, *, op_a="N", op_b="N", order_a="row", order_b="col", sf_vec=32,
         dt_out="f32", pad=127):
    L, M, K = a.shape
    N = b.shape[2]
    sa, sb = (M, K) if op_a == "N" else (K, M), (K, N) if op_b == "N" else (N, K)
    abuf, lda, bsa = to_storage(to_bits(a, "e4m3").reshape(a.shape), op_a, order_a,
                                sa[1] if order_a == "row" else sa[0])
    bbuf, ldb, bsb = to_storage(to_bits(b, "e4m3").reshape(b.shape), op_b, order_b,
                                sb[1] if order_b == "row" else sb[0])
    ldd = N
    p = g.make_problem(M, N, K, L, op_a, op_b, order_a, order_b, "row", "row", lda, ldb, ldd, ldd,
                       bsa, bsb, 0, M * N if L > 1 else 0, 0, "e4m3", "e4m3", dt_out, dt_out, sf_vec=sf_vec)
    sfa = _pack_sf(sfa_codes, pad) if sf_vec else None
    sfb = _pack_sf(sfb_codes, pad) if sf_vec else None
    bits, t = g.gemm_rows(p, abuf, bbuf, want_t=True, sfa=sfa, sfb=sfb)
    return bits.reshape(L, M, N), t.reshape(L, M, N)


@pytest.mark.parametrize("op_a,op_b,order_a,order_b", [("N", "N", "row", "col"), ("T", "N", "row", "row"),
                                                       ("N", "T", "col", "col"), ("T", "T", "col", "row")])
def test_block_scaled_bruteforce_exact(op_a, op_b, order_a, order_b):
    rng = np.random.default_rng(31)
    L, M, N, K = 2, 5, 6, 96
    a, b = _e4m3(rng, (L, M, K), 8), _e4m3(rng, (L, K, N), 8)
    sfa = rng.integers(120, 135, (L, M, K // 32))
    sfb = rng.integers(120, 135, (L, N, K // 32))
    _, t = _run(a, b, sfa, sfb, op_a=op_a, op_b=op_b, order_a=order_a, order_b=order_b)
    for l in range(L):
        for m in range(M):
            for n in range(N):
                want = sum((Fraction(a[l, m, k]) * Fraction(2) ** int(sfa[l, m, k // 32] - 127)) *
                           (Fraction(b[l, k, n]) * Fraction(2) ** int(sfb[l, n, k // 32] - 127)) for k in range(K))
                assert Fraction(t[l, m, n]) == want


def test_unit_scale_factors_reduce_to_the_plain_product():
    rng = np.random.default_rng(32)
    L, M, N, K = 1, 40, 36, 160
    a, b = _e4m3(rng, (L, M, K), 4), _e4m3(rng, (L, K, N), 4)
    ones_a, ones_b = np.full((L, M, K // 32), 127), np.full((L, N, K // 32), 127)
    bits_s, t_s = _run(a, b, ones_a, ones_b)
    bits_p, t_p = _run(a, b, None, None, sf_vec=0)
    assert np.array_equal(t_s, t_p) and np.array_equal(bits_s, bits_p)


def test_constant_scale_factors_scale_the_product_exactly():
    rng = np.random.default_rng(33)
    L, M, N, K = 1, 17, 19, 128
    a, b = _e4m3(rng, (L, M, K), 4), _e4m3(rng, (L, K, N), 4)
    _, t_p = _run(a, b, None, None, sf_vec=0)
    _, t_s = _run(a, b, np.full((L, M, K // 32), 127 + 5), np.full((L, N, K // 32), 127 - 9))
    assert np.array_equal(t_s, t_p * 2.0 ** (5 - 9))


def test_k_not_a_multiple_of_the_block_reads_only_real_factors():
    # K = 80: the third factor of each row covers 16 real elements; the
    # padding factors (code 255 = NaN here) must not be read
    rng = np.random.default_rng(34)
    L, M, N, K = 1, 3, 4, 80
    a, b = _e4m3(rng, (L, M, K), 2), _e4m3(rng, (L, K, N), 2)
    sfa, sfb = rng.integers(124, 131, (L, M, 3)), rng.integers(124, 131, (L, N, 3))
    _, t = _run(a, b, sfa, sfb, pad=255)
    want = np.einsum("lmk,lkn->lmn", a * 2.0 ** (np.repeat(sfa, 32, axis=2)[:, :, :K] - 127),
                     b * 2.0 ** (np.repeat(sfb, 32, axis=2)[:, :, :K].transpose(0, 2, 1) - 127))
    assert np.all(np.isfinite(t)) and np.allclose(t, want, rtol=1e-14, atol=0)


def test_input_generator_layout_agrees_with_the_oracle_index():
    # the workload generator packs factors with its own code; both follow the page
    from dense_gemm_epilogue_sm_gb300 import workloads as wl
    for L, rows, sfk in [(1, 5, 3), (2, 300, 10), (1, 129, 4)]:
        off, per = wl._sf_offsets(L, rows, sfk)
        want = [[[g.sf_index(l, r, f, rows, sfk) for f in range(sfk)] for r in range(rows)] for l in range(L)]
        assert off.tolist() == want
        assert per == ((rows + 127) // 128) * ((sfk + 3) // 4) * 512


def test_generated_mx_inputs_dequantise_close_to_their_source():
    from dense_gemm_epilogue_sm_gb300 import workloads as wl
    spec = wl.Spec("mx_small", 40, 36, 200, dtype_in="e4m3", block_scale="mx", seed=5)
    inputs = wl.make_inputs(spec)
    assert inputs.extras["sfa"].dtype == inputs.extras["sfb"].dtype
    p = g.problem_from_spec(spec, inputs)
    p.sf_vec = 32
    bits, t = g.gemm_rows(p, inputs.A, inputs.B, want_t=True, sfa=inputs.extras["sfa"].numpy(),
                          sfb=inputs.extras["sfb"].numpy())
    assert np.all(np.isfinite(t)) and np.abs(t).max() > 0


# ------------------------------------------------- block-scaled output ----
def test_e4m3_encoder_round_trips_saturates_and_ties_to_even():
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = np.array([g.decode("e4m3", c) for c in finite])
    codes = g.encode_e4m3(vals)
    assert [int(c) for c in codes] == finite                      # every finite code, -0 included
    # halfway between 1.0 (0x38) and 1.125 (0x39) goes to the even code 0x38;
    # halfway between 1.125 and 1.25 (0x3A) goes to 0x3A
    assert g.encode_e4m3(np.array([1.0625, 1.1875])).tolist() == [0x38, 0x3A]
    assert g.encode_e4m3(np.array([448.0, 464.0, 1e9, -1e9, np.inf])).tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0x7E]
    assert g.encode_e4m3(np.array([np.nan])).tolist() == [0x7F]
    assert g.encode_e4m3(np.array([2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10])).tolist() == [0x01, 0x00, 0x02]


def test_mx_output_factor_follows_the_shared_exponent_rule():
    t = np.zeros((3, 70))
    t[0, :32] = np.linspace(-3.0, 3.0, 32)              # amax 3: floor(log2 3) - 8 = -7 -> code 120
    t[0, 32:64] = 448.0 * 4                             # amax 1792 = 448 * 2^2: code 127 + 10 - 8
    t[0, 64:] = 0.0                                     # all zero: code 0
    t[1, 5] = np.nan                                    # a NaN: code 255, NaN elements
    t[2, :] = 500.0                                     # 500 / 2^0 saturates to 448
    codes, q = g.mx_quantise_rows(t)
    assert codes.shape == (3, 3) and codes[0].tolist() == [120, 129, 0]
    assert codes[1, 0] == 255 and np.all(q[1, :32] == 0x7F) and codes[1, 1] == 0
    assert codes[2].tolist() == [127, 127, 127] and np.all(q[2] == 0x7E)
    dq = np.array([g.decode("e4m3", int(c)) for c in q[0, :32]]) * 2.0 ** (int(codes[0, 0]) - 127)
    assert np.array_equal(dq, np.array([g.decode("e4m3", int(c)) for c in g.encode_e4m3(t[0, :32] * 128)]) / 128)
    assert np.all(np.abs(dq - t[0, :32]) <= 2.0 ** -4 * np.abs(t[0, :32]) + 2.0 ** -16)
    dq1 = np.array([g.decode("e4m3", int(c)) for c in q[0, 32:64]]) * 2.0 ** (int(codes[0, 1]) - 127)
    assert np.all(dq1 == 1792.0)


def test_grouped_generator_places_each_groups_factors_in_whole_blocks():
    # grouped block-scaled A: group g's row r has its factors in row
    # 128 * (blocks of the groups before) + r of one basic-block tensor,
    # checked against the oracle's own index function
    import torch
    from dense_gemm_epilogue_sm_gb300 import workloads as wl
    for fmt, dt, sv in (("mx", "e4m3", 32), ("nv", "e2m1", 16)):
        spec = wl.Spec("grp", 700, 64, 96, groups=4, group_sizes=(130, 0, 1, 500), dtype_in=dt, block_scale=fmt,
                       dist="int4", seed=9)
        gen = torch.Generator().manual_seed(spec.seed)
        rows = wl.group_rows_of(spec, gen)                  # explicit sizes: no draws
        pr = wl.grouped_sfa_rows(spec, rows).tolist()
        assert pr[:130] == list(range(130)) and pr[130] == 256 and pr[131:631] == list(range(384, 884))
        one = dataclasses.replace(spec, groups=0, group_sizes=(), batch=1)
        _, codes, _ = wl._bs_operand(one, gen, 1, spec.M)     # the generator's first draws: A's factors
        sfa = wl.make_inputs(spec).extras["sfa"].numpy()
        sfk = (spec.K + sv - 1) // sv
        r_pad = 128 * ((spec.M + 127) // 128 + spec.groups)
        assert sfa.size == (r_pad // 128) * ((sfk + 3) // 4) * 512
        for r in range(631):                                   # every covered row
            got = [int(sfa[g.sf_index(0, pr[r], f, r_pad, sfk)]) for f in range(sfk)]
            assert got == codes[0, r].tolist()
        # rows between groups are padding: factor 1.0
        for r in list(range(130, 256, 7)) + list(range(257, 384, 11)):
            assert all(int(sfa[g.sf_index(0, r, f, r_pad, sfk)]) == wl.SF_ONE[fmt] for f in range(sfk))

"""Grouped GEMM on the GPU (gemm_grouped_create / gemm_grouped_run) against
the oracle.

Each group is a plain GEMM over its rows of A and D with its own B and bias,
so the oracle computes group g as one problem (the whole A, B_g, bias_g)
restricted to the group's rows.  Rows that no group covers must keep the
canary pattern, and so must every element outside D.  Offsets live in device
memory; out-of-range or decreasing offsets are clamped by the kernel, which
the clamping case checks against the clamped reading."""
import dataclasses

import numpy as np
import pytest
import torch

import _harness as H
import dense_gemm_epilogue_sm_gb300 as g
from dense_gemm_epilogue_sm_gb300 import workloads as wl
from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec
from oracle import gemm_ref

pytestmark = pytest.mark.gpu


def _clamped(rows, M):
    """The documented reading of the offsets: each clamped to [0, M], group g
    from the running maximum of offsets 0..g to that of offsets 0..g+1."""
    c = [min(max(int(r), 0), M) for r in rows]
    run = [c[0]]
    for x in c[1:]:
        run.append(max(run[-1], x))
    return [(run[i], run[i + 1]) for i in range(len(rows) - 1)]


def _run(spec, inputs, rows=None, op=None, repeat=1):
    dev = torch.device("cuda", 0)
    op = op or GemmOp(desc_from_spec(spec), groups=spec.groups)
    A, B = inputs.A.to(dev), inputs.B.to(dev)
    C = inputs.C.to(dev) if inputs.C is not None else None
    bias = inputs.bias.to(dev) if inputs.bias is not None else None
    gr = (inputs.extras["group_rows"] if rows is None else rows).to(dev)
    D = H.canary_buffer(spec)
    for _ in range(repeat):
        op.run_grouped(A, B, C, D, gr, bias)
    op.check()
    torch.cuda.synchronize()
    return H.bits_of_tensor(D.cpu()), op


def _oracle_group(spec, inputs, g_, r0, r1, b_stride=None):
    """Oracle rows [r0, r1) of group g_: the whole A with B_g and bias_g."""
    per_b = spec.matrix_elems("b") if b_stride is None else b_stride
    sub = dataclasses.replace(spec, groups=0, group_sizes=())
    B = inputs.B[g_ * per_b: g_ * per_b + spec.matrix_elems("b")].contiguous()
    bias = None if inputs.bias is None else inputs.bias[g_ * spec.N:(g_ + 1) * spec.N].contiguous()
    sub_in = wl.Inputs(sub, inputs.A, B, inputs.C, bias, inputs.scale_a, inputs.scale_b)
    bits, _ = gemm_ref.run_spec_rows(sub, sub_in, rows=np.arange(r0, r1))
    return sub, sub_in, bits


def _check(spec, inputs, bits, ranges, exact=False, b_stride=None):
    assert H.untouched_outside(spec, bits), "write outside the logical D"
    d = H.logical_d(spec, bits).reshape(spec.M, spec.N)
    covered = np.zeros(spec.M, dtype=bool)
    for g_, (r0, r1) in enumerate(ranges):
        if r1 <= r0:
            continue
        covered[r0:r1] = True
        sub, sub_in, ref = _oracle_group(spec, inputs, g_, r0, r1, b_stride)
        _compare_rows(sub, sub_in, d[r0:r1], ref, exact)
    # rows no group covers keep the canary
    assert np.all(d[~covered].astype(np.uint64) == H.CANARY[spec.dtype_d]), "a row outside every group was written"


def _compare_rows(sub, sub_in, got_bits, ref_bits, exact):
    if exact:
        assert np.array_equal(got_bits.astype(np.uint64), ref_bits.astype(np.uint64)), "not bit-exact"
        return
    got = H.from_bits(got_bits, sub.dtype_d).reshape(got_bits.shape)
    ref = H.from_bits(ref_bits, sub.dtype_d).reshape(ref_bits.shape)
    assert np.isfinite(got).all(), "non-finite output (unwritten element?)"
    tol = H.tolerance(sub, sub_in, ref)
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"{int((err > tol).sum())} elements out of tolerance, worst {np.max(err - tol)}"


SPECS = [
    # CTA pairs (>= 64 pair tiles of the whole): ragged groups, an empty one, a one-row one, C, bias, ReLU
    wl.Spec("grp_pair_ragged_fused", 5000, 1000, 520, groups=6, group_sizes=(700, 0, 1, 1299, 2000, 1000),
            alpha=0.5, beta=1.0, act="relu", bias="col", seed=131, pad=8),
    # one CTA: few tiles; fp16 in, fp32 out, GELU
    wl.Spec("grp_single_f32_gelu", 900, 384, 256, groups=3, group_sizes=(100, 250, 550), dtype_in="f16",
            dtype_d="f32", act="gelu", seed=132),
    # e4m3 operands, B transposed in storage (still K-contiguous), rows left over past the last group
    wl.Spec("grp_e4m3_tail_uncovered", 3000, 512, 1024, groups=4, group_sizes=(257, 1000, 3, 1500),
            dtype_in="e4m3", op_b="T", order_b="row", dist="uniform1", seed=133),
    # A stored transposed (op T, column-major: K-contiguous), many small groups
    wl.Spec("grp_many_small_at", 2048, 640, 384, groups=40, op_a="T", order_a="col", seed=134),
    # drawn group sizes, pair tiles, N ragged
    wl.Spec("grp_drawn_pair", 8192, 1100, 512, groups=12, bias="col", seed=135),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_grouped_matches_oracle(spec):
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs)
    rows = inputs.extras["group_rows"].tolist()
    _check(spec, inputs, bits, _clamped(rows, spec.M))
    op.close()


def test_grouped_integer_sums_bit_exact():
    spec = wl.Spec("grp_int", 4000, 768, 1024, groups=5, group_sizes=(1000, 129, 0, 2000, 871), dtype_in="f16",
                   dtype_d="f32", dist="int4", seed=136)
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs, repeat=2)
    _check(spec, inputs, bits, _clamped(inputs.extras["group_rows"].tolist(), spec.M), exact=True)
    op.close()


def test_offsets_are_clamped_and_nothing_outside_is_written():
    spec = wl.Spec("grp_clamp", 1500, 256, 256, groups=4, group_sizes=(1, 1, 1, 1), seed=137)
    inputs = wl.make_inputs(spec)
    rows = torch.tensor([-5, 100, 50, 3000, 4000], dtype=torch.int64)      # negative, decreasing, past M
    bits, op = _run(spec, inputs, rows=rows)
    ranges = _clamped(rows.tolist(), spec.M)
    assert ranges == [(0, 100), (100, 100), (100, 1500), (1500, 1500)]
    _check(spec, inputs, bits, ranges)
    op.close()


def test_offsets_written_on_the_device_and_new_offsets_on_the_same_handle():
    spec = wl.Spec("grp_device_offsets", 3000, 384, 320, groups=3, group_sizes=(1000, 1000, 1000), beta=1.0,
                   seed=138)
    inputs = wl.make_inputs(spec)
    dev = torch.device("cuda", 0)
    op = GemmOp(desc_from_spec(spec), groups=spec.groups)
    A, B, C = inputs.A.to(dev), inputs.B.to(dev), inputs.C.to(dev)
    for sizes in ((1000, 1000, 1000), (17, 2900, 83), (0, 0, 3000)):
        # the offsets come from a device computation on the same stream
        counts = torch.tensor(sizes, dtype=torch.int64, device=dev)
        gr = torch.cat([torch.zeros(1, dtype=torch.int64, device=dev), torch.cumsum(counts, 0)])
        D = H.canary_buffer(spec)
        op.run_grouped(A, B, C, D, gr)
        op.check()
        bits = H.bits_of_tensor(D.cpu())
        _check(spec, inputs, bits, _clamped(gr.cpu().tolist(), spec.M))
    op.close()


def test_one_b_for_every_group():
    spec = wl.Spec("grp_shared_b", 2500, 512, 256, groups=3, group_sizes=(800, 900, 800), seed=139)
    inputs = wl.make_inputs(spec)
    desc = desc_from_spec(spec)
    desc.stride_b = 0
    op = GemmOp(desc, groups=spec.groups)
    bits, _ = _run(spec, inputs, op=op)
    _check(spec, inputs, bits, _clamped(inputs.extras["group_rows"].tolist(), spec.M), b_stride=0)
    op.close()


def test_grouped_full_size_sampled_rows():
    spec = wl.get("grouped_16x_bf16")
    inputs = wl.make_inputs(spec)
    bits, op = _run(spec, inputs)
    d = H.logical_d(spec, bits).reshape(spec.M, spec.N)
    rows = inputs.extras["group_rows"].tolist()
    rng = np.random.default_rng(5)
    for g_ in range(spec.groups):
        r0, r1 = rows[g_], rows[g_ + 1]
        pick = np.unique(np.concatenate([[r0, r1 - 1], rng.integers(r0, r1, 6)]))
        sub = dataclasses.replace(spec, groups=0, group_sizes=())
        per = spec.matrix_elems("b")
        sub_in = wl.Inputs(sub, inputs.A, inputs.B[g_ * per:(g_ + 1) * per].contiguous(), None,
                           inputs.bias[g_ * spec.N:(g_ + 1) * spec.N].contiguous())
        ref, _ = gemm_ref.run_spec_rows(sub, sub_in, rows=pick)
        _compare_rows(sub, sub_in, d[pick], ref, exact=False)
    op.close()


def test_grouped_argument_errors():
    spec = SPECS[1]
    inputs = wl.make_inputs(spec)
    dev = torch.device("cuda", 0)
    op = GemmOp(desc_from_spec(spec), groups=spec.groups)
    A, B = inputs.A.to(dev), inputs.B.to(dev)
    D = H.canary_buffer(spec)
    with pytest.raises(g.GemmError) as e:
        op(A, B, None, D)                                    # no offsets through gemm_run
    assert e.value.status == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_grouped_run(op.handle, A.data_ptr(), B.data_ptr(), None, D.data_ptr(), None, None, None)
    assert e.value.status == g.ERR_INVALID_ARG
    raw = torch.zeros(8, dtype=torch.int64, device=dev)
    with pytest.raises(g.GemmError) as e:
        g.gemm_grouped_run(op.handle, A.data_ptr(), B.data_ptr(), None, D.data_ptr(), None, raw.data_ptr() + 4, None)
    assert e.value.status == g.ERR_MISALIGNED
    with pytest.raises(g.GemmError) as e:
        op.set_schedule(g.SCHED_STREAM_K)
    assert e.value.status == g.ERR_UNSUPPORTED
    plain = GemmOp(desc_from_spec(dataclasses.replace(spec, groups=0)))
    with pytest.raises(g.GemmError) as e:
        plain.run_grouped(A, B, None, D, raw)                # a plain handle takes no offsets
    assert e.value.status == g.ERR_INVALID_ARG
    plain.close()
    op.close()


# ------------------------------------------------- block-scaled groups ----
U = 2.0 ** -24


def _bs_group_problem(spec, inputs, g_, r0, r1):
    """Group g_ of a grouped block-scaled workload as a problem of its own:
    its rows of A (and C), its factor blocks of A, B_g, SFB_g and bias_g."""
    nv = spec.block_scale == "nv"
    div = 2 if nv else 1                                    # e2m1: two elements per stored byte
    lda, per_b = spec.ld("a"), spec.matrix_elems("b")
    sv = 16 if nv else 32
    kb = ((spec.K + sv - 1) // sv + 3) // 4
    first = int(wl.grouped_sfa_rows(spec, inputs.extras["group_rows"])[r0]) // 128
    nblk = (r1 - r0 + 127) // 128
    sub = dataclasses.replace(spec, M=r1 - r0, groups=0, group_sizes=(), batch=1)
    per_sfb = ((spec.N + 127) // 128) * kb * 512
    C = None if inputs.C is None else inputs.C[r0 * spec.ld("c"): r1 * spec.ld("c")].contiguous()
    bias = None if inputs.bias is None else inputs.bias[g_ * spec.N:(g_ + 1) * spec.N].contiguous()
    extras = {"sfa": inputs.extras["sfa"][first * kb * 512:(first + nblk) * kb * 512].contiguous(),
              "sfb": inputs.extras["sfb"][g_ * per_sfb:(g_ + 1) * per_sfb].contiguous()}
    A = inputs.A[r0 * lda // div: r1 * lda // div].contiguous()
    B = inputs.B[g_ * per_b // div:(g_ + 1) * per_b // div].contiguous()
    return sub, wl.Inputs(sub, A, B, C, bias, inputs.scale_a, inputs.scale_b, extras=extras)


def _clear_sign(t):
    if t.dtype == torch.uint8:
        return t & 0x77
    return (t.view(torch.uint8) & 0x7F).view(torch.float8_e4m3fn)


def _run_bs(spec, inputs):
    dev = torch.device("cuda", 0)
    op = GemmOp(desc_from_spec(spec, inputs.scale_a, inputs.scale_b), groups=spec.groups)
    to = lambda t: None if t is None else t.to(dev)
    D = H.canary_buffer(spec)
    op.run_grouped(to(inputs.A), to(inputs.B), to(inputs.C), D, to(inputs.extras["group_rows"]), to(inputs.bias),
                   sfa=to(inputs.extras["sfa"]), sfb=to(inputs.extras["sfb"]))
    op.check()
    torch.cuda.synchronize()
    info = g.gemm_plan(desc_from_spec(dataclasses.replace(spec, groups=0, group_sizes=())))
    op.close()
    return H.bits_of_tensor(D.cpu()), info


def _check_bs(spec, inputs, bits, exact):
    assert H.untouched_outside(spec, bits), "write outside the logical D"
    d = H.logical_d(spec, bits).reshape(spec.M, spec.N)
    rows = inputs.extras["group_rows"].tolist()
    covered = np.zeros(spec.M, dtype=bool)
    for g_ in range(spec.groups):
        r0, r1 = rows[g_], rows[g_ + 1]
        if r1 <= r0:
            continue
        covered[r0:r1] = True
        sub, sub_in = _bs_group_problem(spec, inputs, g_, r0, r1)
        ref, t = gemm_ref.run_spec_rows(sub, sub_in, want_t=True)
        if exact:
            assert np.array_equal(d[r0:r1].astype(np.uint64), ref.astype(np.uint64)), f"group {g_} not bit-exact"
            continue
        abs_spec = dataclasses.replace(sub, alpha=1.0, beta=0.0, bias="none", act="none", dtype_d="f32", ldd=0)
        abs_in = wl.Inputs(abs_spec, _clear_sign(sub_in.A), _clear_sign(sub_in.B), None, None, sub_in.scale_a,
                           sub_in.scale_b, extras=sub_in.extras)
        _, tabs = gemm_ref.run_spec_rows(abs_spec, abs_in, want_t=True)
        got = H.from_bits(d[r0:r1], spec.dtype_d).reshape(r1 - r0, spec.N)
        want = H.from_bits(ref, spec.dtype_d).reshape(r1 - r0, spec.N)
        tol = H.SLOPE[spec.act] * (2 * spec.K * U * abs(spec.alpha) * tabs + 4 * U * np.abs(t)) + \
            H.ulp(want, spec.dtype_d)
        err = np.abs(got - want)
        assert np.all(err <= tol), f"group {g_}: {int((err > tol).sum())} elements out of tolerance"
    assert np.all(d[~covered].astype(np.uint64) == H.CANARY[spec.dtype_d]), "a row outside every group was written"


@pytest.mark.parametrize("fmt", ["mx", "nv"])
@pytest.mark.parametrize("shape", ["pair", "single"])
def test_grouped_block_scaled_bit_exact(fmt, shape):
    dt = "e4m3" if fmt == "mx" else "e2m1"
    if shape == "pair":
        spec = wl.Spec(f"grp_bs_{fmt}_pair", 5000, 1024, 512, groups=6, group_sizes=(700, 0, 1, 1299, 2000, 900),
                       dtype_in=dt, dtype_d="f32", dist="int4", block_scale=fmt, seed=160)
    else:
        spec = wl.Spec(f"grp_bs_{fmt}_single", 900, 384, 256, groups=3, group_sizes=(100, 250, 550), dtype_in=dt,
                       dtype_d="f32", dist="int4", block_scale=fmt, seed=161)
    inputs = wl.make_inputs(spec)
    bits, info = _run_bs(spec, inputs)
    assert info.cta_group == (2 if shape == "pair" else 1)
    _check_bs(spec, inputs, bits, exact=True)


@pytest.mark.parametrize("fmt", ["mx", "nv"])
def test_grouped_block_scaled_matches_oracle(fmt):
    dt = "e4m3" if fmt == "mx" else "e2m1"
    spec = wl.Spec(f"grp_bs_{fmt}_fused", 4100, 1100, 640, groups=5, group_sizes=(129, 1000, 0, 2500, 300),
                   dtype_in=dt, block_scale=fmt, alpha=0.5, beta=1.0, act="relu", bias="col", seed=162)
    inputs = wl.make_inputs(spec)
    bits, _ = _run_bs(spec, inputs)
    _check_bs(spec, inputs, bits, exact=False)

"""NVFP4 output (GEMM_OUT_SCALE_NV) on the GPU: D in e2m1, two elements per
byte, with one ue4m3 factor per 16 elements of a D row under the output's
global scale g, against the oracle's quantisation of its t.

Both sides round the exact quotients (amax / (6 g) for the factor,
t / (factor g) for an element) to the nearest even code, so they can differ
only because t does: the GPU accumulates in fp32, the oracle in fp64, apart
by at most the accumulation bound e.  A code may then differ by one step, and
only where the oracle's quotient lies within e (in the quotient's units) of
the midpoint between the two codes; such cases are counted and must stay
rare.  Elements are compared under the GPU's own factors.  Where t is
integer-valued both sides round the same quotients: factors and elements
compared bit for bit.  Bytes of D and of the factor tensor that name no real
element are never written."""
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
GUARD = 4096


def _sfd_bytes(spec):
    sfk = (spec.N + 15) // 16
    return spec.batch * ((spec.M + 127) // 128) * ((sfk + 3) // 4) * 512


def _oracle_t(spec, inputs):
    _, t = gemm_ref.run_spec_rows(dataclasses.replace(spec, dtype_d="f32"), inputs, want_t=True)
    return t


U = 2.0 ** -24


def _clear_sign(t):
    if t.dtype == torch.uint8:                  # two e2m1 codes per byte, sign in bit 3 of each
        return t & 0x77
    return (t.view(torch.uint8) & 0x7F).view(torch.float8_e4m3fn)


def _bound(spec, inputs, t):
    """Accumulation bound per element: the method's stated tolerance for
    per-tensor operands; for block-scaled ones the fp32 bound
    2 K u |alpha| sum|a b| + 4 u |t|, sum|a b| from the oracle on the
    sign-cleared operands (factors included)."""
    if spec.block_scale == "none":
        return np.full(t.shape, H.accumulation_bound(spec, inputs))
    abs_spec = dataclasses.replace(spec, alpha=1.0, beta=0.0, bias="none", act="none", dtype_d="f32", pad=0, ldd=0)
    abs_in = wl.Inputs(abs_spec, _clear_sign(inputs.A), _clear_sign(inputs.B), None, None, inputs.scale_a,
                       inputs.scale_b, extras=inputs.extras)
    _, tabs = gemm_ref.run_spec_rows(abs_spec, abs_in, want_t=True)
    return H.SLOPE[spec.act] * (2 * spec.K * U * abs(spec.alpha) * tabs + 4 * U * np.abs(t))


def _scale_for(t):
    """An output global scale that keeps every factor below 448: the format's
    amax / (448 * 6) rounded up to a power of two."""
    amax = float(np.max(np.abs(t)))
    return float(2.0 ** np.ceil(np.log2(max(amax, 1e-30) / (448.0 * 6.0))))


def _run(spec, inputs):
    op = GemmOp(desc_from_spec(spec, inputs.scale_a, inputs.scale_b))
    dev = torch.device("cuda", 0)
    to = lambda t: None if t is None else t.to(dev)
    ex = inputs.extras or {}
    nbytes = spec.batch * spec.matrix_elems("d") // 2
    D = torch.full((nbytes + GUARD,), 0xFF, dtype=torch.uint8, device=dev)
    sfd = torch.full((_sfd_bytes(spec) + 512,), 0xFF, dtype=torch.uint8, device=dev)
    op.run_args(to(inputs.A), to(inputs.B), None, D, to(inputs.bias), sfa=to(ex.get("sfa")), sfb=to(ex.get("sfb")),
                sfd=sfd)
    op.check()
    torch.cuda.synchronize()
    info = g.gemm_plan(op.desc)
    op.close()
    return D.cpu().numpy(), sfd.cpu().numpy(), info


def _unpack(spec, dbytes):
    """(L*M, N) element codes from D's bytes; asserts that no byte outside the
    logical D was written."""
    L, M, N, ldb = spec.batch, spec.M, spec.N, spec.ld("d") // 2
    per = spec.matrix_elems("d") // 2
    body = dbytes[: L * per].reshape(L, M, ldb)
    assert np.all(body[:, :, N // 2:] == 0xFF) and np.all(dbytes[L * per:] == 0xFF), "write outside the logical D"
    b = body[:, :, : N // 2].reshape(L * M, N // 2)
    q = np.empty((L * M, N), dtype=np.uint8)
    q[:, 0::2] = b & 0xF
    q[:, 1::2] = b >> 4
    return q


def _codes(spec, sfd):
    L, M, sfk = spec.batch, spec.M, (spec.N + 15) // 16
    idx = np.array([[[gemm_ref.sf_index(l, m, f, M, sfk) for f in range(sfk)] for m in range(M)] for l in range(L)])
    written = np.zeros(sfd.size, dtype=bool)
    written[idx.reshape(-1)] = True
    assert np.all(sfd[~written] == 0xFF), "factor bytes written outside the real (row, block) pairs"
    return sfd[idx].reshape(L * M, sfk)


def _e2m1(q):
    tab = np.array([gemm_ref.decode("e2m1", c) for c in range(16)])
    return tab[q]


def _e4m3(c):
    tab = np.array([gemm_ref.decode("e4m3", x) if x != 0x7F else np.nan for x in range(256)])
    return tab[c]


def _neighbours_near(got, ref, x, unit, e, grid):
    """Where got != ref (signed grid values): they must be neighbours on the
    signed grid, and the exact quotient x / unit must lie within e / unit of
    the rounding midpoint between them (t itself differs between the GPU's
    fp32 accumulation and the oracle's fp64 by at most e).  Returns the number
    of such differences."""
    signed = np.unique(np.concatenate([-grid, grid]))
    ig = np.searchsorted(signed, got)
    io = np.searchsorted(signed, ref)
    diff = (got != ref) & ~(np.isnan(got) & np.isnan(ref))
    assert np.all(signed[ig[diff]] == got[diff]) and np.all(signed[io[diff]] == ref[diff])
    assert np.all(np.abs(ig - io)[diff] == 1), "a code differs by more than one step"
    mid = (got + ref) / 2.0
    near = np.abs(x - mid * unit) <= e
    assert np.all(near[diff]), f"{int((diff & ~near).sum())} codes differ away from a rounding midpoint"
    return int(diff.sum())


def _check(spec, inputs, dbytes, sfd, t, exact=False):
    q = _unpack(spec, dbytes)
    codes = _codes(spec, sfd)
    gs = spec.scale_d
    ref_codes, ref_q = gemm_ref.nv_quantise_rows(t, gs)
    if exact:
        assert np.array_equal(codes, ref_codes), "factor codes differ"
        # compare values (e2m1 -0 and +0 are the same number)
        assert np.array_equal(_e2m1(q), _e2m1(ref_q)), "element codes differ"
        return
    e = _bound(spec, inputs, t)
    N = spec.N
    nb = codes.shape[1]
    # factors: the nearest-even e4m3 code of amax / (6 g); the oracle's amax
    # is within the block's largest e of the GPU's
    amax = np.zeros((t.shape[0], nb * 16))
    amax[:, :N] = np.abs(t)
    amax = amax.reshape(-1, nb, 16).max(axis=2)
    eb = np.zeros((t.shape[0], nb * 16))
    eb[:, :N] = e
    eb = eb.reshape(-1, nb, 16).max(axis=2)
    grid4 = np.array([gemm_ref.decode("e4m3", c) for c in range(0x7F)])
    nf = _neighbours_near(_e4m3(codes), _e4m3(ref_codes), amax, 6.0 * gs, eb, grid4)
    # elements: the oracle's rule under the GPU's own factors
    ref_q_g = gemm_ref.nv_quantise_elements(t, codes, gs)
    fac = np.repeat(_e4m3(codes), 16, axis=1)[:, :N] * gs
    grid2 = np.array([gemm_ref.decode("e2m1", c) for c in range(8)])
    ne = _neighbours_near(_e2m1(q), _e2m1(ref_q_g), t, fac, e, grid2)
    # each difference needs t within a few fp32 rounding steps of a midpoint: rare
    assert nf <= max(2, codes.size // 1000) and ne <= max(4, q.size // 1000), (nf, ne)
    # and every dequantised element is within half the widest e2m1 step of t
    dq = _e2m1(q) * fac
    tol = e + fac * 1.0 + 1e-30
    err = np.abs(dq - t)
    assert np.all(err <= tol), f"{int((err > tol).sum())} elements out of tolerance, worst {np.max(err - tol)}"


SPECS = [
    wl.Spec("nvo_single", 300, 520, 256, dtype_d="e2m1", alpha=0.5, act="relu", bias="col", seed=141, pad=32),
    wl.Spec("nvo_pair_gelu", 2048, 2048, 512, dtype_d="e2m1", act="gelu", bias="row", seed=142),
    wl.Spec("nvo_batched", 256, 384, 320, batch=3, dtype_d="e2m1", seed=143),
    wl.Spec("nvo_from_mx", 1024, 1024, 512, dtype_in="e4m3", block_scale="mx", dtype_d="e2m1", seed=144),
    wl.Spec("nvo_from_nv", 1024, 1024, 512, dtype_in="e2m1", block_scale="nv", dtype_d="e2m1", seed=145),
    # NVFP4 output with block-scaled inputs on CTA pairs: 256 x 128 tiles with
    # two accumulators (and the ragged last column tile of 2304 / 128 = 18)
    wl.Spec("nvo_from_nv_pair", 2304, 2304, 1024, dtype_in="e2m1", block_scale="nv", dtype_d="e2m1",
            act="relu", seed=146),
    wl.Spec("nvo_from_mx_pair", 2304, 2176, 512, dtype_in="e4m3", block_scale="mx", dtype_d="e2m1",
            bias="col", seed=148),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_nv_output_matches_oracle(spec):
    inputs = wl.make_inputs(spec)
    t = _oracle_t(spec, inputs)
    spec = dataclasses.replace(spec, scale_d=_scale_for(t))
    dbytes, sfd, info = _run(spec, inputs)
    _check(spec, inputs, dbytes, sfd, t)


@pytest.mark.parametrize("M,N", [(512, 400), (2304, 2304)])
def test_nv_output_bit_exact_on_integers(M, N):
    spec = wl.Spec("nvo_int", M, N, 256, dtype_in="f16", dtype_d="e2m1", dist="int4", bias="col", seed=147,
                   scale_d=0.25)
    inputs = wl.make_inputs(spec)
    inputs = dataclasses.replace(inputs, bias=torch.round(inputs.bias * 40))      # integer bias: t integral
    t = _oracle_t(spec, inputs)
    dbytes, sfd, info = _run(spec, inputs)
    assert info.cta_group == (1 if M == 512 else 2)
    _check(spec, inputs, dbytes, sfd, t, exact=True)


def test_nv_output_argument_errors():
    spec = dataclasses.replace(SPECS[0], scale_d=0.03125)
    op = GemmOp(desc_from_spec(spec))
    x = torch.zeros(1 << 22, device="cuda")
    with pytest.raises(g.GemmError) as e:
        op.run_args(x, x, None, x, x)                       # no sfd
    assert e.value.status == g.ERR_INVALID_ARG
    op.close()

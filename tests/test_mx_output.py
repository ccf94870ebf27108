"""MX output (GEMM_OUT_SCALE_MX) on the GPU: D in e4m3 with one ue8m0 factor
per 32 elements of a D row, against the oracle's quantisation of its t.

The factor is the shared exponent of max|t| of a block and the elements are
the nearest-even e4m3 codes of t / 2^(code-127) (an exact scaling); both
sides apply that rule to their own t, which differ by at most the
accumulation bound e (fp32 accumulation on the GPU, fp64 in the oracle).  So
factors are equal except at blocks whose maximum is within e of a power of
two (one step apart there), and elements, compared under the GPU's own
factors, are equal except one step apart where t lies within e of the
rounding midpoint between the two codes; such cases are counted and must
stay rare.  Factors and elements are bit-exact where t is integer-valued.
Bytes of D or of the factor tensor that name no real element are never
written."""
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


def _sfd_bytes(spec):
    sfk = (spec.N + 31) // 32
    return spec.batch * ((spec.M + 127) // 128) * ((sfk + 3) // 4) * 512


def _run(spec, inputs):
    op = GemmOp(desc_from_spec(spec))
    dev = torch.device("cuda", 0)
    to = lambda t: None if t is None else t.to(dev)
    ex = inputs.extras or {}
    D = H.canary_buffer(spec)
    sfd = torch.full((_sfd_bytes(spec) + 512,), 0xFF, dtype=torch.uint8, device=dev)
    op.run_args(to(inputs.A), to(inputs.B), None, D, to(inputs.bias), sfa=to(ex.get("sfa")), sfb=to(ex.get("sfb")),
                sfd=sfd)
    op.check()
    torch.cuda.synchronize()
    info = g.gemm_plan(op.desc)
    op.close()
    return H.bits_of_tensor(D.cpu()), sfd.cpu().numpy(), info


def _codes_from_tensor(spec, sfd):
    L, M, sfk = spec.batch, spec.M, (spec.N + 31) // 32
    idx = np.array([[[gemm_ref.sf_index(l, m, f, M, sfk) for f in range(sfk)] for m in range(M)] for l in range(L)])
    written = np.zeros(sfd.size, dtype=bool)
    written[idx.reshape(-1)] = True
    return sfd[idx], written


def _check(spec, inputs, bits, sfd, exact=False):
    assert H.untouched_outside(spec, bits), "write outside the logical D"
    L, M, N = spec.batch, spec.M, spec.N
    codes, written = _codes_from_tensor(spec, sfd)
    assert np.all(sfd[~written] == 0xFF), "factor bytes written outside the real (row, block) pairs"
    q = H.logical_d(spec, bits).reshape(L * M, N).astype(np.uint8)
    # t does not depend on D's type; the oracle's own D types are the IEEE ones
    _, t = gemm_ref.run_spec_rows(dataclasses.replace(spec, dtype_d="f32"), inputs, want_t=True)
    ref_codes, ref_q = gemm_ref.mx_quantise_rows(t)
    codes = codes.reshape(L * M, -1)
    if exact:
        assert np.array_equal(codes, ref_codes) and np.array_equal(q, ref_q)
        return
    e = H.accumulation_bound(spec, inputs)
    nb = codes.shape[1]
    blk = np.zeros((L * M, nb * 32))
    blk[:, :N] = np.abs(t)
    amax = blk.reshape(L * M, nb, 32).max(axis=2)
    near = np.abs(amax - np.exp2(np.round(np.log2(np.maximum(amax, 1e-300))))) <= e
    diff = codes.astype(int) - ref_codes.astype(int)
    assert np.all((diff == 0) | (near & (np.abs(diff) == 1))), "factor differs away from a power-of-two boundary"
    nf = int((diff != 0).sum())
    # elements: the oracle's rule under the GPU's own factors; a code may differ
    # by one step only where t / 2^(code-127) lies within e / 2^(code-127) of
    # the midpoint between the two e4m3 values
    ref_q_g = gemm_ref.mx_quantise_elements(t, codes)
    dec = np.array([gemm_ref.decode("e4m3", x) if (x & 0x7F) != 0x7F else np.nan for x in range(256)])
    vg, vo = dec[q], dec[ref_q_g]
    scale = np.exp2(np.repeat(codes.astype(np.int64), 32, axis=1)[:, :N] - 127.0)
    signed = np.unique(np.concatenate([-dec[:0x7F], dec[:0x7F]]))
    d = vg != vo
    ig, io = np.searchsorted(signed, vg), np.searchsorted(signed, vo)
    assert np.all(np.abs(ig - io)[d] == 1), "an element differs by more than one e4m3 step"
    mid = (vg + vo) / 2.0
    assert np.all((np.abs(t - mid * scale) <= e)[d]), "an element differs away from a rounding midpoint"
    ne = int(d.sum())
    assert nf <= max(2, codes.size // 1000) and ne <= max(4, q.size // 1000), (nf, ne)


SPECS = [
    wl.Spec("mxo_single", 300, 520, 256, dtype_d="e4m3", alpha=0.5, act="relu", bias="col", seed=111, pad=16),
    wl.Spec("mxo_pair_gelu", 2048, 2048, 512, dtype_d="e4m3", act="gelu", bias="row", seed=112),
    wl.Spec("mxo_batched", 256, 384, 320, batch=3, dtype_d="e4m3", seed=113),
    wl.Spec("mxo_from_mx", 1024, 1024, 512, dtype_in="e4m3", block_scale="mx", dtype_d="e4m3", seed=114),
    wl.Spec("mxo_from_mx_pair", 2304, 1152, 1024, dtype_in="e4m3", block_scale="mx", dtype_d="e4m3", act="relu",
            seed=115),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_mx_output_matches_oracle(spec):
    inputs = wl.make_inputs(spec)
    bits, sfd, _ = _run(spec, inputs)
    _check(spec, inputs, bits, sfd)


@pytest.mark.parametrize("M,N", [(512, 400), (2304, 2304)])
def test_mx_output_bit_exact_on_integers(M, N):
    spec = wl.Spec("mxo_int", M, N, 256, dtype_in="f16", dtype_d="e4m3", dist="int4", bias="col", seed=116)
    inputs = wl.make_inputs(spec)
    inputs = dataclasses.replace(inputs, bias=torch.round(inputs.bias * 40))      # integer bias: t integral
    bits, sfd, _ = _run(spec, inputs)
    _check(spec, inputs, bits, sfd, exact=True)


def test_mx_output_argument_errors():
    spec = SPECS[0]
    op = GemmOp(desc_from_spec(spec))
    x = torch.zeros(1 << 22, device="cuda")
    with pytest.raises(g.GemmError) as e:
        op.run_args(x, x, None, x, x)                       # no sfd
    assert e.value.status == g.ERR_INVALID_ARG
    op.close()

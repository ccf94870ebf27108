"""MX output (GEMM_OUT_SCALE_MX) on the GPU: D in e4m3 with one ue8m0 factor
per 32 elements of a D row, against the oracle's quantisation of its t.

The factor is a rounding decision on max|t| of a block; GPU (fp32
accumulation) and oracle (fp64, then rounded to fp32) can land on different
sides of a power of two only where the oracle's block maximum is within the
accumulation bound e of one.  So: factors equal except at such blocks (one
step apart there); every dequantised element q * 2^(code-127) within
e + 2^-3 |t| + 2^(code-127-9) of t (an e4m3 ulp is at most 2^-3 of the
value, plus the subnormal quantum); factors and elements bit-exact where t
is integer-valued.  Bytes of D or of the factor tensor that name no real
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
    blk[:, :N] = np.abs(t.astype(np.float32).astype(np.float64))
    amax = blk.reshape(L * M, nb, 32).max(axis=2)
    near = np.abs(amax - np.exp2(np.round(np.log2(np.maximum(amax, 1e-300))))) <= 2 * e
    diff = codes.astype(int) - ref_codes.astype(int)
    assert np.all((diff == 0) | (near & (np.abs(diff) == 1))), "factor differs away from a power-of-two boundary"
    dq = np.vectorize(lambda c: gemm_ref.decode("e4m3", int(c)))(q) * np.exp2(np.repeat(codes, 32, axis=1)[:, :N] - 127.0)
    scale = np.exp2(np.repeat(codes, 32, axis=1)[:, :N] - 127.0)
    tol = e + 2.0 ** -3 * np.abs(t) + scale * 2.0 ** -9
    assert np.all(np.abs(dq - t) <= tol), f"{int((np.abs(dq - t) > tol).sum())} elements out of tolerance"


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

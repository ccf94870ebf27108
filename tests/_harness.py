"""Shared test plumbing: run a workload through the CUDA path (C ABI) and
through the oracle, and compare them with the parity bar.

Parity bar (per element, from the method's stated tolerance):
    |D - D_ref| <= tau * sqrt(K) * max|A| * max|B| + ulp_D(|D_ref|)
with tau = 1e-3 for 16-bit operands and 2e-2 for e4m3 (max|A|, max|B| are
dequantised magnitudes), and bit-exact equality where every sum is an exact
integer (the fp16 integer workload).
"""
import math

import numpy as np
import torch

from dense_gemm_epilogue_sm_gb300 import workloads as wl
from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec
from oracle import gemm_ref

from _dtypes import BITS, bits_of_tensor, from_bits, torch_from_bits
from _storage import from_storage

TAU = {"f16": 1e-3, "bf16": 1e-3, "e4m3": 2e-2}
MBITS = {"f32": 23, "f16": 10, "bf16": 7}
EMIN = {"f32": -126, "f16": -14, "bf16": -126}
# a bit pattern no correct result takes (a NaN with a payload), used to see
# which elements the kernel wrote
CANARY = {"f32": 0x7FC0DEAD, "f16": 0x7E5A, "bf16": 0x7FA5, "e4m3": 0xFF}


def ulp(x, dtype):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(x > 0, x, 1.0)))
    e = np.maximum(np.where(x > 0, e, EMIN[dtype]), EMIN[dtype])
    return np.exp2(e - MBITS[dtype])


# An accumulation error e in the pre-activation value moves the output by at
# most slope * e: 1 for none/ReLU, max |d/dx x*Phi(x)| < 1.13 for GELU.
SLOPE = {"none": 1.0, "relu": 1.0, "gelu": 1.13}


def accumulation_bound(spec, inputs):
    """tau * sqrt(K) * max|A| * max|B|, times the activation's slope."""
    if spec.K == 0:
        return 0.0
    a = inputs.A.to(torch.float32).abs().max().item() * inputs.scale_a
    b = inputs.B.to(torch.float32).abs().max().item() * inputs.scale_b
    return SLOPE[spec.act] * TAU[spec.dtype_in] * math.sqrt(spec.K) * a * b


def tolerance(spec, inputs, d_ref):
    return accumulation_bound(spec, inputs) + ulp(d_ref, spec.dtype_d)


def canary_buffer(spec, extra=4096, device="cuda"):
    """D storage followed by a guard band, all set to the canary pattern."""
    n = spec.batch * spec.matrix_elems("d") + extra
    _, npi = BITS[spec.dtype_d]
    return torch_from_bits(np.full(n, CANARY[spec.dtype_d], dtype=npi), spec.dtype_d).to(device)


def run_gpu(spec, inputs, *, alias_c=False, op=None, repeat=1, stream=None):
    """Runs the workload on cuda:0 through the C ABI.  Returns (D storage
    incl. guard band as raw bits, the op).  With alias_c, D is C's own buffer
    (followed by a canary guard band)."""
    dev = torch.device("cuda", 0)
    A = inputs.A.to(dev)
    B = inputs.B.to(dev)
    C = inputs.C.to(dev) if inputs.C is not None else None
    bias = inputs.bias.to(dev) if inputs.bias is not None else None
    if op is None:
        op = GemmOp(desc_from_spec(spec, inputs.scale_a, inputs.scale_b))
    if alias_c:
        assert C is not None
        D = torch.cat([C, canary_buffer(spec)[spec.batch * spec.matrix_elems("d"):]])
        C = D[: C.numel()]
    else:
        D = canary_buffer(spec)
    for _ in range(repeat):
        op(A, B, C, D, bias, stream)
    op.check()
    torch.cuda.synchronize()
    return bits_of_tensor(D.cpu()), op


def logical_d(spec, bits):
    """(L, M, N) raw bits of D from its storage (guard band ignored)."""
    n = spec.batch * spec.matrix_elems("d")
    return from_storage(bits[:n], spec.batch, spec.M, spec.N, spec.order_d, spec.ld("d"),
                        spec.matrix_elems("d"))


def untouched_outside(spec, bits, before=None):
    """True when every element outside the logical D (padding, guard band)
    still holds what it held before the run: the canary pattern, or the
    matching elements of `before` (raw bits) where given."""
    n = spec.batch * spec.matrix_elems("d")
    canary = CANARY[spec.dtype_d]
    if before is not None:
        canary = np.asarray(before).astype(np.uint64)
    mask = np.ones(bits.shape[0], dtype=bool)
    idx = np.arange(n)
    L, per, ld = spec.batch, spec.matrix_elems("d"), spec.ld("d")
    local = idx % per
    inner = local % ld
    outer = local // ld
    rows, cols = (spec.M, spec.N) if spec.order_d == "row" else (spec.N, spec.M)
    inside = (inner < cols) & (outer < rows)
    mask[:n] = ~inside
    want = canary[mask] if isinstance(canary, np.ndarray) else canary
    return bool(np.all(bits[mask].astype(np.uint64) == want))


def oracle_rows(spec, inputs, rows=None):
    bits, _ = gemm_ref.run_spec_rows(spec, inputs, rows=rows)
    return bits


def compare(spec, inputs, d_bits_logical, ref_bits, rows=None, exact=False):
    """d_bits_logical: (L, M, N) bits from the GPU; ref_bits: oracle rows
    (all rows when rows is None).  Returns the worst normalised error."""
    got = d_bits_logical.reshape(spec.batch * spec.M, spec.N)
    if rows is not None:
        got = got[np.asarray(rows)]
    if exact:
        assert np.array_equal(got.astype(np.uint64), ref_bits.astype(np.uint64)), "not bit-exact"
        return 0.0
    g = from_bits(got, spec.dtype_d).reshape(got.shape)
    r = from_bits(ref_bits, spec.dtype_d).reshape(ref_bits.shape)
    assert np.isfinite(g).all(), "non-finite output (unwritten element?)"
    tol = tolerance(spec, inputs, r)
    err = np.abs(g - r)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} elements out of tolerance; first at {tuple(i)}: "
                             f"got {g[tuple(i)]}, want {r[tuple(i)]}, tol {np.broadcast_to(tol, r.shape)[tuple(i)]}")
    return float(np.max(err / np.maximum(tol, 1e-30))) if err.size else 0.0


def sample_rows(spec, per_tile=4, seed=0):
    """Rows l*M + m spanning every 128-row tile of every batch, incl. the last row."""
    rng = np.random.default_rng(seed)
    rows = set()
    for l in range(spec.batch):
        for t0 in range(0, spec.M, 128):
            hi = min(spec.M, t0 + 128)
            rows.update(int(x) + l * spec.M for x in rng.integers(t0, hi, per_tile))
        rows.add(l * spec.M + spec.M - 1)
        rows.add(l * spec.M)
    return np.array(sorted(rows), dtype=np.int64)

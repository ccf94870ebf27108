"""Python face of the C GEMM oracle.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this module.  It marshals numpy/torch CPU buffers into the oracle's
own ``oracle_problem_t`` and calls ``oracle_gemm_rows``; all arithmetic lives in
``gemm_oracle.c``.  See that file's header for what is computed and where the
pages define it.
"""
import ctypes
import os

import numpy as np

from . import build as _build

# The oracle's own element-type codes.
F32, F16, BF16, E4M3, UE8M0, E2M1, UE4M3 = 0, 1, 2, 3, 4, 5, 6
_NAMES = {"f32": F32, "f16": F16, "bf16": BF16, "e4m3": E4M3, "ue8m0": UE8M0, "e2m1": E2M1, "ue4m3": UE4M3}
# scale-factor vector size of each block-scaled format: mx_float8 (ue8m0
# per 32), nv_float4 (ue4m3 per 16)
SF_VEC = {"mx": 32, "nv": 16}
_BYTES = {F32: 4, F16: 2, BF16: 2, E4M3: 1}
_BITS_NP = {F32: np.uint32, F16: np.uint16, BF16: np.uint16, E4M3: np.uint8}


class Problem(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("L", ctypes.c_int64),
        ("op_a", ctypes.c_int32), ("op_b", ctypes.c_int32),
        ("order_a", ctypes.c_int32), ("order_b", ctypes.c_int32),
        ("order_c", ctypes.c_int32), ("order_d", ctypes.c_int32),
        ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64), ("ldd", ctypes.c_int64),
        ("stride_a", ctypes.c_int64), ("stride_b", ctypes.c_int64), ("stride_c", ctypes.c_int64),
        ("stride_d", ctypes.c_int64), ("stride_bias", ctypes.c_int64),
        ("dtype_a", ctypes.c_int32), ("dtype_b", ctypes.c_int32),
        ("dtype_c", ctypes.c_int32), ("dtype_d", ctypes.c_int32),
        ("alpha", ctypes.c_double), ("beta", ctypes.c_double),
        ("scale_a", ctypes.c_double), ("scale_b", ctypes.c_double),
        ("has_bias", ctypes.c_int32), ("bias_per_row", ctypes.c_int32), ("act", ctypes.c_int32),
        ("sf_vec", ctypes.c_int32),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        l = ctypes.CDLL(path)
        l.oracle_gemm_rows.restype = ctypes.c_int
        l.oracle_gemm_rows.argtypes = [ctypes.POINTER(Problem), ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        l.oracle_gemm_rows_sf.restype = ctypes.c_int
        l.oracle_gemm_rows_sf.argtypes = [ctypes.POINTER(Problem), ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int]
        l.oracle_sf_index.restype = ctypes.c_int64
        l.oracle_sf_index.argtypes = [ctypes.c_int64] * 5
        l.oracle_encode_e4m3.restype = ctypes.c_uint32
        l.oracle_encode_e4m3.argtypes = [ctypes.c_double]
        l.oracle_encode_e4m3_array.restype = None
        l.oracle_encode_e4m3_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        l.oracle_encode_e2m1_array.restype = None
        l.oracle_encode_e2m1_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        l.oracle_decode.restype = ctypes.c_double
        l.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
        l.oracle_encode.restype = ctypes.c_uint32
        l.oracle_encode.argtypes = [ctypes.c_int, ctypes.c_double]
        l.oracle_max_threads.restype = ctypes.c_int
        l.oracle_scatter_d.restype = ctypes.c_int
        l.oracle_scatter_d.argtypes = [ctypes.POINTER(Problem), ctypes.c_void_p, ctypes.c_void_p]
        _lib = l
    return _lib


def dtype_code(name: str) -> int:
    return _NAMES[name]


def decode(dtype: str, bits: int) -> float:
    return lib().oracle_decode(_NAMES[dtype], bits)


def encode(dtype: str, value: float) -> int:
    return lib().oracle_encode(_NAMES[dtype], value)


def max_threads() -> int:
    return lib().oracle_max_threads()


def _addr(buf):
    """Address of a CPU buffer: a numpy array or a contiguous CPU torch tensor."""
    if buf is None:
        return None
    if isinstance(buf, np.ndarray):
        assert buf.flags["C_CONTIGUOUS"]
        return buf.ctypes.data
    assert buf.device.type == "cpu" and buf.is_contiguous()
    return buf.data_ptr()


def make_problem(M, N, K, L=1, op_a="N", op_b="N", order_a="row", order_b="col",
                 order_c="row", order_d="row", lda=None, ldb=None, ldc=None, ldd=None,
                 stride_a=0, stride_b=0, stride_c=0, stride_d=0, stride_bias=0,
                 dtype_a="bf16", dtype_b="bf16", dtype_c="bf16", dtype_d="bf16",
                 alpha=1.0, beta=0.0, scale_a=1.0, scale_b=1.0, has_bias=False,
                 bias_per_row=False, act="none", sf_vec=0):
    """Builds an oracle problem; leading dimensions default to the tight ones."""

    def tight(order, rows, cols):
        return cols if order == "row" else rows

    a_rows, a_cols = (M, K) if op_a == "N" else (K, M)
    b_rows, b_cols = (K, N) if op_b == "N" else (N, K)
    p = Problem()
    p.M, p.N, p.K, p.L = M, N, K, L
    p.op_a, p.op_b = int(op_a == "T"), int(op_b == "T")
    p.order_a, p.order_b = int(order_a == "row"), int(order_b == "row")
    p.order_c, p.order_d = int(order_c == "row"), int(order_d == "row")
    p.lda = lda if lda is not None else max(1, tight(order_a, a_rows, a_cols))
    p.ldb = ldb if ldb is not None else max(1, tight(order_b, b_rows, b_cols))
    p.ldc = ldc if ldc is not None else max(1, tight(order_c, M, N))
    p.ldd = ldd if ldd is not None else max(1, tight(order_d, M, N))
    p.stride_a, p.stride_b, p.stride_c, p.stride_d, p.stride_bias = (
        stride_a, stride_b, stride_c, stride_d, stride_bias)
    p.dtype_a, p.dtype_b = _NAMES[dtype_a], _NAMES[dtype_b]
    p.dtype_c, p.dtype_d = _NAMES[dtype_c], _NAMES[dtype_d]
    p.alpha, p.beta, p.scale_a, p.scale_b = alpha, beta, scale_a, scale_b
    p.has_bias, p.bias_per_row = int(bool(has_bias)), int(bool(bias_per_row))
    p.act = {"none": 0, "relu": 1, "gelu": 2}[act]
    p.sf_vec = sf_vec
    return p


def gemm_rows(p: Problem, A, B, C=None, bias=None, rows=None, nthreads=0, want_t=False, sfa=None, sfb=None):
    """Runs the oracle on the listed rows (l*M + m; default: all rows).

    Returns (bits, t): ``bits`` is a (len(rows), N) array of D's raw bit
    patterns (uint16 for 16-bit types, uint32 for fp32); ``t`` the fp64
    values before rounding when ``want_t`` is set, else None.  ``sfa`` /
    ``sfb``: the scale-factor bytes (ue8m0 for p.sf_vec = 32, ue4m3 for 16;
    basic-block layout, see sf_index) when the problem is block-scaled.
    """
    if rows is None:
        rows = np.arange(p.L * p.M, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((len(rows), p.N), dtype=_BITS_NP[p.dtype_d])
    t = np.zeros((len(rows), p.N), dtype=np.float64) if want_t else None
    rc = lib().oracle_gemm_rows_sf(ctypes.byref(p), _addr(A), _addr(B), _addr(sfa), _addr(sfb), _addr(C),
                                   _addr(bias), len(rows), rows.ctypes.data, out.ctypes.data,
                                   None if t is None else t.ctypes.data, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_rows failed with code {rc}")
    return out, t


def bits_to_float64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of raw bit patterns, via the oracle's own decoder."""
    code = _NAMES[dtype]
    flat = bits.reshape(-1)
    if dtype == "f32":
        return flat.view(np.float32).astype(np.float64).reshape(bits.shape)
    if dtype == "f16":
        return flat.view(np.float16).astype(np.float64).reshape(bits.shape)
    if dtype == "bf16":
        widened = (flat.astype(np.uint32) << 16).view(np.float32)
        return widened.astype(np.float64).reshape(bits.shape)
    dec = lib().oracle_decode
    return np.array([dec(code, int(x)) for x in flat], dtype=np.float64).reshape(bits.shape)


def problem_from_spec(spec, inputs):
    """Oracle problem for a workload spec and its generated inputs (duck-typed:
    any object with the workload's attribute names)."""
    L = spec.batch
    stride = lambda w: spec.matrix_elems(w) if L > 1 else 0
    bias_len = 0 if spec.bias == "none" else (spec.N if spec.bias == "col" else spec.M)
    return make_problem(
        spec.M, spec.N, spec.K, L, spec.op_a, spec.op_b, spec.order_a, spec.order_b, spec.order_c, spec.order_d,
        spec.ld("a"), spec.ld("b"), spec.ld("c"), spec.ld("d"),
        stride("a"), stride("b"), stride("c"), stride("d"), bias_len if L > 1 else 0,
        spec.dtype_in, spec.dtype_in, spec.dtype_d, spec.dtype_d,
        spec.alpha, spec.beta, inputs.scale_a, inputs.scale_b,
        spec.bias != "none", spec.bias == "row", spec.act)


def run_spec_rows(spec, inputs, rows=None, nthreads=0, want_t=False):
    """Oracle rows (l*M + m) of a workload; returns (bits, t) as gemm_rows."""
    p = problem_from_spec(spec, inputs)
    ex = getattr(inputs, "extras", None) or {}
    if getattr(spec, "block_scale", "none") != "none":
        p.sf_vec = SF_VEC[spec.block_scale]
    return gemm_rows(p, inputs.A, inputs.B, inputs.C, inputs.bias, rows=rows, nthreads=nthreads, want_t=want_t,
                     sfa=ex.get("sfa"), sfb=ex.get("sfb"))


def sf_index(l, row, kf, rows, sfk):
    """Byte offset of scale factor (row, kf) of batch l in the basic-block
    layout ("Scale Factor Layouts"): the oracle's own index function."""
    return lib().oracle_sf_index(l, row, kf, rows, sfk)


# ------------------------------------------------------------ reductions --
# Per-row and per-column reductions of the epilogue's output ("Technical
# Documentation: NVIDIA/cutlass", "What's New in CUTLASS 4.8": custom
# epilogue fusions support per-row or per-column reductions).  Reading: the
# reduced value is t, the epilogue result before it is rounded to D's type,
# reduced over the whole (l, m, :) row or (l, :, n) column; the abs-max is
# max |t| over each batch.  ``t`` is the (L, M, N) fp64 array of gemm_rows /
# run_spec_rows with want_t, every row present.

def row_sums(t):
    """(L, M): sum over n of t(l, m, n)."""
    return np.sum(t, axis=2)


def col_sums(t):
    """(L, N): sum over m of t(l, m, n)."""
    return np.sum(t, axis=1)


def abs_max(t):
    """(L,): max over m, n of |t(l, m, n)| (NaN if any t is NaN)."""
    return np.max(np.abs(t), axis=(1, 2))


# ------------------------------------------------- block-scaled output ----
# MX output of the epilogue ("Technical Documentation: NVIDIA/cutlass",
# "Blackwell SM100 GEMMs": an epilogue fusion that writes elements plus a
# block scale factor per SFDVectorSize elements along an output dimension).
# Reading for mx_float8 output: blocks of 32 consecutive elements of a D row
# (D row-major), factor ue8m0 from the OCP MX rule (shared exponent
# floor(log2 amax) - 8, where 8 is the exponent of e4m3's largest power of
# two, code clamped to [0, 254]; a block with a NaN or infinite element gets
# code 255 and NaN elements), elements = e4m3(t / 2^(code-127)) rounded to
# nearest even and saturated at +-448.  Everything is taken on the exact
# (fp64) t: the exponent by frexp, the division by a power of two exactly,
# and one rounding into e4m3.

def encode_e4m3(values):
    """fp64 array -> e4m3 codes (uint8), round to nearest even, saturating."""
    v = np.ascontiguousarray(values, dtype=np.float64).reshape(-1)
    out = np.empty(v.size, dtype=np.uint8)
    lib().oracle_encode_e4m3_array(v.ctypes.data, v.size, out.ctypes.data)
    return out.reshape(np.shape(values))


def mx_quantise_rows(t):
    """t: (R, N) epilogue values -> (codes (R, ceil(N/32)) uint8, elements
    (R, N) e4m3 codes uint8)."""
    t = np.asarray(t, dtype=np.float64)
    R, N = t.shape
    nb = (N + 31) // 32
    blk = np.zeros((R, nb * 32))
    blk[:, :N] = t
    blk = blk.reshape(R, nb, 32)
    with np.errstate(invalid="ignore"):
        a = np.abs(blk)
        bad = ~np.isfinite(a).all(axis=2)
        amax = np.where(bad, 0.0, a.max(axis=2))
    _, e = np.frexp(amax)                        # amax = f * 2^e, f in [0.5, 1): floor(log2 amax) = e - 1
    code = np.where(amax > 0, np.clip(e - 1 - 8 + 127, 0, 254), 0).astype(np.int64)
    code = np.where(bad, 255, code).astype(np.uint8)
    return code, mx_quantise_elements(t, code)


def mx_quantise_elements(t, codes):
    """The MX element rule alone, under given ue8m0 codes (R, ceil(N/32)):
    e4m3(t / 2^(code-127)), nearest even, saturated; NaN (0x7F) where the
    code is 255.  (R, N) e4m3 codes."""
    t = np.asarray(t, dtype=np.float64)
    R, N = t.shape
    c = np.repeat(codes.astype(np.int64), 32, axis=1)[:, :N]
    scaled = t / np.ldexp(1.0, np.minimum(c, 254) - 127)      # exact: a power of two
    q = encode_e4m3(scaled)
    return np.where(c == 255, np.uint8(0x7F), q).astype(np.uint8)


# NVFP4 output ("Blackwell SM100 GEMMs": LinCombBlockScaleFactor with
# SFDVectorSize = 16).  Reading (the page leaves the rule open): blocks of 16
# consecutive elements of a D row; with the output's fp32 global scale g,
# factor = e4m3(amax / (6 g)) (ue4m3, nearest even, saturating at 448) and
# elements = e2m1(t / (factor * g)) (nearest even, saturating at 6), zero
# where the factor is 0; a block holding NaN or inf gets factor 0x7F and zero
# elements.  Both roundings are of the exact quotient of the exact t.

def encode_e2m1(values):
    """fp64 array -> e2m1 codes (uint8, 0..15), round to nearest even, saturating."""
    v = np.ascontiguousarray(values, dtype=np.float64).reshape(-1)
    out = np.empty(v.size, dtype=np.uint8)
    lib().oracle_encode_e2m1_array(v.ctypes.data, v.size, out.ctypes.data)
    return out.reshape(np.shape(values))


def _grid(dtype, ncodes):
    """Magnitudes of the non-negative codes 0 .. ncodes-1 (ascending)."""
    return np.array([decode(dtype, c) for c in range(ncodes)], dtype=np.float64)


def rne_quotient(num, den, grid):
    """Round-to-nearest-even of num / den onto a grid of magnitudes, with
    saturation: returns the index i of grid[i] nearest to the exact quotient
    (num >= 0, den > 0, arrays of one shape), the even index of the two on a
    tie, the last index beyond the last midpoint.  Index parity is the code's
    last mantissa bit for the grids used here (positive e4m3 and e2m1 codes).

    Decided without dividing: num / den lies above midpoint mid_j exactly when
    num > mid_j * den.  Every product here is exact in fp64: a midpoint has at
    most 5 significant bits and den (6 g, or factor * g, g an fp32 value) at
    most 28, so the comparisons see the exact quotient."""
    num = np.asarray(num, dtype=np.float64)
    den = np.asarray(den, dtype=np.float64)
    mids = (grid[:-1] + grid[1:]) / 2.0
    prod = den[..., None] * mids
    n = num[..., None]
    idx = np.sum(n > prod, axis=-1)              # midpoints strictly below the quotient
    tie = n == prod                              # quotient exactly on midpoint j: idx == j
    on_tie = tie.any(axis=-1)
    odd = (idx % 2) == 1                         # between j (odd) and j + 1 (even): go up
    return np.where(on_tie & odd, idx + 1, idx)


def nv_quantise_rows(t, scale_d):
    """t: (R, N) epilogue values, scale_d: the output's global scale ->
    (factor codes (R, ceil(N/16)) uint8, element codes (R, N) uint8)."""
    t = np.asarray(t, dtype=np.float64)
    R, N = t.shape
    nb = (N + 15) // 16
    blk = np.zeros((R, nb * 16))
    blk[:, :N] = t
    blk = blk.reshape(R, nb, 16)
    with np.errstate(invalid="ignore"):
        a = np.abs(blk)
        bad = ~np.isfinite(a).all(axis=2)
        amax = np.where(bad, 0.0, a.max(axis=2))
    g = float(np.float32(scale_d))               # the fp32 global scale
    e4m3 = _grid("e4m3", 0x7F)                   # 0 .. 448 (code 0x7E)
    code = rne_quotient(amax, np.full(amax.shape, 6.0 * g), e4m3)
    code = np.where(bad, 0x7F, code).astype(np.uint8)
    return code, nv_quantise_elements(t, code, scale_d)


def nv_quantise_elements(t, codes, scale_d):
    """The element rule alone, under given factor codes (R, ceil(N/16)):
    e2m1(t / (factor * g)) rounded to nearest even and saturated, zero where
    the factor is 0 or NaN (0x7F).  (R, N) codes, sign in bit 3."""
    t = np.asarray(t, dtype=np.float64)
    R, N = t.shape
    g = float(np.float32(scale_d))
    fac = np.where(codes == 0x7F, 0.0, _grid("e4m3", 0x80)[np.minimum(codes, 0x7F)])
    den = np.repeat(fac * g, 16, axis=1)[:, :N]
    live = den > 0
    with np.errstate(invalid="ignore"):
        mag = rne_quotient(np.where(live, np.abs(t), 0.0), np.where(live, den, 1.0), _grid("e2m1", 8))
    neg = np.signbit(t) & live
    return np.where(live, mag | np.where(neg, 8, 0), 0).astype(np.uint8)

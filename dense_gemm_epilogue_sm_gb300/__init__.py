"""GB300 (sm_103a) fused-epilogue dense GEMM: thin Python binding.

Mirrors the C ABI of ``include/gemm.h`` and ``include/gemm_layout.h`` name for
name.  This module only marshals arguments (ctypes structures, raw pointers,
a CUDA stream handle); every step of the computation runs in the CUDA
library ``libgemm_sm103.so`` built from ``csrc/``.  There is no fallback: if
the library is missing, importing this package raises.

    D = act(alpha * scale_a * scale_b * op(A) @ op(B) + beta * C + bias)

Typical use with torch tensors::

    import dense_gemm_epilogue_sm_gb300 as g
    d = g.make_desc(M, N, K, dtype_a=g.BF16, dtype_b=g.BF16, dtype_d=g.BF16,
                    order_a=g.ROW_MAJOR, order_b=g.COL_MAJOR, order_d=g.ROW_MAJOR,
                    alpha=0.5, beta=1.0, bias=g.BIAS_COL, act=g.ACT_RELU)
    h = g.gemm_create(d)
    g.gemm_run(h, A.data_ptr(), B.data_ptr(), C.data_ptr(), D.data_ptr(),
               bias.data_ptr(), torch.cuda.current_stream().cuda_stream)
    g.gemm_check(h)
    g.gemm_destroy(h)
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# The diagnostic builds (GEMM_DEBUG index checks, GEMM_STAMPS timestamps; see
# _build.py) are separate libraries, chosen by naming one in
# GEMM_SM103_LIBRARY; the default is the normal build next to this file.
LIBRARY_PATH = os.environ.get("GEMM_SM103_LIBRARY") or os.path.join(_HERE, "libgemm_sm103.so")

# gemm_status_t
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_CUDA, ERR_TIMEOUT, ERR_NO_DEVICE, ERR_BOUNDS = range(8)
# gemm_dtype_t
F32, F16, BF16, E4M3, E2M1 = 0, 1, 2, 3, 4
# gemm_order_t
COL_MAJOR, ROW_MAJOR = 0, 1
# gemm_op_t
OP_N, OP_T = 0, 1
# gemm_act_t
ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2
# gemm_reduce_t (flags)
REDUCE_NONE, REDUCE_ROW_SUM, REDUCE_COL_SUM, REDUCE_ABS_MAX = 0, 1, 2, 4
# gemm_block_scale_t
BLOCK_SCALE_NONE, BLOCK_SCALE_MX, BLOCK_SCALE_NV = 0, 1, 2
# gemm_out_scale_t
OUT_SCALE_NONE, OUT_SCALE_MX, OUT_SCALE_NV = 0, 1, 2
# gemm_bias_t
BIAS_NONE, BIAS_COL, BIAS_ROW = 0, 1, 2
# gemm_sched_t
SCHED_AUTO, SCHED_DATA_PARALLEL, SCHED_STREAM_K, SCHED_SPLIT_TAIL, SCHED_DYNAMIC = 0, 1, 2, 3, 4

DTYPE_BYTES = {F32: 4, F16: 2, BF16: 2, E4M3: 1}


class GemmDesc(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("batch", ctypes.c_int64),
        ("op_a", ctypes.c_int32), ("op_b", ctypes.c_int32),
        ("order_a", ctypes.c_int32), ("order_b", ctypes.c_int32),
        ("order_c", ctypes.c_int32), ("order_d", ctypes.c_int32),
        ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64), ("ldd", ctypes.c_int64),
        ("stride_a", ctypes.c_int64), ("stride_b", ctypes.c_int64), ("stride_c", ctypes.c_int64),
        ("stride_d", ctypes.c_int64), ("stride_bias", ctypes.c_int64),
        ("dtype_a", ctypes.c_int32), ("dtype_b", ctypes.c_int32),
        ("dtype_c", ctypes.c_int32), ("dtype_d", ctypes.c_int32),
        ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
        ("scale_a", ctypes.c_float), ("scale_b", ctypes.c_float),
        ("act", ctypes.c_int32), ("bias", ctypes.c_int32), ("reduce", ctypes.c_int32),
        ("block_scale", ctypes.c_int32), ("out_scale", ctypes.c_int32), ("scale_d", ctypes.c_float),
    ]


class GemmArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("A", "B", "C", "D", "bias", "sfa", "sfb", "row_sum", "col_sum",
                                                "abs_max", "sfd")]


class GemmPlanInfo(ctypes.Structure):
    _fields_ = [
        ("swapped", ctypes.c_int32), ("a_k_major", ctypes.c_int32), ("b_k_major", ctypes.c_int32),
        ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
        ("cta_group", ctypes.c_int32), ("stages", ctypes.c_int32), ("raster_group", ctypes.c_int32),
        ("epi_cols", ctypes.c_int32),
        ("tiles_m", ctypes.c_int64), ("tiles_n", ctypes.c_int64), ("tiles", ctypes.c_int64),
        ("kernel_m", ctypes.c_int64), ("kernel_n", ctypes.c_int64),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemmError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__(f"{where}: {gemm_status_str(status)} (status {status})" if where else gemm_status_str(status))


def _load():
    if not os.path.exists(LIBRARY_PATH):
        raise ImportError(
            f"{LIBRARY_PATH} is missing; build it first (python -c 'import __graft_entry__ as g; g.build()' "
            "or python dense_gemm_epilogue_sm_gb300/_build.py)")
    lib = ctypes.CDLL(LIBRARY_PATH)
    vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    sigs = {
        "gemm_plan": (i32, [ctypes.POINTER(GemmDesc), ctypes.POINTER(GemmPlanInfo)]),
        "gemm_create": (i32, [ctypes.POINTER(vp), ctypes.POINTER(GemmDesc)]),
        "gemm_run": (i32, [vp, vp, vp, vp, vp, vp, vp]),
        "gemm_run_ex": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "gemm_run_args": (i32, [vp, ctypes.POINTER(GemmArgs), vp]),
        "gemm_grouped_create": (i32, [ctypes.POINTER(vp), ctypes.POINTER(GemmDesc), i32]),
        "gemm_grouped_run": (i32, [vp, vp, vp, vp, vp, vp, vp, vp]),
        "gemm_grouped_run_args": (i32, [vp, ctypes.POINTER(GemmArgs), vp, vp]),
        "gemm_check": (i32, [vp]),
        "gemm_destroy": (i32, [vp]),
        "gemm_set_debug": (i32, [vp, i32, u32]),
        "gemm_set_stamps": (i32, [vp, vp]),
        "gemm_build_flags": (i32, []),
        "gemm_launch_count": (ctypes.c_uint64, [vp]),
        "gemm_set_schedule": (i32, [vp, i32]),
        "gemm_get_schedule": (i32, [vp, ctypes.POINTER(i32), ctypes.POINTER(i64), ctypes.POINTER(i64),
                                    ctypes.POINTER(i32)]),
        "gemm_status_str": (ctypes.c_char_p, [i32]),
        "gemm_run_noalloc": (i32, [ctypes.POINTER(GemmDesc), vp, vp, vp, vp, vp, vp, i32]),
        "gemm_layout_query": (ctypes.c_int, [ctypes.c_char_p, ctypes.c_char_p, ctypes.POINTER(i64)]),
        "gemm_layout_eval": (ctypes.c_int, [ctypes.c_char_p, ctypes.POINTER(i64), i32, ctypes.POINTER(i64)]),
        "gemm_layout_op": (ctypes.c_int, [ctypes.c_char_p, ctypes.c_char_p, ctypes.c_char_p, i64,
                                          ctypes.c_char_p, ctypes.c_size_t]),
        "gemm_layout_gather_f32": (ctypes.c_int, [ctypes.c_char_p, vp, vp, i64, vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()
EXPORTED = ("gemm_plan", "gemm_create", "gemm_run", "gemm_run_ex", "gemm_run_args", "gemm_grouped_create",
            "gemm_grouped_run", "gemm_grouped_run_args", "gemm_check", "gemm_destroy", "gemm_set_debug",
            "gemm_set_stamps", "gemm_build_flags", "gemm_set_schedule", "gemm_get_schedule", "gemm_launch_count", "gemm_status_str", "gemm_run_noalloc",
            "gemm_layout_query", "gemm_layout_eval", "gemm_layout_op", "gemm_layout_gather_f32")


def make_desc(M, N, K, batch=1, op_a=OP_N, op_b=OP_N, order_a=ROW_MAJOR, order_b=COL_MAJOR,
              order_c=ROW_MAJOR, order_d=ROW_MAJOR, lda=None, ldb=None, ldc=None, ldd=None,
              stride_a=0, stride_b=0, stride_c=0, stride_d=0, stride_bias=0,
              dtype_a=BF16, dtype_b=BF16, dtype_c=None, dtype_d=BF16, alpha=1.0, beta=0.0,
              scale_a=1.0, scale_b=1.0, act=ACT_NONE, bias=BIAS_NONE, reduce=REDUCE_NONE,
              block_scale=BLOCK_SCALE_NONE, out_scale=OUT_SCALE_NONE, scale_d=1.0):
    """Fills a GemmDesc; leading dimensions default to the tight ones and the
    batch strides of A, B, C, D to the tight matrix sizes when batch > 1."""

    def tight(order, rows, cols):
        return max(1, cols if order == ROW_MAJOR else rows)

    a_rows, a_cols = (M, K) if op_a == OP_N else (K, M)
    b_rows, b_cols = (K, N) if op_b == OP_N else (N, K)
    d = GemmDesc()
    d.M, d.N, d.K, d.batch = M, N, K, batch
    d.op_a, d.op_b = op_a, op_b
    d.order_a, d.order_b, d.order_c, d.order_d = order_a, order_b, order_c, order_d
    d.lda = lda if lda is not None else tight(order_a, a_rows, a_cols)
    d.ldb = ldb if ldb is not None else tight(order_b, b_rows, b_cols)
    d.ldc = ldc if ldc is not None else tight(order_c, M, N)
    d.ldd = ldd if ldd is not None else tight(order_d, M, N)
    if batch > 1:
        stride_a = stride_a or d.lda * (a_rows if order_a == ROW_MAJOR else a_cols)
        stride_b = stride_b or d.ldb * (b_rows if order_b == ROW_MAJOR else b_cols)
        stride_c = stride_c or d.ldc * (M if order_c == ROW_MAJOR else N)
        stride_d = stride_d or d.ldd * (M if order_d == ROW_MAJOR else N)
    d.stride_a, d.stride_b, d.stride_c, d.stride_d, d.stride_bias = (
        stride_a, stride_b, stride_c, stride_d, stride_bias)
    d.dtype_a, d.dtype_b = dtype_a, dtype_b
    d.dtype_d = dtype_d
    d.dtype_c = dtype_d if dtype_c is None else dtype_c
    d.alpha, d.beta, d.scale_a, d.scale_b = alpha, beta, scale_a, scale_b
    d.act, d.bias, d.reduce, d.block_scale, d.out_scale = act, bias, reduce, block_scale, out_scale
    d.scale_d = scale_d
    return d


def gemm_status_str(status):
    return lib.gemm_status_str(status).decode()


def gemm_plan(desc):
    info = GemmPlanInfo()
    s = lib.gemm_plan(ctypes.byref(desc), ctypes.byref(info))
    if s != OK:
        raise GemmError(s, "gemm_plan")
    return info


def gemm_create(desc):
    h = ctypes.c_void_p()
    s = lib.gemm_create(ctypes.byref(h), ctypes.byref(desc))
    if s != OK:
        raise GemmError(s, "gemm_create")
    return h


def gemm_run(handle, A, B, C, D, bias, stream):
    """Pointers are integers (device addresses) or None; stream is a
    cudaStream_t as an integer (torch: ``stream.cuda_stream``) or None."""
    s = lib.gemm_run(handle, A, B, C, D, bias, stream)
    if s != OK:
        raise GemmError(s, "gemm_run")


def gemm_run_ex(handle, A, B, C, D, bias, row_sum, col_sum, abs_max, stream):
    """gemm_run plus the descriptor's reductions into fp32 device arrays
    (pointers as integers; None where not asked for)."""
    s = lib.gemm_run_ex(handle, A, B, C, D, bias, row_sum, col_sum, abs_max, stream)
    if s != OK:
        raise GemmError(s, "gemm_run_ex")


def gemm_run_args(handle, stream, **buffers):
    """Every buffer by name (A, B, C, D, bias, sfa, sfb, row_sum, col_sum,
    abs_max: device addresses as integers, or None)."""
    a = GemmArgs(**{k: v for k, v in buffers.items() if v is not None})
    s = lib.gemm_run_args(handle, ctypes.byref(a), stream)
    if s != OK:
        raise GemmError(s, "gemm_run_args")


def gemm_grouped_create(desc, groups):
    h = ctypes.c_void_p()
    s = lib.gemm_grouped_create(ctypes.byref(h), ctypes.byref(desc), groups)
    if s != OK:
        raise GemmError(s, "gemm_grouped_create")
    return h


def gemm_grouped_run(handle, A, B, C, D, bias, group_rows, stream):
    """group_rows: device address of groups + 1 int64 row offsets."""
    s = lib.gemm_grouped_run(handle, A, B, C, D, bias, group_rows, stream)
    if s != OK:
        raise GemmError(s, "gemm_grouped_run")


def gemm_grouped_run_args(handle, group_rows, stream, **buffers):
    """Grouped run with every buffer by name (see gemm_run_args)."""
    a = GemmArgs(**{k: v for k, v in buffers.items() if v is not None})
    s = lib.gemm_grouped_run_args(handle, ctypes.byref(a), group_rows, stream)
    if s != OK:
        raise GemmError(s, "gemm_grouped_run_args")


def gemm_check(handle):
    s = lib.gemm_check(handle)
    if s != OK:
        raise GemmError(s, "gemm_check")


def gemm_destroy(handle):
    lib.gemm_destroy(handle)


def gemm_set_debug(handle, inject_fault, timeout_ms):
    s = lib.gemm_set_debug(handle, inject_fault, timeout_ms)
    if s != OK:
        raise GemmError(s, "gemm_set_debug")


def gemm_set_stamps(handle, stamps_ptr):
    """Diagnostic timestamps (GEMM_STAMPS builds): a device buffer of 8 uint64 per CTA."""
    s = lib.gemm_set_stamps(handle, stamps_ptr)
    if s != OK:
        raise GemmError(s, "gemm_set_stamps")


BUILD_DEBUG, BUILD_STAMPS = 1, 2


def gemm_build_flags():
    """Bit 0: index-checked (GEMM_DEBUG) build; bit 1: timestamp (GEMM_STAMPS) build."""
    return int(lib.gemm_build_flags())


def gemm_set_schedule(handle, mode):
    s = lib.gemm_set_schedule(handle, mode)
    if s != OK:
        raise GemmError(s, "gemm_set_schedule")


def gemm_get_schedule(handle):
    """(workers, tiles computed whole, K-block iterations of the cut tiles,
    ranges they are cut into)."""
    w, dp, sk, nr = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    s = lib.gemm_get_schedule(handle, ctypes.byref(w), ctypes.byref(dp), ctypes.byref(sk), ctypes.byref(nr))
    if s != OK:
        raise GemmError(s, "gemm_get_schedule")
    return w.value, dp.value, sk.value, nr.value


def gemm_launch_count(handle):
    return int(lib.gemm_launch_count(handle))


def gemm_run_noalloc(desc, A, B, C, D, bias, stream, wait=True):
    """Allocation-free launch (see gemm.h): no handle, scratch in a fixed
    device array; with wait=True it synchronises and reports timeouts."""
    s = lib.gemm_run_noalloc(ctypes.byref(desc), A, B, C, D, bias, stream, 1 if wait else 0)
    if s != OK:
        raise GemmError(s, "gemm_run_noalloc")


class LayoutError(ValueError):
    pass


def _layout_check(rc, what):
    if rc == 2:
        raise LayoutError(f"{what}: undefined (divisibility condition fails)")
    if rc != 0:
        raise LayoutError(f"{what}: error {rc}")


def gemm_layout_query(layout, what):
    out = ctypes.c_int64()
    _layout_check(lib.gemm_layout_query(layout.encode(), what.encode(), ctypes.byref(out)), what)
    return out.value


def gemm_layout_eval(layout, coord):
    coords = list(coord) if isinstance(coord, (tuple, list)) else [coord]
    arr = (ctypes.c_int64 * len(coords))(*coords)
    out = ctypes.c_int64()
    _layout_check(lib.gemm_layout_eval(layout.encode(), arr, len(coords), ctypes.byref(out)), "eval")
    return out.value


def gemm_layout_op(op, a, b=None, m=0):
    buf = ctypes.create_string_buffer(1024)
    _layout_check(lib.gemm_layout_op(op.encode(), a.encode(), None if b is None else b.encode(), m, buf, 1024), op)
    return buf.value.decode()


def gemm_layout_gather_f32(layout, src_ptr, dst_ptr, n, stream):
    _layout_check(lib.gemm_layout_gather_f32(layout.encode(), src_ptr, dst_ptr, n, stream), "gather")

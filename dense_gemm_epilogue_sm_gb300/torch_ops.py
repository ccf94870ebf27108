"""Torch-facing helpers over the C ABI: descriptor construction from a
workload spec and a handle wrapper that passes tensor pointers and the
current CUDA stream.  Argument marshalling only; the GEMM runs in
``libgemm_sm103.so``."""
import torch

from . import (ACT_GELU, ACT_NONE, ACT_RELU, BF16, BIAS_COL, BIAS_NONE, BIAS_ROW, COL_MAJOR, E2M1, E4M3, F16, F32, OP_N,
               OP_T, REDUCE_ABS_MAX, REDUCE_COL_SUM, REDUCE_ROW_SUM, ROW_MAJOR, BLOCK_SCALE_MX, BLOCK_SCALE_NONE, BLOCK_SCALE_NV,
               OUT_SCALE_MX, OUT_SCALE_NONE, OUT_SCALE_NV,
               gemm_check, gemm_create, gemm_destroy, gemm_get_schedule, gemm_grouped_create, gemm_grouped_run,
               gemm_grouped_run_args,
               gemm_launch_count, gemm_run, gemm_run_args, gemm_run_ex, gemm_set_schedule, make_desc)

DTYPE_CODE = {"f32": F32, "f16": F16, "bf16": BF16, "e4m3": E4M3, "e2m1": E2M1}
BLOCK_SCALE_CODE = {"none": BLOCK_SCALE_NONE, "mx": BLOCK_SCALE_MX, "nv": BLOCK_SCALE_NV}
ORDER_CODE = {"row": ROW_MAJOR, "col": COL_MAJOR}
OP_CODE = {"N": OP_N, "T": OP_T}
ACT_CODE = {"none": ACT_NONE, "relu": ACT_RELU, "gelu": ACT_GELU}
REDUCE_CODE = {"row": REDUCE_ROW_SUM, "col": REDUCE_COL_SUM, "amax": REDUCE_ABS_MAX}


def reduce_code(names):
    """'none' or a '+'-joined subset of row, col, amax -> gemm_reduce_t flags."""
    if names in ("", "none"):
        return 0
    code = 0
    for n in names.split("+"):
        code |= REDUCE_CODE[n]
    return code
BIAS_CODE = {"none": BIAS_NONE, "col": BIAS_COL, "row": BIAS_ROW}


def desc_from_spec(spec, scale_a=1.0, scale_b=1.0):
    L = spec.batch
    grouped = getattr(spec, "groups", 0) > 0
    # grouped: A, C, D one matrix each; B and the bias one per group
    stride = lambda w: spec.matrix_elems(w) if (L > 1 and not grouped) or (grouped and w == "b") else 0
    bias_len = 0 if spec.bias == "none" else (spec.N if spec.bias == "col" else spec.M)
    return make_desc(
        spec.M, spec.N, spec.K, L, OP_CODE[spec.op_a], OP_CODE[spec.op_b], ORDER_CODE[spec.order_a],
        ORDER_CODE[spec.order_b], ORDER_CODE[spec.order_c], ORDER_CODE[spec.order_d],
        spec.ld("a"), spec.ld("b"), spec.ld("c"), spec.ld("d"),
        stride("a"), stride("b"), stride("c"), stride("d"), bias_len if (L > 1 or grouped) else 0,
        DTYPE_CODE[spec.dtype_in], DTYPE_CODE[spec.dtype_in], DTYPE_CODE[spec.dtype_d], DTYPE_CODE[spec.dtype_d],
        spec.alpha, spec.beta, scale_a, scale_b, ACT_CODE[spec.act], BIAS_CODE[spec.bias],
        reduce_code(getattr(spec, "reduce", "none")),
        BLOCK_SCALE_CODE[getattr(spec, "block_scale", "none")],
        {"e4m3": OUT_SCALE_MX, "e2m1": OUT_SCALE_NV}.get(spec.dtype_d, OUT_SCALE_NONE),
        scale_d=getattr(spec, "scale_d", 1.0))


def _ptr(t):
    return None if t is None else t.data_ptr()


class GemmOp:
    """One planned GEMM (a handle) bound to a device; call with device tensors."""

    def __init__(self, desc, groups=0):
        self.desc = desc
        self.groups = groups
        self.handle = gemm_grouped_create(desc, groups) if groups else gemm_create(desc)

    def run_grouped(self, A, B, C, D, group_rows, bias=None, stream=None, sfa=None, sfb=None):
        """Grouped handle: group_rows is an int64 device tensor of groups + 1 row offsets;
        sfa / sfb for block-scaled descriptors."""
        s = stream if stream is not None else torch.cuda.current_stream()
        if sfa is not None or sfb is not None:
            gemm_grouped_run_args(self.handle, _ptr(group_rows), s.cuda_stream, A=_ptr(A), B=_ptr(B), C=_ptr(C),
                                  D=_ptr(D), bias=_ptr(bias), sfa=_ptr(sfa), sfb=_ptr(sfb))
        else:
            gemm_grouped_run(self.handle, _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(bias), _ptr(group_rows),
                             s.cuda_stream)

    def __call__(self, A, B, C, D, bias=None, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream()
        gemm_run(self.handle, _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(bias), s.cuda_stream)

    def run_ex(self, A, B, C, D, bias=None, row_sum=None, col_sum=None, abs_max=None, stream=None):
        """With the descriptor's reductions (fp32 device tensors)."""
        s = stream if stream is not None else torch.cuda.current_stream()
        gemm_run_ex(self.handle, _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(bias), _ptr(row_sum), _ptr(col_sum),
                    _ptr(abs_max), s.cuda_stream)

    def run_args(self, A, B, C=None, D=None, bias=None, sfa=None, sfb=None, row_sum=None, col_sum=None,
                 abs_max=None, sfd=None, stream=None):
        """Every buffer by name (device tensors); the call for block-scaled descriptors."""
        s = stream if stream is not None else torch.cuda.current_stream()
        gemm_run_args(self.handle, s.cuda_stream, A=_ptr(A), B=_ptr(B), C=_ptr(C), D=_ptr(D), bias=_ptr(bias),
                      sfa=_ptr(sfa), sfb=_ptr(sfb), row_sum=_ptr(row_sum), col_sum=_ptr(col_sum),
                      abs_max=_ptr(abs_max), sfd=_ptr(sfd))

    def check(self):
        gemm_check(self.handle)

    def set_schedule(self, mode):
        gemm_set_schedule(self.handle, mode)

    @property
    def schedule(self):
        """(workers, tiles computed whole, K-block iterations of the cut tiles,
        ranges they are cut into)."""
        return gemm_get_schedule(self.handle)

    @property
    def launches(self):
        return gemm_launch_count(self.handle)

    def close(self):
        if self.handle is not None:
            gemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

"""The C ABI without a GPU: the library loads, exports every symbol the
public headers declare, validates descriptors and plans them (host only)."""
import ctypes
import glob
import os
import re

import pytest

import dense_gemm_epilogue_sm_gb300 as g
from dense_gemm_epilogue_sm_gb300 import workloads as wl
from dense_gemm_epilogue_sm_gb300.torch_ops import desc_from_spec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names.update(re.findall(r"^GEMM_API\s+[\w\s\*]+?\b(gemm_\w+)\s*\(", text, flags=re.M))
    return names


def test_headers_declare_something():
    names = _declared_symbols()
    assert {"gemm_create", "gemm_run", "gemm_destroy", "gemm_plan", "gemm_layout_eval"} <= names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(g.LIBRARY_PATH)
    missing = [n for n in sorted(_declared_symbols()) if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert set(g.EXPORTED) == _declared_symbols()


def test_status_strings():
    for s in range(7):
        assert g.gemm_status_str(s)
    assert "unknown" in g.gemm_status_str(99)


def _desc(**kw):
    base = dict(M=256, N=512, K=128)
    base.update(kw)
    M, N, K = base.pop("M"), base.pop("N"), base.pop("K")
    return g.make_desc(M, N, K, **base)


def _status(desc):
    info = g.GemmPlanInfo()
    return g.lib.gemm_plan(ctypes.byref(desc), ctypes.byref(info)), info


@pytest.mark.parametrize("field,value,want", [
    ("M", -1, g.ERR_INVALID_ARG), ("K", -5, g.ERR_INVALID_ARG), ("batch", 0, g.ERR_INVALID_ARG),
    ("op_a", 2, g.ERR_INVALID_ARG), ("order_d", 7, g.ERR_INVALID_ARG), ("act", 3, g.ERR_INVALID_ARG),
    ("bias", 9, g.ERR_INVALID_ARG), ("dtype_a", 11, g.ERR_INVALID_ARG),
    ("lda", 64, g.ERR_INVALID_ARG),           # row-major A needs lda >= K = 128
    ("lda", 132, g.ERR_MISALIGNED),           # 264 bytes: not a multiple of 16
    ("ldd", 516, g.ERR_MISALIGNED),
])
def test_rejects_bad_descriptors(field, value, want):
    d = _desc()
    setattr(d, field, value)
    assert _status(d)[0] == want


def test_rejects_unsupported_combinations():
    d = _desc(dtype_a=g.F16, dtype_b=g.BF16)          # one operand type per MMA
    assert _status(d)[0] == g.ERR_UNSUPPORTED
    d = _desc(dtype_a=g.F32, dtype_b=g.F32)
    assert _status(d)[0] == g.ERR_UNSUPPORTED
    d = _desc(beta=1.0, dtype_c=g.F32, dtype_d=g.BF16)
    assert _status(d)[0] == g.ERR_UNSUPPORTED
    d = _desc(beta=1.0, order_c=g.COL_MAJOR, order_d=g.ROW_MAJOR)
    assert _status(d)[0] == g.ERR_UNSUPPORTED
    d = _desc(dtype_d=g.E4M3)
    assert _status(d)[0] == g.ERR_UNSUPPORTED


def test_e4m3_needs_16_element_alignment():
    d = _desc(dtype_a=g.E4M3, dtype_b=g.E4M3, K=136)   # lda = 136 bytes
    assert _status(d)[0] == g.ERR_MISALIGNED
    d = _desc(dtype_a=g.E4M3, dtype_b=g.E4M3, K=144)
    assert _status(d)[0] == g.OK


def test_batch_d_must_not_overlap():
    d = _desc(batch=2)
    d.stride_d = 10
    assert _status(d)[0] == g.ERR_INVALID_ARG


def test_plan_orientation_and_majorness():
    # row-major D: no swap; A row-major op N is K-major; B column-major op N is K-major
    s, info = _status(_desc(order_a=g.ROW_MAJOR, order_b=g.COL_MAJOR, order_d=g.ROW_MAJOR))
    assert s == g.OK and not info.swapped and info.a_k_major and info.b_k_major
    assert (info.kernel_m, info.kernel_n) == (256, 512)
    # column-major D: computed as D^T; the kernel's A is op(B)^T, its B is op(A)
    s, info = _status(_desc(order_a=g.COL_MAJOR, order_b=g.COL_MAJOR, order_c=g.COL_MAJOR, order_d=g.COL_MAJOR))
    assert s == g.OK and info.swapped
    assert (info.kernel_m, info.kernel_n) == (512, 256)
    assert info.a_k_major and not info.b_k_major       # B col-major is K-contiguous; A col-major is M-contiguous
    # transposes flip majorness
    s, info = _status(_desc(op_a=g.OP_T, order_a=g.ROW_MAJOR, lda=256))
    assert s == g.OK and not info.a_k_major


def test_plan_tiles_for_the_named_workloads():
    # (cta_group, tile_m, tile_n, tiles_m, tiles_n, tiles)
    want = {
        "bf16_4096": (2, 256, 256, 16, 16, 256),
        "fused_bf16_8192": (2, 256, 256, 32, 32, 1024),
        "fp8_e4m3_8192": (2, 256, 256, 32, 32, 1024),
        "skinny_65536x256x4096": (2, 256, 256, 256, 1, 256),
        "batched_32x512": (2, 256, 256, 2, 2, 128),
        "tiny_exact_fp16_256": (1, 128, 128, 2, 2, 4),
        "odd_1000_at": (1, 128, 128, 8, 8, 64),
    }
    for name, w in want.items():
        spec = wl.get(name)
        info = g.gemm_plan(desc_from_spec(spec))
        got = (info.cta_group, info.tile_m, info.tile_n, info.tiles_m, info.tiles_n, info.tiles)
        assert got == w, (name, got)
        assert info.tile_k == (128 if spec.dtype_in == "e4m3" else 64)
    info = g.gemm_plan(desc_from_spec(wl.get("tiny_exact_fp16_256")))
    assert info.swapped and info.epi_cols == 32
    info = g.gemm_plan(desc_from_spec(wl.get("odd_1000_at")))
    assert info.a_k_major and info.b_k_major


def test_raster_order_is_a_bijection():
    # The persistent scheduler's tile order, built from the plan exactly as
    # the planner does, must visit every tile once.
    for tm, tn in [(64, 32), (20, 3), (16, 16), (1, 7), (37, 5)]:
        G = min(tm, 16)
        full = tm // G
        tail = tm - full * G
        order = []
        lay_full = f"({G},{tn},{max(full, 1)}):(1,{tm},{G})"
        for t in range(G * tn * full):
            order.append(g.gemm_layout_eval(lay_full, t))
        lay_tail = f"({max(tail, 1)},{tn}):(1,{tm})"
        for t in range(tm * tn - G * tn * full):
            order.append(g.gemm_layout_eval(lay_tail, t) + full * G)
        assert sorted(order) == list(range(tm * tn))
        # consecutive tiles walk G rows of M before the next column of N
        assert [o % tm for o in order[:G]] == list(range(G))


def test_create_without_gpu_reports_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(g.GemmError) as e:
        g.gemm_create(_desc())
    assert e.value.status == g.ERR_NO_DEVICE
    # argument errors are still reported first
    d = _desc()
    d.M = -3
    with pytest.raises(g.GemmError) as e:
        g.gemm_create(d)
    assert e.value.status == g.ERR_INVALID_ARG


def test_block_scaling_needs_e4m3_operands_and_plans_the_mx_kernel():
    d = _desc(dtype_a=g.BF16, dtype_b=g.BF16, block_scale=g.BLOCK_SCALE_MX)
    assert _status(d)[0] == g.ERR_UNSUPPORTED
    d = _desc(dtype_a=g.E4M3, dtype_b=g.E4M3, block_scale=7)
    assert _status(d)[0] == g.ERR_INVALID_ARG
    s, info = _status(_desc(M=4096, N=4096, K=4096, dtype_a=g.E4M3, dtype_b=g.E4M3, block_scale=g.BLOCK_SCALE_MX))
    assert s == g.OK and (info.cta_group, info.tile_m, info.tile_n, info.tile_k, info.stages) == (2, 256, 256, 128, 6)
    s, info = _status(_desc(M=2048, N=1024, K=4096, dtype_a=g.E4M3, dtype_b=g.E4M3, block_scale=g.BLOCK_SCALE_MX))
    assert s == g.OK and (info.cta_group, info.tile_m, info.tile_n, info.tile_k, info.stages) == (2, 256, 128, 128, 6)
    s, info = _status(_desc(M=512, N=512, K=512, dtype_a=g.E4M3, dtype_b=g.E4M3, block_scale=g.BLOCK_SCALE_MX))
    assert s == g.OK and (info.cta_group, info.tile_m, info.tile_n, info.tile_k, info.stages) == (1, 128, 128, 128, 5)


def test_mx_output_needs_e4m3_row_major_d_without_c_or_reductions():
    ok = _desc(dtype_d=g.E4M3, out_scale=g.OUT_SCALE_MX, ldd=512)
    assert _status(ok)[0] == g.OK
    assert _status(_desc(dtype_d=g.E4M3))[0] == g.ERR_UNSUPPORTED                 # e4m3 D needs factors
    assert _status(_desc(out_scale=g.OUT_SCALE_MX))[0] == g.ERR_UNSUPPORTED      # factors need e4m3 D
    assert _status(_desc(dtype_d=g.E4M3, out_scale=g.OUT_SCALE_MX, beta=1.0, dtype_c=g.E4M3))[0] == g.ERR_UNSUPPORTED
    assert _status(_desc(dtype_d=g.E4M3, out_scale=g.OUT_SCALE_MX, order_d=g.COL_MAJOR, ldd=256))[0] == \
        g.ERR_UNSUPPORTED
    assert _status(_desc(dtype_d=g.E4M3, out_scale=g.OUT_SCALE_MX, reduce=g.REDUCE_ROW_SUM))[0] == g.ERR_UNSUPPORTED
    assert _status(_desc(dtype_d=g.E4M3, out_scale=3))[0] == g.ERR_INVALID_ARG


def _nv(**kw):
    base = dict(M=4096, N=4096, K=4096, dtype_a=g.E2M1, dtype_b=g.E2M1, block_scale=g.BLOCK_SCALE_NV,
                lda=4096, ldb=4096, ldd=4096)
    base.update(kw)
    return _desc(**base)


def test_nvfp4_plans_k_major_e2m1_with_256_element_stages():
    s, info = _status(_nv())
    assert s == g.OK and (info.cta_group, info.tile_m, info.tile_n, info.tile_k, info.stages) == (2, 256, 256, 256, 5)
    assert info.a_k_major and info.b_k_major
    s, info = _status(_nv(M=2048, N=1024, ldd=1024))
    assert s == g.OK and (info.cta_group, info.tile_n, info.tile_k, info.stages) == (2, 128, 256, 6)
    # NVFP4 output: 256 x 128 pairs (two accumulators) wherever 64 of them fill the GPU
    s, info = _status(_nv(dtype_d=g.E2M1, out_scale=g.OUT_SCALE_NV, ldd=4096))
    assert s == g.OK and (info.cta_group, info.tile_m, info.tile_n, info.tile_k, info.stages) == (2, 256, 128, 256, 6)
    s, info = _status(_nv(M=512, N=512, K=1000, lda=1024, ldb=1024, ldd=512))
    assert s == g.OK and (info.cta_group, info.tile_n, info.tile_k, info.stages) == (1, 128, 256, 5)
    # column-major D: computed transposed, still K-major on both sides
    s, info = _status(_nv(order_d=g.COL_MAJOR))
    assert s == g.OK and info.swapped and info.a_k_major and info.b_k_major


def test_nvfp4_argument_rules():
    assert _status(_nv(dtype_a=g.E4M3, dtype_b=g.E4M3))[0] == g.ERR_UNSUPPORTED      # e2m1 only
    assert _status(_nv(block_scale=g.BLOCK_SCALE_MX))[0] == g.ERR_UNSUPPORTED        # mx_float8 is e4m3
    assert _status(_nv(block_scale=g.BLOCK_SCALE_NONE))[0] == g.ERR_INVALID_ARG      # e2m1 needs its factors
    assert _status(_nv(dtype_d=g.E2M1))[0] == g.ERR_UNSUPPORTED                      # e2m1 D needs its factors
    assert _status(_nv(K=4095))[0] == g.ERR_UNSUPPORTED                              # odd K: half a byte
    assert _status(_nv(lda=4112))[0] == g.ERR_MISALIGNED                             # 2056 bytes
    assert _status(_nv(order_a=g.COL_MAJOR, lda=4096))[0] == g.ERR_UNSUPPORTED       # MN-major A
    assert _status(_nv(order_b=g.ROW_MAJOR, ldb=4096))[0] == g.ERR_UNSUPPORTED       # MN-major B
    assert _status(_nv(lda=2048))[0] == g.ERR_INVALID_ARG                            # lda < K
    assert _status(_nv(batch=2, stride_a=4096 * 4096 + 16, stride_b=4096 * 4096, stride_d=4096 * 4096))[0] == \
        g.ERR_MISALIGNED


def _grouped_status(desc, groups):
    h = ctypes.c_void_p()
    s = g.lib.gemm_grouped_create(ctypes.byref(h), ctypes.byref(desc), groups)
    if s == g.OK:
        g.lib.gemm_destroy(h)
    return s


def test_grouped_descriptor_rules():
    import torch
    ok = g.ERR_NO_DEVICE if not torch.cuda.is_available() else g.OK
    base = dict(M=4096, N=512, K=256, stride_b=512 * 256)
    assert _grouped_status(_desc(**base), 8) == ok
    assert _grouped_status(_desc(**base), 0) == g.ERR_INVALID_ARG
    assert _grouped_status(_desc(**base), 65536) == g.ERR_INVALID_ARG
    assert _grouped_status(_desc(**dict(base, stride_b=0)), 8) == ok                       # one B for all
    assert _grouped_status(_desc(**dict(base, batch=2)), 8) == g.ERR_INVALID_ARG
    assert _grouped_status(_desc(**dict(base, stride_a=100)), 8) == g.ERR_INVALID_ARG
    assert _grouped_status(_desc(**dict(base, order_d=g.COL_MAJOR, ldd=4096)), 8) == g.ERR_UNSUPPORTED
    assert _grouped_status(_desc(**dict(base, order_a=g.COL_MAJOR, lda=4096)), 8) == g.ERR_UNSUPPORTED   # MN-major A
    assert _grouped_status(_desc(**dict(base, op_a=g.OP_T, order_a=g.COL_MAJOR, lda=256)), 8) == ok   # K-major A
    assert _grouped_status(_desc(**dict(base, reduce=g.REDUCE_ROW_SUM)), 8) == g.ERR_UNSUPPORTED
    assert _grouped_status(_desc(**dict(base, bias=g.BIAS_ROW)), 8) == g.ERR_UNSUPPORTED
    assert _grouped_status(_desc(**dict(base, dtype_a=g.E4M3, dtype_b=g.E4M3, block_scale=g.BLOCK_SCALE_MX)), 8) == ok
    assert _grouped_status(_desc(**dict(base, dtype_a=g.E2M1, dtype_b=g.E2M1, block_scale=g.BLOCK_SCALE_NV,
                                        lda=256, ldb=256)), 8) == ok
    assert _grouped_status(_desc(**dict(base, dtype_a=g.E2M1, dtype_b=g.E2M1, block_scale=g.BLOCK_SCALE_NV,
                                        lda=256, ldb=256, stride_b=512 * 256 + 16)), 8) == g.ERR_MISALIGNED
    assert _grouped_status(_desc(**dict(base, dtype_d=g.E4M3, out_scale=g.OUT_SCALE_MX)), 8) == g.ERR_UNSUPPORTED
    assert _grouped_status(_desc(**dict(base, stride_b=512 * 256 + 4)), 8) == g.ERR_MISALIGNED


def test_nv_output_rules():
    ok = _desc(dtype_d=g.E2M1, out_scale=g.OUT_SCALE_NV, scale_d=0.5, ldd=512)
    s, info = _status(ok)
    assert s == g.OK and info.cta_group in (1, 2)
    assert _status(_desc(dtype_d=g.E2M1, out_scale=g.OUT_SCALE_NV, scale_d=0.0, ldd=512))[0] == g.ERR_INVALID_ARG
    assert _status(_desc(dtype_d=g.E2M1, out_scale=g.OUT_SCALE_NV, scale_d=float("inf"), ldd=512))[0] == \
        g.ERR_INVALID_ARG
    assert _status(_desc(out_scale=g.OUT_SCALE_NV, scale_d=1.0))[0] == g.ERR_UNSUPPORTED        # factors need e2m1 D
    assert _status(_desc(N=511, dtype_d=g.E2M1, out_scale=g.OUT_SCALE_NV, scale_d=1.0, ldd=512))[0] == \
        g.ERR_UNSUPPORTED                                                                       # half a byte
    assert _status(_desc(dtype_d=g.E2M1, out_scale=g.OUT_SCALE_NV, scale_d=1.0, ldd=528))[0] == g.ERR_MISALIGNED
    assert _status(_desc(dtype_d=g.E2M1, out_scale=g.OUT_SCALE_NV, scale_d=1.0, ldd=512, beta=1.0,
                         dtype_c=g.BF16))[0] == g.ERR_UNSUPPORTED
    assert _status(_desc(dtype_d=g.E2M1, out_scale=g.OUT_SCALE_NV, scale_d=1.0, order_d=g.COL_MAJOR,
                         ldd=256))[0] == g.ERR_UNSUPPORTED
    assert _status(_desc(dtype_d=g.E2M1, out_scale=g.OUT_SCALE_NV, scale_d=1.0, ldd=512,
                         reduce=g.REDUCE_ABS_MAX))[0] == g.ERR_UNSUPPORTED

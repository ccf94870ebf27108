"""Parity of the CUDA path (through the C ABI) against the oracle on a GB300.

Small shapes are compared element by element over the whole output; the
full-size workloads are compared on sampled full rows (every 128-row tile,
every column).  Guard bands around D must stay untouched, unwritten elements
show up as NaN canaries, and bounded waits are exercised with a planted
missing load.
"""
import itertools

import numpy as np
import pytest
import torch

import _harness as H
from dense_gemm_epilogue_sm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.init()


def _full_check(spec, exact=False, alias_c=False):
    inputs = wl.make_inputs(spec)
    bits, op = H.run_gpu(spec, inputs, alias_c=alias_c)
    assert op.launches >= (1 if spec.M and spec.N else 0)
    before = None
    if alias_c:   # D's padding is C's padding: it must keep C's values
        c_bits = H.bits_of_tensor(inputs.C)
        before = np.concatenate([c_bits, np.full(bits.shape[0] - c_bits.shape[0], H.CANARY[spec.dtype_d])])
    assert H.untouched_outside(spec, bits, before), "write outside the logical D"
    d = H.logical_d(spec, bits)
    ref = H.oracle_rows(spec, inputs)
    return H.compare(spec, inputs, d, ref, exact=exact)


# --------------------------------------------------------------- exact ----
def test_tiny_exact_fp16_integer_workload_bit_exact():
    spec = wl.get("tiny_exact_fp16_256")
    _full_check(spec, exact=True)


@pytest.mark.parametrize("order_a,order_b,op_a,op_b", [
    ("row", "col", "N", "N"), ("col", "col", "N", "N"), ("row", "row", "N", "N"), ("col", "row", "T", "T"),
    ("row", "row", "T", "N"), ("col", "col", "N", "T")])
@pytest.mark.parametrize("order_d", ["row", "col"])
def test_integer_inputs_bit_exact_all_layouts(order_a, order_b, op_a, op_b, order_d):
    spec = wl.Spec("int_layouts", 200, 136, 264, op_a=op_a, op_b=op_b, order_a=order_a, order_b=order_b,
                   order_c=order_d, order_d=order_d, dtype_in="f16", dtype_d="f32", dist="int4", seed=11, pad=8)
    _full_check(spec, exact=True)


def test_e4m3_integer_draws_fp32_out():
    spec = wl.Spec("int_e4m3", 300, 260, 384, dtype_in="e4m3", dtype_d="f32", dist="int4", seed=12)
    _full_check(spec)


# ------------------------------------------------------------- sweeps ----
SHAPES = [(1, 1, 1), (7, 9, 16), (63, 64, 65), (64, 65, 63), (127, 129, 128), (129, 127, 200), (300, 520, 72),
          (520, 300, 1000), (128, 256, 64), (257, 513, 33)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_shape_sweep_bf16_fused(M, N, K):
    spec = wl.Spec("sweep", M, N, K, alpha=0.5, beta=1.0, act="relu", bias="col", seed=M * 7 + N + K, pad=3)
    _full_check(spec)


@pytest.mark.parametrize("op_a,op_b", list(itertools.product("NT", "NT")))
@pytest.mark.parametrize("order_a,order_b", [("row", "col"), ("col", "row"), ("row", "row"), ("col", "col")])
def test_layouts_bf16(op_a, op_b, order_a, order_b):
    spec = wl.Spec("layouts", 190, 300, 136, op_a=op_a, op_b=op_b, order_a=order_a, order_b=order_b,
                   beta=1.0, bias="col", seed=5, pad=5)
    _full_check(spec)


@pytest.mark.parametrize("dtype_in,dtype_d", [("f16", "f16"), ("f16", "f32"), ("bf16", "f32"), ("e4m3", "bf16"),
                                              ("e4m3", "f16"), ("bf16", "f16")])
@pytest.mark.parametrize("order_d", ["row", "col"])
def test_dtypes(dtype_in, dtype_d, order_d):
    dist = "uniform1" if dtype_in == "e4m3" else "normal"
    spec = wl.Spec("dtypes", 333, 290, 256, dtype_in=dtype_in, dtype_d=dtype_d, order_c=order_d, order_d=order_d,
                   beta=0.75, bias="row", act="relu", alpha=1.5, dist=dist, seed=9)
    _full_check(spec)


@pytest.mark.parametrize("op_a,op_b,order_a,order_b", [("N", "N", "row", "row"), ("T", "T", "col", "row"),
                                                       ("N", "T", "col", "col")])
def test_e4m3_layouts(op_a, op_b, order_a, order_b):
    spec = wl.Spec("e4m3_layouts", 256, 384, 256, op_a=op_a, op_b=op_b, order_a=order_a, order_b=order_b,
                   dtype_in="e4m3", dist="uniform1", seed=21)
    _full_check(spec)


def test_batched_with_bias_and_c():
    spec = wl.Spec("batched", 200, 136, 96, batch=3, beta=1.0, bias="col", act="relu", seed=13, pad=8)
    _full_check(spec)


def test_d_aliases_c():
    spec = wl.Spec("alias", 257, 300, 128, beta=1.0, alpha=2.0, seed=14)
    _full_check(spec, alias_c=True)


def test_k_zero_gives_epilogue_of_c_and_bias():
    spec = wl.Spec("kzero", 130, 200, 0, beta=1.0, bias="col", seed=15)
    _full_check(spec)


def test_empty_m_or_n_launches_nothing():
    for M, N in [(0, 64), (64, 0)]:
        spec = wl.Spec("empty", M, N, 64, seed=16)
        inputs = wl.make_inputs(spec)
        bits, op = H.run_gpu(spec, inputs)
        assert op.launches == 0
        assert H.untouched_outside(spec, bits)


def test_deterministic_run_to_run():
    spec = wl.Spec("determinism", 600, 700, 1000, beta=1.0, bias="col", seed=17)
    inputs = wl.make_inputs(spec)
    a, op = H.run_gpu(spec, inputs)
    b, _ = H.run_gpu(spec, inputs, op=op)
    assert np.array_equal(a, b)


# ------------------------------------------------------ CTA pairs ---------
PAIR_SPECS = [
    wl.Spec("pair_fused", 2100, 2100, 200, alpha=0.5, beta=1.0, act="relu", bias="col", seed=41, pad=3),
    wl.Spec("pair_colmajor_d", 2050, 2300, 136, op_a="T", order_a="col", order_b="row", order_c="col",
            order_d="col", beta=1.0, bias="row", seed=42),
    wl.Spec("pair_mn_major", 2304, 2048, 128, order_a="col", order_b="row", dtype_in="f16", dtype_d="f32",
            seed=43),
    wl.Spec("pair_e4m3", 2100, 2060, 256, dtype_in="e4m3", dist="uniform1", bias="col", seed=44),
    wl.Spec("pair_batched", 256, 256, 96, batch=64, beta=1.0, seed=45),
    wl.Spec("pair_exact", 2048, 2048, 264, order_a="col", order_b="col", order_c="col", order_d="col",
            dtype_in="f16", dtype_d="f32", dist="int4", seed=46),
]


@pytest.mark.parametrize("spec", PAIR_SPECS, ids=lambda s: s.name)
def test_cta_pair_kernel(spec):
    from dense_gemm_epilogue_sm_gb300 import gemm_plan
    from dense_gemm_epilogue_sm_gb300.torch_ops import desc_from_spec
    assert gemm_plan(desc_from_spec(spec)).cta_group == 2
    _full_check(spec, exact=spec.dist == "int4")


def test_cta_pair_odd_stage_count_wraps_the_ring():
    # K = 136 bf16 is 3 K blocks per tile; 256 pair tiles over the pairs give
    # 3 or 4 tiles each, so a pair issues 9 or 12 stages: the ring (6 stages,
    # released in groups) wraps and the last group is only partly refilled.
    # The run must finish without any bounded wait running out.
    from dense_gemm_epilogue_sm_gb300 import gemm_plan
    from dense_gemm_epilogue_sm_gb300.torch_ops import desc_from_spec
    spec = wl.Spec("pair_odd_stages", 4096, 4096, 136, beta=1.0, seed=47)
    assert gemm_plan(desc_from_spec(spec)).cta_group == 2
    inputs = wl.make_inputs(spec)
    bits, op = H.run_gpu(spec, inputs)          # raises on a timeout status
    d = H.logical_d(spec, bits)
    rows = H.sample_rows(spec, per_tile=2)
    H.compare(spec, inputs, d, H.oracle_rows(spec, inputs, rows), rows=rows)


# ---------------------------------------------------- full workloads ------
@pytest.mark.parametrize("name", ["odd_1000_at", "batched_32x512"])
def test_workload_full_parity(name):
    _full_check(wl.get(name))


@pytest.mark.parametrize("name", ["bf16_4096", "fused_bf16_8192", "plain_bf16_8192", "fp8_e4m3_8192",
                                  "skinny_65536x256x4096"])
def test_workload_sampled_rows(name):
    spec = wl.get(name)
    inputs = wl.make_inputs(spec)
    bits, op = H.run_gpu(spec, inputs)
    assert H.untouched_outside(spec, bits)
    d = H.logical_d(spec, bits)
    full = H.from_bits(d.reshape(-1), spec.dtype_d)
    assert np.isfinite(full).all(), "unwritten output elements"
    rows = H.sample_rows(spec)
    ref = H.oracle_rows(spec, inputs, rows)
    H.compare(spec, inputs, d, ref, rows=rows)


# ---------------------------------------------------- bounded waits -------
def test_missing_load_times_out_and_context_survives():
    from dense_gemm_epilogue_sm_gb300 import ERR_TIMEOUT, GemmError, gemm_set_debug
    spec = wl.Spec("timeout", 256, 512, 256, seed=18)
    inputs = wl.make_inputs(spec)
    from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec
    op = GemmOp(desc_from_spec(spec))
    gemm_set_debug(op.handle, 1, 100)
    dev = torch.device("cuda", 0)
    A, B = inputs.A.to(dev), inputs.B.to(dev)
    D = H.canary_buffer(spec)
    op(A, B, None, D)
    with pytest.raises(GemmError) as e:
        op.check()
    assert e.value.status == ERR_TIMEOUT
    # the context is still usable and the same handle computes correctly again
    gemm_set_debug(op.handle, 0, 2000)
    bits, _ = H.run_gpu(spec, inputs, op=op)
    H.compare(spec, inputs, H.logical_d(spec, bits), H.oracle_rows(spec, inputs))


# ------------------------------------------------------- layout on GPU ----
@pytest.mark.parametrize("layout", ["((16,16),(16,8)):((128,1),(2048,16))", "(4,(2,4)):(2,(1,8))",
                                    "((2,2),3):((24,2),8)"])
def test_layout_gather_device_matches_host(layout):
    from dense_gemm_epilogue_sm_gb300 import gemm_layout_eval, gemm_layout_gather_f32, gemm_layout_query
    n = gemm_layout_query(layout, "size")
    cos = gemm_layout_query(layout, "cosize")
    src = torch.arange(cos, dtype=torch.float32, device="cuda")
    dst = torch.full((n,), -1.0, dtype=torch.float32, device="cuda")
    gemm_layout_gather_f32(layout, src.data_ptr(), dst.data_ptr(), n, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = [gemm_layout_eval(layout, i) for i in range(n)]
    assert dst.cpu().to(torch.int64).tolist() == host

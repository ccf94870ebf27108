"""K-split work schedules (gemm_set_schedule: stream-K, split tail) on the GPU.

The split changes only which worker sums which K blocks of a tile; the
result is the same GEMM.  Every case below checks that tiles really are cut
between workers, then compares against the oracle (sampled rows in every
tile, or every element), against the data-parallel split where the sums are
exact, across new inputs on the same handle (a stale partial-sum flag would
let an owner read the previous launch's partials), and after a timed-out
launch.
"""
import dataclasses

import numpy as np
import pytest
import torch

import _harness as H
import dense_gemm_epilogue_sm_gb300 as g
from dense_gemm_epilogue_sm_gb300 import workloads as wl
from dense_gemm_epilogue_sm_gb300.torch_ops import GemmOp, desc_from_spec

pytestmark = pytest.mark.gpu

SPECS = [
    wl.Spec("sk_pair_ragged", 2300, 2310, 1000, alpha=0.5, beta=1.0, act="relu", bias="col", seed=41, pad=3),
    wl.Spec("sk_pair_f32_colmajor", 2200, 2600, 768, op_a="T", order_a="col", order_c="col", order_d="col",
            dtype_d="f32", beta=0.75, bias="row", seed=42),
    wl.Spec("sk_pair_e4m3", 2560, 2560, 2048, dtype_in="e4m3", dist="uniform1", seed=43),
    wl.Spec("sk_pair_batched", 512, 1024, 1024, batch=12, beta=1.0, seed=44),
    wl.Spec("sk_single_n128", 20000, 128, 520, bias="col", act="relu", seed=45),
    # fewer tiles than workers: the split cuts a single, ragged wave
    wl.Spec("sk_one_wave_pair", 768, 1024, 2048, beta=1.0, bias="row", seed=47),
    wl.Spec("sk_one_wave_ragged", 1000, 1000, 1000, op_a="T", order_a="col", act="relu", seed=48, pad=2),
]


def _op(spec, inputs, mode):
    op = GemmOp(desc_from_spec(spec, inputs.scale_a, inputs.scale_b))
    op.set_schedule(mode)
    return op


def _num_kb(spec):
    info = g.gemm_plan(desc_from_spec(spec))
    return -(-spec.K // info.tile_k)


def _cut_tiles(op, spec):
    """Tiles whose K blocks are shared by two or more workers."""
    workers, dp, sk, ranges = op.schedule
    kb = _num_kb(spec)
    starts = [sk * j // ranges for j in range(1, ranges)]
    return {dp + s // kb for s in starts if s % kb and s < sk}


def _run(op, spec, inputs):
    bits, _ = H.run_gpu(spec, inputs, op=op)
    assert H.untouched_outside(spec, bits), "write outside the logical D"
    return bits


MODES = {"stream_k": g.SCHED_STREAM_K, "split_tail": g.SCHED_SPLIT_TAIL}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_split_matches_oracle(spec, mode):
    inputs = wl.make_inputs(spec)
    op = _op(spec, inputs, MODES[mode])
    assert _cut_tiles(op, spec), "the split cuts no tile: the case tests nothing"
    bits = _run(op, spec, inputs)
    d = H.logical_d(spec, bits)
    assert np.isfinite(H.from_bits(d.reshape(-1), spec.dtype_d)).all(), "unwritten output elements"
    rows = H.sample_rows(spec)
    H.compare(spec, inputs, d, H.oracle_rows(spec, inputs, rows), rows=rows)
    op.close()


@pytest.mark.parametrize("size", [2304, 1024])
@pytest.mark.parametrize("mode", list(MODES))
def test_split_integer_sums_equal_data_parallel_bit_for_bit(mode, size):
    # integers in [-4, 4] with K = 1024: every partial and total sum is exact
    # (2304: a full wave and a ragged one; 1024: a single ragged wave)
    spec = wl.Spec("sk_int_exact", size, size, 1024, dtype_in="f16", dtype_d="f32", dist="int4", seed=46)
    inputs = wl.make_inputs(spec)
    sk_op = _op(spec, inputs, MODES[mode])
    assert _cut_tiles(sk_op, spec)
    dp_op = _op(spec, inputs, g.SCHED_DATA_PARALLEL)
    assert dp_op.schedule[2] == 0
    sk_bits = H.logical_d(spec, _run(sk_op, spec, inputs))
    dp_bits = H.logical_d(spec, _run(dp_op, spec, inputs))
    assert np.array_equal(sk_bits, dp_bits)
    H.compare(spec, inputs, sk_bits, H.oracle_rows(spec, inputs), exact=True)


def test_new_inputs_on_the_same_handle_and_repeat_launches():
    spec = SPECS[0]
    op = None
    for seed in (51, 52):
        s = dataclasses.replace(spec, seed=seed)
        inputs = wl.make_inputs(s)
        if op is None:
            op = _op(s, inputs, g.SCHED_STREAM_K)
        bits, _ = H.run_gpu(s, inputs, op=op, repeat=3)
        d = H.logical_d(s, bits)
        rows = H.sample_rows(s)
        H.compare(s, inputs, d, H.oracle_rows(s, inputs, rows), rows=rows)
    op.close()


def test_timed_out_launch_leaves_the_handle_usable():
    spec = SPECS[3]
    inputs = wl.make_inputs(spec)
    op = _op(spec, inputs, g.SCHED_STREAM_K)
    assert _cut_tiles(op, spec)
    g.gemm_set_debug(op.handle, 1, 100)
    dev = torch.device("cuda", 0)
    A, B, C = inputs.A.to(dev), inputs.B.to(dev), inputs.C.to(dev)
    D = H.canary_buffer(spec)
    op(A, B, C, D)
    with pytest.raises(g.GemmError) as e:
        op.check()
    assert e.value.status == g.ERR_TIMEOUT
    g.gemm_set_debug(op.handle, 0, 2000)
    bits = _run(op, spec, inputs)
    d = H.logical_d(spec, bits)
    rows = H.sample_rows(spec)
    H.compare(spec, inputs, d, H.oracle_rows(spec, inputs, rows), rows=rows)
    op.close()


@pytest.mark.parametrize("name", ["fused_bf16_8192", "bf16_4096", "fp8_e4m3_8192", "skinny_65536x256x4096",
                                  "batched_32x512", "odd_1000_at", "tiny_exact_fp16_256"])
def test_auto_schedule_follows_the_stated_rule(name):
    spec = wl.get(name)
    op = GemmOp(desc_from_spec(spec))
    workers, dp, sk, ranges = op.schedule
    info = g.gemm_plan(desc_from_spec(spec))
    tiles, kb = info.tiles, _num_kb(spec)
    op.set_schedule(g.SCHED_DATA_PARALLEL)
    assert op.schedule[1:] == (tiles, 0, 0)
    dp_workers = op.schedule[0]
    # S, the workers the GPU holds at once: the data-parallel worker count
    # when there are more tiles; else every SM's CTA (or pair: all fit at once)
    slots = dp_workers if tiles > dp_workers else \
        torch.cuda.get_device_properties(0).multi_processor_count // info.cta_group
    waves, rest = divmod(tiles, slots)
    pieces = min(slots // rest, kb) if rest else 0
    use = waves >= 1 and rest != 0 and pieces >= 2 and kb // pieces >= 4
    want = (waves * slots, rest * kb, rest * pieces) if use else (tiles, 0, 0)
    assert (dp, sk, ranges) == want
    assert workers == (max(dp_workers, ranges) if use else dp_workers)
    op.close()

"""The C++ layout module (through the C ABI) against the pages' worked
examples and against the independent CPU layout oracle (no GPU needed)."""
import random

import pytest

import dense_gemm_epilogue_sm_gb300 as g
from _golden import ints, parse_coord, records
from oracle import layout_ref as lr


def _coord_list(c):
    if isinstance(c, int):
        return c
    # top-level coordinate: each mode given as an int; nested coordinates
    # are evaluated through the oracle's splitting rule only, so flatten them
    # here to the 1-D coordinate of that mode
    return list(c)


@pytest.mark.parametrize("lineno,kind,fields", records(), ids=lambda x: str(x))
def test_golden_example(lineno, kind, fields):
    if kind == "table":
        lay, rows, cols, want = fields[0], int(fields[1]), int(fields[2]), ints(fields[3])
        got = [g.gemm_layout_eval(lay, (i, j)) for i in range(rows) for j in range(cols)]
        assert got == want
    elif kind == "eval":
        c = parse_coord(fields[1])
        if isinstance(c, tuple) and any(isinstance(x, tuple) for x in c):
            # fully nested coordinate: map each nested mode coordinate to its 1-D form
            lay = lr.parse(fields[0])
            flat = []
            for i, ci in enumerate(c):
                sub = lay.mode(i)
                if isinstance(ci, tuple):
                    ext = [lr.product(s) for s in sub.shape]
                    v, mul = 0, 1
                    for x, e in zip(ci, ext):
                        v += x * mul
                        mul *= e
                    flat.append(v)
                else:
                    flat.append(ci)
            c = tuple(flat)
        assert g.gemm_layout_eval(fields[0], c) == int(fields[2])
    elif kind == "values":
        want = ints(fields[1])
        assert [g.gemm_layout_eval(fields[0], i) for i in range(len(want))] == want
    elif kind in ("size", "cosize", "rank"):
        assert g.gemm_layout_query(fields[0], kind) == int(fields[1])
    elif kind == "mode":
        assert g.gemm_layout_op("mode", fields[0], None, int(fields[1])) == fields[2]
    elif kind == "coalesce":
        assert g.gemm_layout_op("coalesce", fields[0]) == fields[1]
    elif kind == "composition":
        assert g.gemm_layout_op("composition", fields[0], fields[1]) == fields[2]
    elif kind == "composition_fails":
        with pytest.raises(g.LayoutError):
            g.gemm_layout_op("composition", fields[0], fields[1])
    elif kind == "complement":
        assert g.gemm_layout_op("complement", fields[0], None, int(fields[1])) == fields[2]
    elif kind == "logical_divide":
        assert g.gemm_layout_op("logical_divide", fields[0], fields[1]) == fields[2]
    elif kind == "zipped_divide":
        assert g.gemm_layout_op("zipped_divide", fields[0], fields[1]) == fields[2]
    else:
        raise AssertionError(kind)


def test_parse_errors():
    for bad in ["", "4", "(4,8):(1)", "(4,8:(1,4)", "0:1", "(4,x):(1,4)"]:
        with pytest.raises(g.LayoutError):
            g.gemm_layout_query(bad, "size")


def _rand_layout(rng):
    k = rng.randint(1, 4)
    shape = tuple(rng.choice([1, 2, 3, 4, 8]) for _ in range(k))
    stride = tuple(rng.choice([0, 1, 2, 4, 8, 16, 32]) for _ in range(k))
    if rng.random() < 0.3 and k >= 2:
        return lr.Layout((shape[0], shape[1:]), (stride[0], stride[1:]))
    return lr.Layout(shape, stride)


def test_random_layouts_agree_with_oracle():
    rng = random.Random(1234)
    compared = 0
    for _ in range(400):
        a = _rand_layout(rng)
        text = repr(a)
        assert g.gemm_layout_query(text, "size") == a.size()
        for i in range(min(a.size(), 64)):
            assert g.gemm_layout_eval(text, i) == a(i)
        assert g.gemm_layout_op("coalesce", text) == repr(lr.coalesce(a))
        b = lr.Layout(rng.choice([1, 2, 4]), rng.choice([1, 2, 4]))
        try:
            want = repr(lr.composition(a, b))
        except lr.LayoutError:
            with pytest.raises(g.LayoutError):
                g.gemm_layout_op("composition", text, repr(b))
        else:
            assert g.gemm_layout_op("composition", text, repr(b)) == want
            compared += 1
        m = rng.choice([16, 32, 64, 128])
        try:
            want = repr(lr.complement(a, m))
        except lr.LayoutError:
            with pytest.raises(g.LayoutError):
                g.gemm_layout_op("complement", text, None, m)
        else:
            assert g.gemm_layout_op("complement", text, None, m) == want
    assert compared > 100


def test_zipped_divide_agrees_with_oracle():
    for shape, stride, tiles in [((256, 128), (128, 1), (16, 16)), ((64, 48), (1, 64), (8, 16)),
                                 ((16, 8), (1, 16), (4, 2)), ((12, 6), (6, 1), (3, 2))]:
        a = lr.Layout(shape, stride)
        want = repr(lr.zipped_divide(a, [lr.Layout(t) for t in tiles]))
        assert g.gemm_layout_op("zipped_divide", repr(a), ",".join(map(str, tiles))) == want

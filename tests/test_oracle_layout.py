"""Pins the CPU layout-algebra oracle to the pages' worked examples and to
properties the definitions fix (no GPU needed)."""
import random

import pytest

from _golden import ints, parse_coord, records
from oracle import layout_ref as lr


def _tiler(text):
    return [lr.Layout(int(x)) for x in text.split(",")]


@pytest.mark.parametrize("lineno,kind,fields", records(), ids=lambda x: str(x))
def test_golden_example(lineno, kind, fields):
    if kind == "table":
        lay, rows, cols, want = lr.parse(fields[0]), int(fields[1]), int(fields[2]), ints(fields[3])
        got = [lay((i, j)) for i in range(rows) for j in range(cols)]
        assert got == want
    elif kind == "eval":
        assert lr.parse(fields[0])(parse_coord(fields[1])) == int(fields[2])
    elif kind == "values":
        lay, want = lr.parse(fields[0]), ints(fields[1])
        assert [lay(i) for i in range(len(want))] == want
    elif kind == "size":
        assert lr.parse(fields[0]).size() == int(fields[1])
    elif kind == "cosize":
        assert lr.parse(fields[0]).cosize() == int(fields[1])
    elif kind == "rank":
        assert lr.parse(fields[0]).rank() == int(fields[1])
    elif kind == "mode":
        assert lr.parse(fields[0]).mode(int(fields[1])) == lr.parse(fields[2])
    elif kind == "coalesce":
        assert repr(lr.coalesce(lr.parse(fields[0]))) == repr(lr.parse(fields[1]))
    elif kind == "composition":
        a, b = lr.parse(fields[0]), lr.parse(fields[1])
        r = lr.composition(a, b)
        assert repr(r) == repr(lr.parse(fields[2]))
        assert all(r(i) == a(b(i)) for i in range(b.size()))
    elif kind == "composition_fails":
        with pytest.raises(lr.LayoutError):
            lr.composition(lr.parse(fields[0]), lr.parse(fields[1]))
    elif kind == "complement":
        got = lr.complement(lr.parse(fields[0]), int(fields[1]))
        assert repr(got) == repr(lr.parse(fields[2]))
    elif kind == "logical_divide":
        got = lr.logical_divide(lr.parse(fields[0]), lr.parse(fields[1]))
        assert repr(got) == repr(lr.parse(fields[2]))
    elif kind == "zipped_divide":
        got = lr.zipped_divide(lr.parse(fields[0]), _tiler(fields[1]))
        assert repr(got) == repr(lr.parse(fields[2]))
    else:
        raise AssertionError(f"unknown record kind {kind} (line {lineno})")


def test_logical_divide_tiles_printed():
    # "CuTe's layout algebra", "Complement and division": the six tiles of
    # logical_divide(24:1, 4:2).
    d = lr.logical_divide(lr.Layout(24), lr.parse("4:2"))
    tiles = [[d((i, k)) for i in range(4)] for k in range(d.mode(1).size())]
    assert tiles == [[0, 2, 4, 6], [1, 3, 5, 7], [8, 10, 12, 14], [9, 11, 13, 15],
                     [16, 18, 20, 22], [17, 19, 21, 23]]


def test_complement_covers_once():
    a = lr.parse("4:2")
    both = lr.concat(a, lr.complement(a, 24))
    assert sorted(both(i) for i in range(24)) == list(range(24))


def test_partition_printed_values():
    # "CuTe's layout algebra", "From tiles to threads": a 16x8 column-major
    # tile.  One 2x2 block per thread: threads 0, 1, 8 own these values; a
    # (16,2) thread layout: threads 0, 1, 16 own these.
    tile = lr.Layout((16, 8))
    z = lr.zipped_divide(tile, [lr.Layout(2), lr.Layout(2)])
    assert [[z((v, t)) for v in range(4)] for t in (0, 1, 8)] == [[0, 1, 16, 17], [2, 3, 18, 19], [32, 33, 48, 49]]
    thr = lr.Layout((16, 2))
    got = [[lr.local_partition_index(tile, thr, t, v) for v in range(4)] for t in (0, 1, 16)]
    assert got == [[0, 32, 64, 96], [1, 33, 65, 97], [16, 48, 80, 112]]


def _sectors(addresses, elem_bytes=4):
    return len({a * elem_bytes // 32 for a in addresses})


def test_sector_utilisation_printed():
    # Same section: 8 sectors at 50% for one fp32 per thread of a 2x2 block,
    # 8 sectors at 100% for two, 4 sectors at 100% for the (16,2) threads.
    tile = lr.Layout((16, 8))
    z = lr.zipped_divide(tile, [lr.Layout(2), lr.Layout(2)])
    one = [z((0, t)) for t in range(32)]
    two = [z((v, t)) for t in range(32) for v in (0, 1)]
    assert _sectors(one) == 8 and len(one) * 4 / (8 * 32) == 0.5
    assert _sectors(two) == 8 and len(two) * 4 / (8 * 32) == 1.0
    thr = lr.Layout((16, 2))
    q = [lr.local_partition_index(tile, thr, t, 0) for t in range(32)]
    assert _sectors(q) == 4


# "CuTe's layout algebra", "A Tensor Core's register layout is a layout too":
# the (thread, value) layouts of mma.sync m16n8k16 against the PTX fragment
# tables (g = lane/4, t = lane%4).
MMA_A = lr.parse("((4,8),(2,2,2)):((32,1),(16,8,128))")
MMA_B = lr.parse("((4,8),(2,2)):((16,1),(8,64))")
MMA_C = lr.parse("((4,8),(2,2)):((32,1),(16,8))")


def test_mma_tv_layouts_match_ptx_tables():
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for i in range(8):
            idx = MMA_A((lane, i))
            assert (idx % 16, idx // 16) == (g + 8 * (i // 2 % 2), 2 * t + i % 2 + 8 * (i // 4))
        for i in range(4):
            idx = MMA_B((lane, i))
            assert (idx // 8, idx % 8) == (2 * t + i % 2 + 8 * (i // 2), g)
            idx = MMA_C((lane, i))
            assert (idx % 16, idx // 16) == (g + 8 * (i // 2), 2 * t + i % 2)


def test_mma_printed_rows():
    rc = lambda idx: (idx % 16, idx // 16)
    assert [rc(MMA_A((0, i))) for i in range(8)] == [(0, 0), (0, 1), (8, 0), (8, 1), (0, 8), (0, 9), (8, 8), (8, 9)]
    assert [rc(MMA_A((1, i))) for i in range(8)] == [(0, 2), (0, 3), (8, 2), (8, 3), (0, 10), (0, 11), (8, 10), (8, 11)]
    assert [rc(MMA_A((4, i))) for i in range(8)] == [(1, 0), (1, 1), (9, 0), (9, 1), (1, 8), (1, 9), (9, 8), (9, 9)]
    owner = {rc(MMA_C((l, i))): l for l in range(32) for i in range(4)}
    assert [[owner[(r, c)] for c in range(8)] for r in range(4)] == [
        [0, 0, 1, 1, 2, 2, 3, 3], [4, 4, 5, 5, 6, 6, 7, 7],
        [8, 8, 9, 9, 10, 10, 11, 11], [12, 12, 13, 13, 14, 14, 15, 15]]
    # exercise 3: lane 5, value 3 -> index 57 = row 9, column 3
    assert MMA_C((5, 3)) == 57 and rc(57) == (9, 3)


def test_tiled_copy_tv_exercise():
    # Exercise 2: TV ((8,16),8):((128,1),16) over a 16x64 column-major tile;
    # thread t owns row t/8, columns 8(t%8) .. 8(t%8)+7.
    tv = lr.parse("((8,16),8):((128,1),16)")
    for t in range(128):
        cells = sorted((tv((t, v)) % 16, tv((t, v)) // 16) for v in range(8))
        assert cells == [(t // 8, 8 * (t % 8) + j) for j in range(8)]


def test_zipped_divide_matches_hand_tiling():
    # "cute_layouts.cu", gate 2: a 256x128 row-major matrix divided into 16x16
    # tiles gives (tileRow*16 + r)*128 + tileCol*16 + c at every element.
    a = lr.Layout((256, 128), (128, 1))
    z = lr.zipped_divide(a, [lr.Layout(16), lr.Layout(16)])
    for tr in range(16):
        for tc in range(8):
            for r in range(16):
                for c in range(16):
                    assert z(((r, c), (tr, tc))) == (tr * 16 + r) * 128 + tc * 16 + c


def test_zipped_mode0_equals_composition():
    # "cute_layouts.cu", gate 3: layout<0>(zipped_divide(A, B)) == A o B.
    a = lr.Layout((256, 128), (128, 1))
    tiler = [lr.Layout(16), lr.Layout(16)]
    z = lr.zipped_divide(a, tiler)
    comp = lr.composition(a, tiler)
    inner = z.mode(0)
    assert all(inner(i) == comp(i) for i in range(256))


def _random_layout(rng, max_modes=4):
    shape, stride = [], []
    for _ in range(rng.randint(1, max_modes)):
        shape.append(rng.choice([1, 2, 3, 4, 6, 8]))
        stride.append(rng.choice([0, 1, 2, 3, 4, 8, 16, 24]))
    return lr.Layout(tuple(shape), tuple(stride))


def test_coalesce_preserves_function_random():
    rng = random.Random(7)
    for _ in range(500):
        a = _random_layout(rng)
        c = lr.coalesce(a)
        assert c.size() == a.size()
        assert all(c(i) == a(i) for i in range(a.size()))


def test_composition_definition_random():
    # Whenever composition is defined it must satisfy R(i) = A(B(i)) on B's domain.
    rng = random.Random(11)
    checked = 0
    for _ in range(3000):
        a = lr.Layout(tuple(rng.choice([2, 4, 8]) for _ in range(rng.randint(1, 3))))
        a = lr.Layout(a.shape, tuple(rng.choice([1, 2, 4, 16]) * s for s in lr.leaves(a.stride)))
        b = lr.Layout(rng.choice([1, 2, 4, 8]), rng.choice([1, 2, 4, 8]))
        if b.size() * max(1, b.stride) > a.size() * 4:
            continue
        try:
            r = lr.composition(a, b)
        except lr.LayoutError:
            continue
        checked += 1
        assert all(r(i) == a(b(i)) for i in range(b.size()))
    assert checked > 200


def test_complement_bijection_random():
    # For A = (s0,s1):(d0, d0*s0*k) every stride is a multiple of the reach of
    # the modes below it, so complement(A, M) is defined; for M a multiple of
    # the top reach s1*d1, (A, A*) must cover [0, M) exactly once.
    rng = random.Random(3)
    for _ in range(300):
        s0, s1 = rng.choice([1, 2, 4]), rng.choice([2, 3])
        d0, k, r = rng.choice([1, 2, 3]), rng.choice([1, 2]), rng.choice([1, 2, 3])
        a = lr.Layout((s0, s1), (d0, d0 * s0 * k))
        m = s1 * d0 * s0 * k * r
        both = lr.concat(a, lr.complement(a, m))
        assert both.size() == m
        assert sorted(both(i) for i in range(m)) == list(range(m)), (a, m)

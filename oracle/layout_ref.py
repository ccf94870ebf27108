"""CPU reference of the shape:stride layout algebra.  TEST INFRASTRUCTURE ONLY.

Only the test suite imports this.  It is an independent restatement, in plain
Python, of the definitions on the page "CuTe's layout algebra" (Advanced CUDA
notebook); it shares nothing with the C++ layout module of the CUDA path.

Definitions followed (section of that page in brackets):

* [A layout: shape and stride] A layout is a pair of congruent (possibly
  nested) integer tuples.  It maps a coordinate to the inner product of the
  coordinate with the stride.  An integer coordinate against a tuple shape is
  first split colexicographically (mode 0 fastest); the last mode is not
  reduced modulo its extent, so a coordinate past the end continues along it.
  size = product of the shape, cosize = L(size-1) + 1, rank = number of
  top-level modes; the default stride is the compact column-major one.
* [Coalescing] coalesce flattens, drops extent-1 modes, and merges a mode into
  its predecessor when predecessor.shape * predecessor.stride equals its
  stride.  It preserves L(i) for every one-dimensional i.
* [Composition: a layout over a layout] R = A o B, R(c) = A(B(c)), with B's
  shape.  For one mode n:d of B: walk A's coalesced modes, first stepping over
  d elements, then collecting n; undefined (an error here) unless, at every
  mode, the extent and the remaining step divide one another and the count
  still wanted is a multiple of what the mode supplies.  A's last mode is
  unbounded.  A tuple of layouts as B composes mode by mode.
* [Complement and division] complement(A, M) lays out the indices of [0, M)
  that A does not reach, in increasing stride order, so that (A, A*) covers
  [0, M) exactly once; logical_divide(A, B) = A o (B, complement(B, size A));
  zipped_divide regroups a mode-wise division as ((tile modes), (rest modes)).
* [From tiles to threads] local_tile fixes the rest (tile-index) mode of a
  zipped division to a CTA's tile coordinate; local_partition fixes the tile
  mode to a thread's coordinate.
"""
from __future__ import annotations

from functools import reduce


class LayoutError(ValueError):
    """Raised where the pages call an operation undefined (divisibility)."""


def _is_tup(x) -> bool:
    return isinstance(x, tuple)


def leaves(t):
    """Leaves of an integer tuple, left to right."""
    if not _is_tup(t):
        return [t]
    out = []
    for x in t:
        out.extend(leaves(x))
    return out


def product(t) -> int:
    return reduce(lambda a, b: a * b, leaves(t), 1)


def _same_structure(a, b) -> bool:
    if _is_tup(a) != _is_tup(b):
        return False
    if not _is_tup(a):
        return True
    return len(a) == len(b) and all(_same_structure(x, y) for x, y in zip(a, b))


def _regroup(flat_iter, like):
    """Rebuilds the nesting of `like` from an iterator of leaves."""
    if not _is_tup(like):
        return next(flat_iter)
    return tuple(_regroup(flat_iter, x) for x in like)


def fmt(t) -> str:
    if _is_tup(t):
        return "(" + ",".join(fmt(x) for x in t) + ")"
    return str(t)


class Layout:
    __slots__ = ("shape", "stride")

    def __init__(self, shape, stride=None):
        if stride is None:
            running, flat = 1, []
            for s in leaves(shape):
                flat.append(running)
                running *= s
            stride = _regroup(iter(flat), shape)
        if not _same_structure(shape, stride):
            raise LayoutError(f"shape {fmt(shape)} and stride {fmt(stride)} are not congruent")
        self.shape = shape
        self.stride = stride

    # -- queries --------------------------------------------------------------
    def size(self) -> int:
        return product(self.shape)

    def rank(self) -> int:
        return len(self.shape) if _is_tup(self.shape) else 1

    def mode(self, i: int) -> "Layout":
        if not _is_tup(self.shape):
            if i != 0:
                raise IndexError(i)
            return self
        return Layout(self.shape[i], self.stride[i])

    def cosize(self) -> int:
        n = self.size()
        return self(n - 1) + 1 if n > 0 else 0

    def flat(self):
        return list(zip(leaves(self.shape), leaves(self.stride)))

    # -- the function -----------------------------------------------------------
    def __call__(self, coord) -> int:
        return _index(coord, self.shape, self.stride)

    def __eq__(self, other) -> bool:
        return isinstance(other, Layout) and self.shape == other.shape and self.stride == other.stride

    def __repr__(self) -> str:
        return f"{fmt(self.shape)}:{fmt(self.stride)}"


def _index(coord, shape, stride) -> int:
    if _is_tup(coord):
        if not _is_tup(shape) or len(coord) != len(shape):
            raise LayoutError("coordinate does not match the shape's modes")
        return sum(_index(c, s, d) for c, s, d in zip(coord, shape, stride))
    if not _is_tup(shape):
        return coord * stride
    # integer against a tuple: peel the modes off, fastest first; the last
    # mode takes whatever is left
    total, rest = 0, coord
    for s, d in zip(shape[:-1], stride[:-1]):
        extent = product(s)
        total += _index(rest % extent, s, d)
        rest //= extent
    return total + _index(rest, shape[-1], stride[-1])


def parse(text: str) -> Layout:
    """Parses the printed form "shape:stride", e.g. "(4,(2,4)):(2,(1,8))"."""
    text = text.replace(" ", "").replace("_", "")
    depth = 0
    for i, ch in enumerate(text):
        depth += ch == "("
        depth -= ch == ")"
        if ch == ":" and depth == 0:
            return Layout(_parse_tuple(text[:i]), _parse_tuple(text[i + 1:]))
    raise LayoutError(f"no top-level ':' in {text!r}")


def _parse_tuple(s: str):
    pos = 0

    def node():
        nonlocal pos
        if s[pos] == "(":
            pos += 1
            items = [node()]
            while s[pos] == ",":
                pos += 1
                items.append(node())
            if s[pos] != ")":
                raise LayoutError(f"expected ')' at {pos} in {s!r}")
            pos += 1
            return tuple(items)
        start = pos
        while pos < len(s) and (s[pos].isdigit() or s[pos] == "-"):
            pos += 1
        if start == pos:
            raise LayoutError(f"expected an integer at {pos} in {s!r}")
        return int(s[start:pos])

    value = node()
    if pos != len(s):
        raise LayoutError(f"trailing text in {s!r}")
    return value


def concat(*layouts: Layout) -> Layout:
    """Places layouts side by side as the top-level modes of one layout."""
    return Layout(tuple(l.shape for l in layouts), tuple(l.stride for l in layouts))


def _from_modes(modes) -> Layout:
    if not modes:
        return Layout(1, 0)
    if len(modes) == 1:
        return Layout(modes[0][0], modes[0][1])
    return Layout(tuple(s for s, _ in modes), tuple(d for _, d in modes))


def coalesce(a: Layout) -> Layout:
    merged = []
    for s, d in a.flat():
        if s == 1:
            continue
        if merged and merged[-1][0] * merged[-1][1] == d:
            merged[-1] = (merged[-1][0] * s, merged[-1][1])
        else:
            merged.append((s, d))
    return _from_modes(merged)


def _compose_single(a: Layout, n: int, d: int) -> Layout:
    """A o (n:d) for one leaf mode of B."""
    if d == 0:
        return Layout(n, 0)
    if n == 1:
        return Layout(1, 0)        # a single coordinate: extent-1 modes print with stride 0
    modes = coalesce(a).flat()
    picked = []
    want, step = n, d
    for extent, stride in modes[:-1]:
        if want == 1:
            break
        if extent % step != 0 and step % extent != 0:
            raise LayoutError(f"stride divisibility fails: extent {extent} vs step {step}")
        supply = extent // step if extent > step else 1
        if supply > 1:
            take = min(supply, want)
            if want % take != 0:
                raise LayoutError(f"shape divisibility fails: want {want}, mode gives {take}")
            picked.append((take, step * stride))
            want //= take
        step = -(-step // extent)      # steps left over once past this mode
    if want != 1:
        picked.append((want, step * modes[-1][1]))   # the last mode is unbounded
    return _from_modes(picked)


def composition(a: Layout, b) -> Layout:
    if isinstance(b, (tuple, list)):           # a tiler: one layout per mode of a
        parts = [composition(a.mode(i), bi) for i, bi in enumerate(b)]
        parts += [a.mode(i) for i in range(len(b), a.rank())]
        return concat(*parts)
    if _is_tup(b.shape):
        return concat(*[composition(a, b.mode(i)) for i in range(b.rank())])
    return _compose_single(a, b.shape, b.stride)


def complement(a: Layout, cotarget: int = 1) -> Layout:
    modes = sorted((d, s) for s, d in a.flat() if s != 1 and d != 0)
    out, reach = [], 1
    for d, s in modes:
        if d % reach != 0:
            raise LayoutError("modes overlap; complement undefined")
        out.append((d // reach, reach))
        reach = s * d
    out.append((-(-cotarget // reach), reach))
    return coalesce(Layout(tuple(s for s, _ in out), tuple(d for _, d in out)))


def logical_divide(a: Layout, b) -> Layout:
    if isinstance(b, (tuple, list)):
        parts = [logical_divide(a.mode(i), bi) for i, bi in enumerate(b)]
        parts += [a.mode(i) for i in range(len(b), a.rank())]
        return concat(*parts)
    return composition(a, concat(b, complement(b, a.size())))


def _as_tiler(tiler):
    return [t if isinstance(t, Layout) else Layout(t) for t in tiler]


def zipped_divide(a: Layout, tiler) -> Layout:
    tl = _as_tiler(tiler)
    d = logical_divide(a, tl)
    inner = concat(*[d.mode(i).mode(0) for i in range(len(tl))])
    outer = concat(*[d.mode(i).mode(1) for i in range(len(tl))])
    return concat(inner, outer)


def local_tile_index(a: Layout, tiler, tile_coord, in_tile_coord) -> int:
    """Index of element `in_tile_coord` of tile `tile_coord` (local_tile)."""
    z = zipped_divide(a, tiler)
    return z((in_tile_coord, tile_coord))


def local_partition_index(a: Layout, thread_layout: Layout, tid: int, value: int) -> int:
    """Index of value `value` owned by thread `tid` (local_partition): the
    thread's position inside the thread layout fixes the tile mode."""
    z = zipped_divide(a, [Layout(s) for s in leaves(thread_layout.shape)])
    positions = [thread_layout(j) for j in range(thread_layout.size())]
    return z((positions.index(tid), value))

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
* [Coalescing] coalesce flattens, drops extent-1 modes, and joins two
  neighbouring modes whenever the first's shape * stride equals the second's
  stride, until no two join.  It preserves L(i) for every 1-D i < size.
* [Composition: a layout over a layout] R = A o B, R(c) = A(B(c)), with B's
  shape; several modes of B compose separately, side by side.  For one mode
  n:d the points A(0), A(d), ..., A((n-1) d) are evaluated (A coalesced, its
  last mode unbounded) and read back as the layout that has them as its 1-D
  function.  Composition is undefined where the page says so: when the
  selected elements fall inside a mode of A that one stride cannot express,
  or when the count wanted cannot be split into whole counts per mode; both
  are checked as conditions on the prefix products of A's coalesced extents.
* [Complement and division] complement(A, M) is the layout A* for which
  (A, A*) covers every index of [0, M) exactly once: the set A reaches is
  widened by copies shifted by its first gap until it is an interval, then
  repeated up to M.  logical_divide(A, B) = A o (B, complement(B, size A));
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


def _flat_coordinate(coord, shape):
    """The fully expanded coordinate of `coord` against `shape`, as a list of
    one value per leaf (left to right).  An integer facing a tuple shape is
    split colexicographically over that shape's leaves (the leftmost leaf
    varies fastest); the last leaf keeps the quotient unreduced, so a
    coordinate past the end continues along it."""
    if _is_tup(coord):
        if not _is_tup(shape) or len(coord) != len(shape):
            raise LayoutError("coordinate does not match the shape's modes")
        out = []
        for c, s in zip(coord, shape):
            out.extend(_flat_coordinate(c, s))
        return out
    extents = leaves(shape)
    digits = []
    for e in extents[:-1]:
        coord, r = divmod(coord, e)
        digits.append(r)
    return digits + [coord]


def _index(coord, shape, stride) -> int:
    """The layout function: the inner product of the expanded coordinate with
    the stride."""
    return sum(c * d for c, d in zip(_flat_coordinate(coord, shape), leaves(stride)))


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
    """Flattens, drops modes of extent 1, and joins neighbouring modes that
    meet end to end (extent x stride of the first equals the stride of the
    second) until no two do.  L(i) is unchanged for every 1-D i."""
    modes = [(s, d) for s, d in a.flat() if s != 1]
    joined = True
    while joined:
        joined = False
        for k in range(len(modes) - 1):
            (s0, d0), (s1, d1) = modes[k], modes[k + 1]
            if s0 * d0 == d1:
                modes[k:k + 2] = [(s0 * s1, d0)]
                joined = True
                break
    return _from_modes(modes)


def _as_layout(values):
    """The layout whose 1-D function is the integer sequence `values` (index i
    -> values[i], values[0] = 0), in its coalesced form, or LayoutError when
    no layout with that many coordinates has that function.  Each mode in
    turn takes the longest stretch over which the sequence advances by one
    fixed stride per copy of everything found so far; the stretch must split
    the remaining count into whole copies."""
    n = len(values)
    modes, block = [], 1
    while block < n:
        stride = values[block]
        extent = 1
        while block * (extent + 1) <= n and all(
                values[extent * block + i] == values[i] + extent * stride for i in range(block)):
            extent += 1
        if (n // block) % extent:
            raise LayoutError("the composed points do not split into whole modes")
        modes.append((extent, stride))
        block *= extent
    return _from_modes(modes)


def _check_composable(a: Layout, n: int, d: int) -> None:
    """The two conditions under which A o (n:d) is defined, in terms of the
    prefix products P_k of A's coalesced extents (P_0 = 1), for every bounded
    mode k the selected points reach (P_(k-1) < n d):
    - the step d lands on whole modes: P_k divides d, or d divides P_k
      (otherwise an element falls inside a mode that one stride cannot
      express: the page's ∘ 4:4);
    - whole counts per mode: once d divides P_k, the n points either end
      inside mode k (n d <= P_k) or use all of it (P_k divides n d)
      (otherwise the count wanted cannot be split: the page's ∘ 4:2)."""
    if n == 1 or d == 0:
        return
    extents = [s for s, _ in coalesce(a).flat()][:-1]      # the last mode is unbounded
    prev = 1
    for e in extents:
        p = prev * e
        if prev >= n * d:
            break
        if d % p == 0:
            prev = p
            continue
        if p % d != 0:
            raise LayoutError(f"stride divisibility fails: prefix {p} vs step {d}")
        if n * d > p and (n * d) % p != 0:
            raise LayoutError(f"shape divisibility fails: {n} points of step {d} over prefix {p}")
        prev = p


def composition(a: Layout, b) -> Layout:
    """R = A o B with R(i) = A(B(i)): computed point by point and read back as
    a layout, mode by mode of B (a tuple of layouts composes with A's modes
    one by one, leaving the rest).  A is taken in its coalesced form, as the
    page's walk starts from it: the same function on [0, size A), and points
    past the end continue along the coalesced layout's last mode."""
    if isinstance(b, (tuple, list)):           # a tiler: one layout per mode of a
        parts = [composition(a.mode(i), bi) for i, bi in enumerate(b)]
        parts += [a.mode(i) for i in range(len(b), a.rank())]
        return concat(*parts)
    if _is_tup(b.shape):
        return concat(*[composition(a, b.mode(i)) for i in range(b.rank())])
    n, d = b.shape, b.stride
    _check_composable(a, n, d)
    if n == 1:
        return Layout(1, 0)        # a single coordinate: extent-1 modes print with stride 0
    ac = coalesce(a)
    return _as_layout([ac(i * d) for i in range(n)])


def complement(a: Layout, cotarget: int = 1) -> Layout:
    """A* with (A, A*) covering [0, M) exactly once, M >= cotarget: the set
    of indices A reaches (modes of extent 1 or stride 0 add none) is widened
    by copies shifted by its first gap, as many as stay disjoint, until it is
    [0, R); R < cotarget adds a last mode of ceil(cotarget / R) copies at
    stride R.  LayoutError when A repeats an index or a gap cannot be filled
    without overlap."""
    active = [(s, d) for s, d in a.flat() if s != 1 and d != 0]
    reached = {0}
    for s, d in active:
        reached = {x + j * d for x in reached for j in range(s)}
    if len(reached) != product(tuple(s for s, _ in active)):
        raise LayoutError("modes overlap; complement undefined")
    modes = []
    while True:
        gap = next(x for x in range(len(reached) + 1) if x not in reached)
        if gap == len(reached):                 # [0, R) is covered
            break
        copies = 1
        while not any((x + copies * gap) in reached for x in reached):
            copies += 1
        if copies == 1:
            raise LayoutError("modes overlap; complement undefined")
        reached = {x + j * gap for x in reached for j in range(copies)}
        modes.append((copies, gap))
    span = len(reached)
    if span < cotarget:
        modes.append((-(-cotarget // span), span))
    return coalesce(_from_modes(modes))


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

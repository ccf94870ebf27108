// layout.hpp - shape:stride layouts for the GEMM's index math.
//
// Definitions from the page "CuTe's layout algebra" (Advanced CUDA notebook):
//  * "A layout: shape and stride": a layout is a pair of congruent nested
//    integer tuples; coordinate -> inner product with the stride; an integer
//    coordinate splits colexicographically (mode 0 fastest) and the last mode
//    takes whatever is left; size, cosize = L(size-1)+1, rank.
//  * "Coalescing": flatten, drop extent-1 modes, merge neighbours whose
//    shape*stride equals the next stride.  Preserves L(i) for every i.
//  * "Composition: a layout over a layout": (A o B)(c) = A(B(c)) with B's
//    shape; per leaf n:d of B, step over d of A's coalesced elements then
//    collect n, defined only when extents and steps divide each other.
//  * "Complement and division": complement, logical_divide = A o (B, B*),
//    zipped_divide = ((tile modes), (rest modes)).
//
// Two types live here.  `Layout` is a nested tree (host only) used by the
// planner; `FlatLayout` is its flattened, fixed-size form that host and
// device evaluate identically (the tile scheduler and the gather check run
// it on the GPU).
#pragma once

#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define GL_HD __host__ __device__ __forceinline__
#else
#define GL_HD inline
#endif

namespace gl {

enum Err { kOk = 0, kParse = 1, kUndefined = 2, kCapacity = 3 };

// ---------------------------------------------------------------------------
// Flattened layout: leaves only, in order.  Evaluation of a 1-D coordinate
// depends only on the leaves (the nesting changes nothing for it).
// ---------------------------------------------------------------------------
struct FlatLayout {
    static constexpr int kMaxModes = 8;
    int32_t rank;
    int64_t shape[kMaxModes];
    int64_t stride[kMaxModes];

    GL_HD int64_t operator()(int64_t c) const {
        int64_t idx = 0;
        for (int i = 0; i + 1 < rank; ++i) {
            idx += (c % shape[i]) * stride[i];
            c /= shape[i];
        }
        return rank > 0 ? idx + c * stride[rank - 1] : 0;
    }
    GL_HD int64_t size() const {
        int64_t s = 1;
        for (int i = 0; i < rank; ++i) s *= shape[i];
        return s;
    }
};

// ---------------------------------------------------------------------------
// Nested layout, stored as a pre-order node list.  Node 0 is the root; a
// tuple node is followed by its children's subtrees.
// ---------------------------------------------------------------------------
struct Layout {
    static constexpr int kMaxNodes = 64;
    int32_t count = 0;
    int8_t is_leaf[kMaxNodes];
    int16_t children[kMaxNodes];
    int64_t shape[kMaxNodes];
    int64_t stride[kMaxNodes];
};

// Index just past the subtree rooted at node i.
inline int subtree_end(const Layout& l, int i) {
    if (l.is_leaf[i]) return i + 1;
    int j = i + 1;
    for (int c = 0; c < l.children[i]; ++c) j = subtree_end(l, j);
    return j;
}

// Index of child c of tuple node i.
inline int child_node(const Layout& l, int i, int c) {
    int j = i + 1;
    for (int k = 0; k < c; ++k) j = subtree_end(l, j);
    return j;
}

inline bool push_leaf(Layout& l, int64_t s, int64_t d) {
    if (l.count >= Layout::kMaxNodes) return false;
    l.is_leaf[l.count] = 1;
    l.children[l.count] = 0;
    l.shape[l.count] = s;
    l.stride[l.count] = d;
    ++l.count;
    return true;
}

inline bool push_tuple(Layout& l, int nchildren) {
    if (l.count >= Layout::kMaxNodes) return false;
    l.is_leaf[l.count] = 0;
    l.children[l.count] = (int16_t)nchildren;
    l.shape[l.count] = 0;
    l.stride[l.count] = 0;
    ++l.count;
    return true;
}

inline bool push_subtree(Layout& dst, const Layout& src, int i) {
    const int e = subtree_end(src, i);
    for (int j = i; j < e; ++j) {
        if (dst.count >= Layout::kMaxNodes) return false;
        dst.is_leaf[dst.count] = src.is_leaf[j];
        dst.children[dst.count] = src.children[j];
        dst.shape[dst.count] = src.shape[j];
        dst.stride[dst.count] = src.stride[j];
        ++dst.count;
    }
    return true;
}

inline Layout leaf(int64_t s, int64_t d) {
    Layout l;
    push_leaf(l, s, d);
    return l;
}

inline Layout subtree(const Layout& l, int i) {
    Layout out;
    push_subtree(out, l, i);
    return out;
}

// Side-by-side: the parts become the top-level modes of one layout.
inline int concat(const Layout* parts, int k, Layout* out) {
    Layout r;
    if (!push_tuple(r, k)) return kCapacity;
    for (int i = 0; i < k; ++i)
        if (!push_subtree(r, parts[i], 0)) return kCapacity;
    *out = r;
    return kOk;
}

inline int rank(const Layout& l) { return l.is_leaf[0] ? 1 : l.children[0]; }

inline Layout mode(const Layout& l, int i) {
    if (l.is_leaf[0]) return l;
    return subtree(l, child_node(l, 0, i));
}

inline int leaves(const Layout& l, int64_t* s, int64_t* d, int cap) {
    int n = 0;
    for (int i = 0; i < l.count; ++i)
        if (l.is_leaf[i]) {
            if (n >= cap) return -1;
            s[n] = l.shape[i];
            d[n] = l.stride[i];
            ++n;
        }
    return n;
}

inline int64_t size(const Layout& l) {
    int64_t p = 1;
    for (int i = 0; i < l.count; ++i)
        if (l.is_leaf[i]) p *= l.shape[i];
    return p;
}

inline int64_t eval(const Layout& l, int64_t c) {
    int64_t idx = 0, last = -1;
    for (int i = 0; i < l.count; ++i)
        if (l.is_leaf[i]) last = i;
    for (int i = 0; i < l.count; ++i) {
        if (!l.is_leaf[i]) continue;
        if (i == last) return idx + c * l.stride[i];
        idx += (c % l.shape[i]) * l.stride[i];
        c /= l.shape[i];
    }
    return idx;
}

// One integer coordinate per top-level mode.
inline int64_t eval_modes(const Layout& l, const int64_t* coord, int n) {
    if (l.is_leaf[0]) return eval(l, coord[0]);
    int64_t idx = 0;
    for (int m = 0; m < n && m < rank(l); ++m) idx += eval(mode(l, m), coord[m]);
    return idx;
}

inline int64_t cosize(const Layout& l) {
    const int64_t n = size(l);
    return n > 0 ? eval(l, n - 1) + 1 : 0;
}

inline bool flatten(const Layout& l, FlatLayout* f) {
    const int n = leaves(l, f->shape, f->stride, FlatLayout::kMaxModes);
    if (n < 0) return false;
    f->rank = n;
    return true;
}

// Builds a rank-1 leaf or a flat tuple from (shape, stride) pairs; an empty
// list is the single-point layout 1:0.
inline int from_pairs(const int64_t* s, const int64_t* d, int n, Layout* out) {
    Layout r;
    if (n == 0) {
        push_leaf(r, 1, 0);
    } else if (n == 1) {
        push_leaf(r, s[0], d[0]);
    } else {
        if (!push_tuple(r, n)) return kCapacity;
        for (int i = 0; i < n; ++i)
            if (!push_leaf(r, s[i], d[i])) return kCapacity;
    }
    *out = r;
    return kOk;
}

inline Layout coalesce(const Layout& l) {
    int64_t s[Layout::kMaxNodes], d[Layout::kMaxNodes], ms[Layout::kMaxNodes], md[Layout::kMaxNodes];
    const int n = leaves(l, s, d, Layout::kMaxNodes);
    int k = 0;
    for (int i = 0; i < n; ++i) {
        if (s[i] == 1) continue;
        if (k > 0 && ms[k - 1] * md[k - 1] == d[i]) {
            ms[k - 1] *= s[i];
        } else {
            ms[k] = s[i];
            md[k] = d[i];
            ++k;
        }
    }
    Layout out;
    from_pairs(ms, md, k, &out);
    return out;
}

// A o (n:d) for a single leaf of B.
inline int compose_leaf(const Layout& a, int64_t n, int64_t d, Layout* out) {
    if (d == 0) { *out = leaf(n, 0); return kOk; }
    if (n == 1) { *out = leaf(1, 0); return kOk; }
    int64_t as[Layout::kMaxNodes], ad[Layout::kMaxNodes];
    const Layout ca = coalesce(a);
    const int na = leaves(ca, as, ad, Layout::kMaxNodes);
    int64_t ps[Layout::kMaxNodes], pd[Layout::kMaxNodes];
    int np = 0;
    int64_t want = n, step = d;
    for (int j = 0; j + 1 < na && want > 1; ++j) {
        const int64_t extent = as[j];
        if (extent % step != 0 && step % extent != 0) return kUndefined;
        if (extent > step) {
            const int64_t avail = extent / step;
            const int64_t take = avail < want ? avail : want;
            if (want % take != 0) return kUndefined;
            ps[np] = take;
            pd[np] = step * ad[j];
            ++np;
            want /= take;
        }
        step = (step + extent - 1) / extent;
    }
    if (want != 1) {
        ps[np] = want;
        pd[np] = step * ad[na - 1];
        ++np;
    }
    return from_pairs(ps, pd, np, out);
}

// A o B.  B's nesting is kept: each leaf of B becomes its composition with A.
inline int compose_node(const Layout& a, const Layout& b, int i, Layout* out) {
    if (b.is_leaf[i]) return compose_leaf(a, b.shape[i], b.stride[i], out);
    Layout parts[8];
    const int k = b.children[i];
    if (k > 8) return kCapacity;
    for (int c = 0; c < k; ++c) {
        const int err = compose_node(a, b, child_node(b, i, c), &parts[c]);
        if (err) return err;
    }
    return concat(parts, k, out);
}

inline int composition(const Layout& a, const Layout& b, Layout* out) { return compose_node(a, b, 0, out); }

// Mode-wise composition with a tiler (one layout per leading mode of a).
inline int composition_tiler(const Layout& a, const Layout* tiler, int k, Layout* out) {
    Layout parts[8];
    const int ra = rank(a);
    if (ra > 8 || k > ra) return kCapacity;
    for (int i = 0; i < ra; ++i) {
        if (i < k) {
            const int err = composition(mode(a, i), tiler[i], &parts[i]);
            if (err) return err;
        } else {
            parts[i] = mode(a, i);
        }
    }
    return concat(parts, ra, out);
}

inline int complement(const Layout& a, int64_t cotarget, Layout* out) {
    int64_t s[Layout::kMaxNodes], d[Layout::kMaxNodes];
    const int n = leaves(a, s, d, Layout::kMaxNodes);
    // keep the modes that move, ordered by stride (then extent)
    int64_t ks[Layout::kMaxNodes], kd[Layout::kMaxNodes];
    int k = 0;
    for (int i = 0; i < n; ++i)
        if (s[i] != 1 && d[i] != 0) { ks[k] = s[i]; kd[k] = d[i]; ++k; }
    for (int i = 1; i < k; ++i)
        for (int j = i; j > 0 && (kd[j] < kd[j - 1] || (kd[j] == kd[j - 1] && ks[j] < ks[j - 1])); --j) {
            int64_t t = kd[j]; kd[j] = kd[j - 1]; kd[j - 1] = t;
            t = ks[j]; ks[j] = ks[j - 1]; ks[j - 1] = t;
        }
    int64_t rs[Layout::kMaxNodes], rd[Layout::kMaxNodes];
    int r = 0;
    int64_t reach = 1;
    for (int i = 0; i < k; ++i) {
        if (kd[i] % reach != 0) return kUndefined;
        rs[r] = kd[i] / reach;
        rd[r] = reach;
        ++r;
        reach = ks[i] * kd[i];
    }
    rs[r] = (cotarget + reach - 1) / reach;
    rd[r] = reach;
    ++r;
    Layout raw;
    if (r == 1) {
        raw = leaf(rs[0], rd[0]);
    } else {
        const int err = from_pairs(rs, rd, r, &raw);
        if (err) return err;
    }
    *out = coalesce(raw);
    return kOk;
}

inline int logical_divide(const Layout& a, const Layout& b, Layout* out) {
    Layout comp;
    int err = complement(b, size(a), &comp);
    if (err) return err;
    Layout pair[2] = {b, comp};
    Layout both;
    err = concat(pair, 2, &both);
    if (err) return err;
    return composition(a, both, out);
}

// zipped_divide(a, tiler): ((tile_0, ..., tile_k-1), (rest_0, ..., rest_k-1)).
inline int zipped_divide(const Layout& a, const Layout* tiler, int k, Layout* out) {
    if (k > 8 || k > rank(a)) return kCapacity;
    Layout tiles[8], rests[8];
    for (int i = 0; i < k; ++i) {
        Layout d;
        const int err = logical_divide(mode(a, i), tiler[i], &d);
        if (err) return err;
        tiles[i] = mode(d, 0);
        rests[i] = mode(d, 1);
    }
    Layout halves[2];
    int err = concat(tiles, k, &halves[0]);
    if (err) return err;
    err = concat(rests, k, &halves[1]);
    if (err) return err;
    return concat(halves, 2, out);
}

// ----------------------------------------------------------- text form ----
struct Parser {
    const char* p;
    bool ok = true;

    void skip() { while (*p == ' ' || *p == '_') ++p; }

    // Reads a tuple tree of integers into `vals` (pre-order leaf values) and
    // the structure into is_leaf/children arrays.
    bool node(Layout& l, bool shape_pass, int& leaf_cursor, int& node_cursor) {
        skip();
        if (*p == '(') {
            ++p;
            int self = node_cursor;
            if (shape_pass) {
                if (!push_tuple(l, 0)) return false;
            } else if (self >= l.count || l.is_leaf[self]) {
                return false;
            }
            ++node_cursor;
            int nchild = 0;
            while (true) {
                if (!node(l, shape_pass, leaf_cursor, node_cursor)) return false;
                ++nchild;
                skip();
                if (*p == ',') { ++p; continue; }
                if (*p == ')') { ++p; break; }
                return false;
            }
            if (shape_pass) l.children[self] = (int16_t)nchild;
            else if (l.children[self] != nchild) return false;
            return true;
        }
        bool neg = false;
        if (*p == '-') { neg = true; ++p; }
        if (*p < '0' || *p > '9') return false;
        int64_t v = 0;
        while (*p >= '0' && *p <= '9') { v = v * 10 + (*p - '0'); ++p; }
        if (neg) v = -v;
        if (shape_pass) {
            if (v < 1) return false;
            if (!push_leaf(l, v, 0)) return false;
        } else {
            if (node_cursor >= l.count || !l.is_leaf[node_cursor]) return false;
            l.stride[node_cursor] = v;
        }
        ++node_cursor;
        ++leaf_cursor;
        return true;
    }
};

inline int parse(const char* text, Layout* out) {
    // split at the top-level ':'
    int depth = 0;
    const char* colon = nullptr;
    for (const char* q = text; *q; ++q) {
        if (*q == '(') ++depth;
        else if (*q == ')') --depth;
        else if (*q == ':' && depth == 0) { colon = q; break; }
    }
    if (!colon) return kParse;
    char shape_txt[512];
    const size_t len = (size_t)(colon - text);
    if (len >= sizeof(shape_txt)) return kParse;
    memcpy(shape_txt, text, len);
    shape_txt[len] = 0;
    Layout l;
    Parser ps{shape_txt};
    int lc = 0, nc = 0;
    if (!ps.node(l, true, lc, nc)) return kParse;
    ps.skip();
    if (*ps.p) return kParse;
    Parser pd{colon + 1};
    lc = 0;
    nc = 0;
    if (!pd.node(l, false, lc, nc)) return kParse;
    pd.skip();
    if (*pd.p || nc != l.count) return kParse;
    *out = l;
    return kOk;
}

// Appends the printed form of the subtree at node i (shape if which==0,
// stride otherwise).  Returns false when `cap` would be exceeded.
inline bool print_node(const Layout& l, int i, int which, char* out, size_t cap, size_t& pos) {
    auto put = [&](char c) { if (pos + 1 >= cap) return false; out[pos++] = c; out[pos] = 0; return true; };
    if (l.is_leaf[i]) {
        char buf[24];
        int64_t v = which ? l.stride[i] : l.shape[i];
        int n = 0;
        bool neg = v < 0;
        uint64_t u = neg ? (uint64_t)(-v) : (uint64_t)v;
        do { buf[n++] = (char)('0' + u % 10); u /= 10; } while (u);
        if (neg && !put('-')) return false;
        while (n) if (!put(buf[--n])) return false;
        return true;
    }
    if (!put('(')) return false;
    int j = i + 1;
    for (int c = 0; c < l.children[i]; ++c) {
        if (c && !put(',')) return false;
        if (!print_node(l, j, which, out, cap, pos)) return false;
        j = subtree_end(l, j);
    }
    return put(')');
}

inline int print(const Layout& l, char* out, size_t cap) {
    size_t pos = 0;
    if (cap == 0) return kCapacity;
    out[0] = 0;
    if (!print_node(l, 0, 0, out, cap, pos)) return kCapacity;
    if (pos + 1 >= cap) return kCapacity;
    out[pos++] = ':';
    out[pos] = 0;
    if (!print_node(l, 0, 1, out, cap, pos)) return kCapacity;
    return kOk;
}

}  // namespace gl

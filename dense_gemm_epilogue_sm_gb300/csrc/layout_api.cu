// layout_api.cu - C ABI over layout.hpp (see include/gemm_layout.h): host
// queries and algebra for tests and tools, and a device gather that
// evaluates a layout with the same FlatLayout code the GEMM's tile
// scheduler runs (the host/device agreement check of "cute_layouts.cu",
// gate 4: out[i] = in[L(i)]).
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "../../include/gemm_layout.h"
#include "layout.hpp"

namespace {

__global__ void gather_kernel(const float* __restrict__ in, float* __restrict__ out, gl::FlatLayout lay,
                              int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) out[i] = in[lay(i)];
}

int parse_tiler(const char* text, gl::Layout* tiles, int* k) {
    *k = 0;
    const char* p = text;
    while (*p) {
        if (*k >= 8) return gl::kCapacity;
        int64_t v = 0;
        if (*p < '0' || *p > '9') return gl::kParse;
        while (*p >= '0' && *p <= '9') v = v * 10 + (*p++ - '0');
        if (v < 1) return gl::kParse;
        tiles[(*k)++] = gl::leaf(v, 1);
        if (*p == ',') ++p;
        else if (*p) return gl::kParse;
    }
    return *k ? gl::kOk : gl::kParse;
}

}  // namespace

extern "C" {

int gemm_layout_query(const char* layout, const char* what, int64_t* out) {
    if (!layout || !what || !out) return gl::kParse;
    gl::Layout l;
    const int e = gl::parse(layout, &l);
    if (e) return e;
    if (!strcmp(what, "size")) *out = gl::size(l);
    else if (!strcmp(what, "cosize")) *out = gl::cosize(l);
    else if (!strcmp(what, "rank")) *out = gl::rank(l);
    else return gl::kParse;
    return gl::kOk;
}

int gemm_layout_eval(const char* layout, const int64_t* coord, int32_t ncoord, int64_t* out) {
    if (!layout || !coord || !out || ncoord < 1) return gl::kParse;
    gl::Layout l;
    const int e = gl::parse(layout, &l);
    if (e) return e;
    if (ncoord == 1) {
        *out = gl::eval(l, coord[0]);
        return gl::kOk;
    }
    if (ncoord != gl::rank(l)) return gl::kParse;
    *out = gl::eval_modes(l, coord, ncoord);
    return gl::kOk;
}

int gemm_layout_op(const char* op, const char* a, const char* b, int64_t m, char* out, size_t out_len) {
    if (!op || !a || !out) return gl::kParse;
    gl::Layout la, lb, r;
    int e = gl::parse(a, &la);
    if (e) return e;
    if (!strcmp(op, "coalesce")) {
        r = gl::coalesce(la);
    } else if (!strcmp(op, "composition") || !strcmp(op, "logical_divide")) {
        if (!b) return gl::kParse;
        e = gl::parse(b, &lb);
        if (e) return e;
        e = op[0] == 'c' ? gl::composition(la, lb, &r) : gl::logical_divide(la, lb, &r);
    } else if (!strcmp(op, "complement")) {
        e = gl::complement(la, m, &r);
    } else if (!strcmp(op, "zipped_divide")) {
        gl::Layout tiles[8];
        int k = 0;
        if (!b) return gl::kParse;
        e = parse_tiler(b, tiles, &k);
        if (!e) e = gl::zipped_divide(la, tiles, k, &r);
    } else if (!strcmp(op, "mode")) {
        if (m < 0 || m >= gl::rank(la)) return gl::kParse;
        r = gl::mode(la, (int)m);
    } else {
        return gl::kParse;
    }
    if (e) return e;
    return gl::print(r, out, out_len);
}

int gemm_layout_gather_f32(const char* layout, const float* in, float* out, int64_t n, void* stream) {
    if (!layout || n < 0 || (n > 0 && (!in || !out))) return gl::kParse;
    gl::Layout l;
    const int e = gl::parse(layout, &l);
    if (e) return e;
    gl::FlatLayout f;
    if (!gl::flatten(l, &f)) return gl::kCapacity;
    if (n == 0) return gl::kOk;
    const int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    gather_kernel<<<(unsigned)blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(in, out, f, n);
    return cudaGetLastError() == cudaSuccess ? gl::kOk : 4;
}

}  // extern "C"

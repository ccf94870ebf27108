/*
 * gemm_layout.h - C ABI of the shape:stride layout module used by the GEMM's
 * host planner and tile scheduler.
 *
 * A layout is a pair of congruent, possibly nested, integer tuples written
 * "shape:stride", e.g. "(4,(2,4)):(2,(1,8))".  It maps a coordinate to the
 * inner product of coordinate and stride; an integer coordinate is split
 * colexicographically (mode 0 fastest) and the last mode is unbounded.  The
 * operations follow the page "CuTe's layout algebra" (Advanced CUDA notebook):
 * "A layout: shape and stride" (evaluation, size, cosize, rank), "Coalescing",
 * "Composition: a layout over a layout" (undefined unless the divisibility
 * conditions hold), "Complement and division" (complement, logical_divide,
 * zipped_divide).
 *
 * Strings are NUL-terminated.  Return codes:
 *   0 ok, 1 parse error or bad argument, 2 operation undefined
 *   (divisibility), 3 result exceeds the module's capacity or `out_len`,
 *   4 CUDA error (gather only).
 */
#ifndef GEMM_LAYOUT_H
#define GEMM_LAYOUT_H

#include <stddef.h>
#include <stdint.h>

#ifndef GEMM_API
#define GEMM_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* what = "size" | "cosize" | "rank".  Host only. */
GEMM_API int gemm_layout_query(const char* layout, const char* what, int64_t* out);

/* Evaluates the layout.  ncoord == 1: one integer (1-D) coordinate.
 * ncoord == rank: one integer per top-level mode.  Host only. */
GEMM_API int gemm_layout_eval(const char* layout, const int64_t* coord, int32_t ncoord, int64_t* out);

/* op = "coalesce" (a), "composition" (a o b), "complement" (a, m),
 * "logical_divide" (a, b), "zipped_divide" (a, b = comma-separated tile
 * extents, e.g. "16,16"), "mode" (top-level mode m of a).
 * Writes the printed result to out (capacity out_len).  Host only. */
GEMM_API int gemm_layout_op(const char* op, const char* a, const char* b, int64_t m, char* out, size_t out_len);

/* Device gather through a layout, out[i] = in[L(i)] for i < n, evaluated by
 * the same layout code the kernels use.  `in` and `out` are device pointers;
 * the caller guarantees L(i) < the length of `in`.  Asynchronous on
 * `stream` (a cudaStream_t).  Needs a GPU. */
GEMM_API int gemm_layout_gather_f32(const char* layout, const float* in, float* out, int64_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_LAYOUT_H */

// gemm_variants.h - the kernel variants the library builds and their
// host-side operations.  Declarations only: the dispatcher (gemm_sm103.cu)
// includes this without the kernel, and gemm_ob1/2/4.cu instantiate the
// definitions from gemm_kernel.cuh, so the variants compile in parallel.
#pragma once

#include "gemm_internal.h"

namespace gemm_sm103 {

// CG: CTAs per MMA (1, or a pair), BN: tile columns, OB: output element
// bytes (1 = e4m3 with MX factors), BS: block-scaled operands (0 none,
// 1 MXFP8, 2 NVFP4).
template <int CG, int BN, int OB, int BS>
struct Variant {
    static size_t smem();
    static cudaError_t prepare();
    static cudaError_t launch(const LaunchArgs& a);
    static int max_clusters();
};

#define GEMM_FOR_EACH_VARIANT(X, OB)                                                                  \
    X(2, 256, OB, 0) X(1, 256, OB, 0) X(1, 128, OB, 0) X(2, 256, OB, 1) X(2, 128, OB, 1) X(1, 128, OB, 1)  \
        X(2, 256, OB, 2) X(2, 128, OB, 2) X(1, 128, OB, 2)
#define GEMM_EXTERN_VARIANT(CG, BN, OB, BS) extern template struct Variant<CG, BN, OB, BS>;
#define GEMM_INSTANTIATE_VARIANT(CG, BN, OB, BS) template struct Variant<CG, BN, OB, BS>;

GEMM_FOR_EACH_VARIANT(GEMM_EXTERN_VARIANT, 1)
GEMM_FOR_EACH_VARIANT(GEMM_EXTERN_VARIANT, 2)
GEMM_FOR_EACH_VARIANT(GEMM_EXTERN_VARIANT, 4)

}  // namespace gemm_sm103

// gemm_sm103.cu - picks the kernel variant of a plan: shared-memory size,
// one-time attributes, occupancy and launch.  The kernel itself lives in
// gemm_kernel.cuh; its variants are compiled in gemm_ob1.cu, gemm_ob2.cu and
// gemm_ob4.cu (one output element size each).
#include "gemm_variants.h"

namespace gemm_sm103 {

int stages_for(int cta_group, int tile_n, int block_scaled) {
    if (block_scaled == 2) return (cta_group == 2 && tile_n == 128) ? 6 : 5;
    return block_scaled ? (cta_group == 2 ? 6 : 5) : ((cta_group == 1 && tile_n == 256) ? 4 : 6);
}

// Kernel variants by (CTA group, tile N, output bytes, block scaling).
#define GEMM_OB3(EXPR1, EXPR2, EXPR4) (out_bytes == 1 ? (EXPR1) : out_bytes == 2 ? (EXPR2) : (EXPR4))

#define GEMM_VARIANT3(CG, BN, BS, F, ...)                                                                    \
    GEMM_OB3((Variant<CG, BN, 1, BS>::F(__VA_ARGS__)), (Variant<CG, BN, 2, BS>::F(__VA_ARGS__)),                 \
             (Variant<CG, BN, 4, BS>::F(__VA_ARGS__)))

#define GEMM_DISPATCH(F, ...)                                                                          \
    do {                                                                                               \
        if (block_scaled == 2 && cta_group == 2 && tile_n == 256) return GEMM_VARIANT3(2, 256, 2, F, __VA_ARGS__); \
        if (block_scaled == 2 && cta_group == 2) return GEMM_VARIANT3(2, 128, 2, F, __VA_ARGS__);      \
        if (block_scaled == 2) return GEMM_VARIANT3(1, 128, 2, F, __VA_ARGS__);                        \
        if (block_scaled && cta_group == 2 && tile_n == 256) return GEMM_VARIANT3(2, 256, 1, F, __VA_ARGS__); \
        if (block_scaled && cta_group == 2) return GEMM_VARIANT3(2, 128, 1, F, __VA_ARGS__);           \
        if (block_scaled) return GEMM_VARIANT3(1, 128, 1, F, __VA_ARGS__);                             \
        if (cta_group == 2) return GEMM_VARIANT3(2, 256, 0, F, __VA_ARGS__);                           \
        if (tile_n == 256) return GEMM_VARIANT3(1, 256, 0, F, __VA_ARGS__);                            \
        return GEMM_VARIANT3(1, 128, 0, F, __VA_ARGS__);                                               \
    } while (0)

size_t smem_bytes_for(int cta_group, int tile_n, int out_bytes, int block_scaled) {
    GEMM_DISPATCH(smem);
}

cudaError_t prepare_kernel(int cta_group, int tile_n, int out_bytes, int block_scaled) {
    GEMM_DISPATCH(prepare);
}

int max_active_clusters(int cta_group, int tile_n, int out_bytes, int block_scaled) {
    GEMM_DISPATCH(max_clusters);
}

cudaError_t launch(const LaunchArgs& a) {
    const int cta_group = a.cta_group, tile_n = a.tile_n, out_bytes = a.out_bytes, block_scaled = a.block_scaled;
    GEMM_DISPATCH(launch, a);
}

}  // namespace gemm_sm103

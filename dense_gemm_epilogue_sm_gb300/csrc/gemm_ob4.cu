// gemm_ob4.cu - the kernel variants with 4-byte output elements
// (instantiated here so the variants compile in parallel).
#include "gemm_kernel.cuh"

namespace gemm_sm103 {

GEMM_FOR_EACH_VARIANT(GEMM_INSTANTIATE_VARIANT, 4)

}  // namespace gemm_sm103

// gemm_ob2.cu - the kernel variants with 2-byte output elements
// (instantiated here so the variants compile in parallel).
#include "gemm_kernel.cuh"

namespace gemm_sm103 {

GEMM_FOR_EACH_VARIANT(GEMM_INSTANTIATE_VARIANT, 2)

}  // namespace gemm_sm103

// gemm_ob1.cu - the kernel variants with 1-byte output elements
// (instantiated here so the variants compile in parallel).
#include "gemm_kernel.cuh"

namespace gemm_sm103 {

GEMM_FOR_EACH_VARIANT(GEMM_INSTANTIATE_VARIANT, 1)

}  // namespace gemm_sm103

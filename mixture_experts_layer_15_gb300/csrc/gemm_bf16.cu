// Instantiations of the grouped GEMM kernel for bf16 expert weights.
#include "gemm_kernel.cuh"

namespace moe {
namespace gemm {

cudaError_t launch_gemm_bf16(int fused, int mode, int bt, int na, int out_dtype, const Maps& m,
                                  const KernelArgs& ka, int grid, cudaStream_t s) {
    return launch_gemm<false>(fused, mode, bt, na, out_dtype, m, ka, grid, s);
}

}  // namespace gemm
}  // namespace moe

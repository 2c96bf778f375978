// Instantiations of the grouped GEMM kernel with the finalize folded into the
// GEMM2 epilogue, for MXFP4 expert weights (a translation unit of its own so
// that the kernel variants compile in parallel).
#include "gemm_kernel.cuh"

namespace moe {
namespace gemm {

cudaError_t launch_gemm_final_mxfp4(int fused, int bt, int na, const Maps& m, const KernelArgs& ka, int grid,
                                  cudaStream_t s) {
    return launch_gemm_final<true>(fused, bt, na, m, ka, grid, s);
}

}  // namespace gemm
}  // namespace moe

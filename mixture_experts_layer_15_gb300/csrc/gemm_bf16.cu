// Instantiations of the grouped GEMM kernel for bf16 expert weights.
#include "gemm_kernel.cuh"

namespace moe {
namespace gemm {

cudaError_t launch_gemm_bf16(int mode, int bt, int na, int out_dtype, const CUtensorMap& tmA,
                                  const CUtensorMap& tmS, const CUtensorMap& tmB, const GemmArgs& a, int grid,
                                  cudaStream_t s) {
    return launch_gemm<false>(mode, bt, na, out_dtype, tmA, tmS, tmB, a, grid, s);
}

}  // namespace gemm
}  // namespace moe

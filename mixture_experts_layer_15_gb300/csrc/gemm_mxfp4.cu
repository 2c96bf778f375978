// Instantiations of the grouped GEMM kernel for MXFP4 (e2m1 + E8M0 per 32) expert weights.
#include "gemm_kernel.cuh"

namespace moe {
namespace gemm {

cudaError_t launch_gemm_mxfp4(int mode, int bt, int na, int out_dtype, const CUtensorMap& tmA,
                                   const CUtensorMap& tmS, const CUtensorMap& tmB, const GemmArgs& a, int grid,
                                   cudaStream_t s) {
    return launch_gemm<true>(mode, bt, na, out_dtype, tmA, tmS, tmB, a, grid, s);
}

}  // namespace gemm
}  // namespace moe

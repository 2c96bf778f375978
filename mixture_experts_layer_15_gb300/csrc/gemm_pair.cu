// Instantiations of the CTA-pair grouped GEMM kernel (bf16 weights).
#include "gemm_pair_kernel.cuh"

namespace moe {
namespace gemm {

cudaError_t launch_gemm_pair_bf16(int mode, int bt, int out_dtype, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const GemmArgs& a, int pairs, cudaStream_t s) {
    return launch_gemm_pair(mode, bt, out_dtype, tmA, tmB, a, pairs, s);
}

}  // namespace gemm
}  // namespace moe

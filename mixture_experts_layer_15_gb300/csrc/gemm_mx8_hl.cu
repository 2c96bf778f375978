// Instantiations of the block-scaled grouped GEMM with bf16 activations split
// into two E4M3 terms (MOE_WEIGHTS_MXFP4_A16), a translation unit of its own
// so that it compiles in parallel with the other kernel variants.
#include "gemm_mx8_kernel.cuh"

namespace moe {
namespace gemm {

cudaError_t launch_gemm_mx8_hl(int mode, int bt, int out_dtype, const CUtensorMap& tA, const CUtensorMap& tB,
                               const Mx8Args& m, int grid, cudaStream_t s) {
    if (mode == MODE_SWIGLU) return launch_mx8_bt<MODE_SWIGLU, uint8_t, true>(bt, tA, tB, m, grid, s);
    if (mode == MODE_FINAL) return launch_mx8_bt<MODE_FINAL, float, true>(bt, tA, tB, m, grid, s);
    if (out_dtype == MOE_DTYPE_F32) return launch_mx8_bt<MODE_PLAIN, float, true>(bt, tA, tB, m, grid, s);
    return launch_mx8_bt<MODE_PLAIN, __nv_bfloat16, true>(bt, tA, tB, m, grid, s);
}

}  // namespace gemm
}  // namespace moe

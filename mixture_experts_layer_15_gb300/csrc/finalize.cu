// Finalize: apply the routing weights and reduce over top_k
// (vllm/model_executor/layers/fused_moe/modular_kernel.py,
// FusedMoEPrepareAndFinalize.finalize), then the routed scale and the
// shared-expert add (moe_output.py, MoEOutput: the shared output is folded in
// by whoever finalizes, after the routed scale):
//
//   out[t] = rsf * sum_{j: map[t,j] != -1} w[t,j] * gemm2_permuted[map[t,j]] + shared[t]
//
// gemm2_permuted is read by row through the permute map (moe_output.py,
// UnfinalizedMoEOutput: the consumer indexes it by row). The kernel is
// HBM-bound: it reads R rows of K values, writes M rows. Each thread owns 8
// consecutive columns of one token (16- or 32-byte vector accesses); a block
// covers 1024 columns of one token, the grid covers (M, K/1024).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kCols = 8 * kThreads;

template <typename GT, typename ST, typename OT>
__global__ void __launch_bounds__(kThreads)
finalize_kernel(const GT* __restrict__ g2, int num_rows, const void* __restrict__ w, int wdtype,
                const int32_t* __restrict__ map, int top_k, int K, const ST* __restrict__ shared,
                float rsf, OT* __restrict__ out, int* err) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int c = blockIdx.y * kCols + threadIdx.x * 8;
    if (c >= K) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    const size_t rbase = static_cast<size_t>(t) * top_k;
    for (int j = 0; j < top_k; ++j) {
        const int p = __ldg(map + rbase + j);
        if (p < 0) continue;                              // route to a non-local expert
        if (p >= num_rows) { set_error(err, MOE_ERR_DEVICE_INDEX); continue; }
        const float wt = load_as_f32(w, rbase + j, wdtype);
        float v[8];
        Vec8<GT>::load(g2 + static_cast<size_t>(p) * K + c, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wt, v[i], acc[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= rsf;
    if (shared != nullptr) {
        float sv[8];
        Vec8<ST>::load(shared + static_cast<size_t>(t) * K + c, sv);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += sv[i];
    }
    Vec8<OT>::store(out + static_cast<size_t>(t) * K + c, acc);
}

template <typename GT, typename ST, typename OT>
cudaError_t launch_typed(const void* g2, int num_rows, const void* w, int wdtype, const int32_t* map,
                         int M, int top_k, int K, const void* shared, float rsf, void* out,
                         int* err, cudaStream_t s) {
    const dim3 grid(M, ceil_div(K, kCols));
    return launch_pdl(finalize_kernel<GT, ST, OT>, grid, dim3(kThreads), 0, s, static_cast<const GT*>(g2),
                      num_rows, w, wdtype, map, top_k, K, static_cast<const ST*>(shared), rsf,
                      static_cast<OT*>(out), err);
}

template <typename GT, typename ST>
cudaError_t launch_out(int out_dtype, const void* g2, int num_rows, const void* w, int wdtype,
                       const int32_t* map, int M, int top_k, int K, const void* shared, float rsf,
                       void* out, int* err, cudaStream_t s) {
    if (out_dtype == MOE_DTYPE_F32)
        return launch_typed<GT, ST, float>(g2, num_rows, w, wdtype, map, M, top_k, K, shared, rsf, out, err, s);
    return launch_typed<GT, ST, __nv_bfloat16>(g2, num_rows, w, wdtype, map, M, top_k, K, shared, rsf, out, err, s);
}

template <typename GT>
cudaError_t launch_shared(int shared_dtype, int out_dtype, const void* g2, int num_rows, const void* w,
                          int wdtype, const int32_t* map, int M, int top_k, int K, const void* shared,
                          float rsf, void* out, int* err, cudaStream_t s) {
    if (shared_dtype == MOE_DTYPE_F32)
        return launch_out<GT, float>(out_dtype, g2, num_rows, w, wdtype, map, M, top_k, K, shared, rsf, out, err, s);
    return launch_out<GT, __nv_bfloat16>(out_dtype, g2, num_rows, w, wdtype, map, M, top_k, K, shared, rsf, out, err, s);
}

}  // namespace

cudaError_t launch_finalize(const void* g2, int g2_dtype, int num_rows, const void* w, int wdtype,
                            const int32_t* map, int M, int top_k, int K, const void* shared,
                            int shared_dtype, float rsf, void* out, int out_dtype, int* err,
                            cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    if (g2_dtype == MOE_DTYPE_F32)
        return launch_shared<float>(shared_dtype, out_dtype, g2, num_rows, w, wdtype, map, M, top_k, K, shared, rsf, out, err, s);
    return launch_shared<__nv_bfloat16>(shared_dtype, out_dtype, g2, num_rows, w, wdtype, map, M, top_k, K, shared, rsf, out, err, s);
}

}  // namespace moe

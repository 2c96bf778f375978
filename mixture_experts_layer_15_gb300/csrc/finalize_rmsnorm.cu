// Finalize folded into its consumer, the next layer's residual add + RMSNorm
// (moe_output.py, MoEOutput: an open reduction is left for the consumer,
// typically the next layer's RMSNorm, and with an unfinalized routed output
// the top-k reduction folds into the same kernel):
//
//   r[t] = rsf * sum_{j: map[t,j] != -1} w[t,j] * gemm2_permuted[map[t,j]] + shared[t] + residual[t]
//   residual[t] <- r[t]                                   (the new residual stream)
//   y[t] = r[t] / sqrt(mean_K(r[t]^2) + eps) * gamma
//
// One CTA per token: each thread holds its 8-column chunks of r in registers
// (K <= 16384 with 256 threads: at most 8 chunks), stores the new residual,
// and adds its squares into a block reduction; y follows from the registers.
// The finalize part accumulates like finalize.cu (FMA over the routes in j
// order, x rsf, + shared). HBM-bound: reads k rows of gemm2_permuted, the
// shared output and the residual, writes the residual and y.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRnThreads = 256;
constexpr int kRnChunk = 8 * kRnThreads;   // columns per pass of the block

__device__ __forceinline__ void load8_dt(const void* p, size_t i, int dtype, float (&v)[8]) {
    if (dtype == MOE_DTYPE_F32) Vec8<float>::load(static_cast<const float*>(p) + i, v);
    else Vec8<__nv_bfloat16>::load(static_cast<const __nv_bfloat16*>(p) + i, v);
}
__device__ __forceinline__ void store8_dt(void* p, size_t i, int dtype, const float (&v)[8]) {
    if (dtype == MOE_DTYPE_F32) Vec8<float>::store(static_cast<float*>(p) + i, v);
    else Vec8<__nv_bfloat16>::store(static_cast<__nv_bfloat16*>(p) + i, v);
}

template <typename GT, typename RT, int CH>
__global__ void __launch_bounds__(kRnThreads)
finalize_rmsnorm_kernel(const GT* __restrict__ g2, int num_rows, const void* __restrict__ w, int wdtype,
                        const int32_t* __restrict__ map, int top_k, int K, const void* __restrict__ shared,
                        int sdtype, float rsf, RT* __restrict__ residual, const void* __restrict__ gamma,
                        int gdtype, float eps, void* __restrict__ y, int ydtype, int* err) {
    __shared__ float red[kRnThreads / 32];
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const size_t rbase = static_cast<size_t>(t) * top_k;
    const size_t row = static_cast<size_t>(t) * K;
    float r[CH][8];
    float ss = 0.0f;
#pragma unroll
    for (int ch = 0; ch < CH; ++ch) {
        const int c = ch * kRnChunk + threadIdx.x * 8;
        if (c >= K) continue;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
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
            load8_dt(shared, row + c, sdtype, sv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += sv[i];
        }
        float rv[8];
        Vec8<RT>::load(residual + row + c, rv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            acc[i] += rv[i];
            ss = fmaf(acc[i], acc[i], ss);
            r[ch][i] = acc[i];
        }
        Vec8<RT>::store(residual + row + c, acc);
    }
    // sum of squares over the block
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float total = 0.0f;
#pragma unroll
    for (int i = 0; i < kRnThreads / 32; ++i) total += red[i];
    const float rstd = 1.0f / sqrtf(total / static_cast<float>(K) + eps);
#pragma unroll
    for (int ch = 0; ch < CH; ++ch) {
        const int c = ch * kRnChunk + threadIdx.x * 8;
        if (c >= K) continue;
        float g[8], out[8];
        load8_dt(gamma, c, gdtype, g);
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = r[ch][i] * rstd * g[i];
        store8_dt(y, row + c, ydtype, out);
    }
}

template <typename GT, typename RT, int CH>
cudaError_t launch_rn(const void* g2, int num_rows, const void* w, int wdtype, const int32_t* map, int M, int top_k,
                      int K, const void* shared, int sdtype, float rsf, void* residual, const void* gamma, int gdtype,
                      float eps, void* y, int ydtype, int* err, cudaStream_t s) {
    return launch_pdl(finalize_rmsnorm_kernel<GT, RT, CH>, dim3(M), dim3(kRnThreads), 0, s,
                      static_cast<const GT*>(g2), num_rows, w, wdtype, map, top_k, K, shared, sdtype, rsf,
                      static_cast<RT*>(residual), gamma, gdtype, eps, y, ydtype, err);
}

template <typename GT, typename RT>
cudaError_t launch_rn_ch(int K, const void* g2, int num_rows, const void* w, int wdtype, const int32_t* map, int M,
                         int top_k, const void* shared, int sdtype, float rsf, void* residual, const void* gamma,
                         int gdtype, float eps, void* y, int ydtype, int* err, cudaStream_t s) {
    const int ch = ceil_div(K, kRnChunk);
#define MOE_RN(C) \
    return launch_rn<GT, RT, C>(g2, num_rows, w, wdtype, map, M, top_k, K, shared, sdtype, rsf, residual, gamma, \
                                gdtype, eps, y, ydtype, err, s)
    if (ch <= 1) MOE_RN(1);
    if (ch <= 2) MOE_RN(2);
    if (ch <= 4) MOE_RN(4);
    MOE_RN(8);
#undef MOE_RN
}

}  // namespace

cudaError_t launch_finalize_rmsnorm(const void* g2, int g2_dtype, int num_rows, const void* w, int wdtype,
                                    const int32_t* map, int M, int top_k, int K, const void* shared, int sdtype,
                                    float rsf, void* residual, int rdtype, const void* gamma, int gdtype, float eps,
                                    void* y, int ydtype, int* err, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    if (g2_dtype == MOE_DTYPE_F32) {
        if (rdtype == MOE_DTYPE_F32)
            return launch_rn_ch<float, float>(K, g2, num_rows, w, wdtype, map, M, top_k, shared, sdtype, rsf,
                                              residual, gamma, gdtype, eps, y, ydtype, err, s);
        return launch_rn_ch<float, __nv_bfloat16>(K, g2, num_rows, w, wdtype, map, M, top_k, shared, sdtype, rsf,
                                                  residual, gamma, gdtype, eps, y, ydtype, err, s);
    }
    if (rdtype == MOE_DTYPE_F32)
        return launch_rn_ch<__nv_bfloat16, float>(K, g2, num_rows, w, wdtype, map, M, top_k, shared, sdtype, rsf,
                                                  residual, gamma, gdtype, eps, y, ydtype, err, s);
    return launch_rn_ch<__nv_bfloat16, __nv_bfloat16>(K, g2, num_rows, w, wdtype, map, M, top_k, shared, sdtype,
                                                      rsf, residual, gamma, gdtype, eps, y, ydtype, err, s);
}

}  // namespace moe

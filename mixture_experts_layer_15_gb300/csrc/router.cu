// [Router] step of the MoE layer (vllm/model_executor/layers/fused_moe/
// modular_kernel.py, module header: [Router] -> [Quantize-Dispatch] -> ...).
// The pages pass the router's outputs (topk_ids, topk_weights) but do not
// define its math; the two methods here are softmax -> top-k -> renormalise
// and sigmoid + selection bias -> grouped top-k -> renormalise x scale
// (DeepSeek-V3's published routing rule).
//
// One warp per token. Lane l holds the logits of experts l, l+32, l+64, ...
// in registers (SLOTS = ceil(E/32) per lane). top_k rounds of a warp-wide
// arg-max pick the experts in order (larger key first, equal keys to the
// lower expert id). The kernel is latency-bound: at the largest routing input
// (8192 x 256 f32 = 8 MB) it is a few microseconds at HBM speed.
#include "router_device.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;
using namespace route;

template <int SLOTS>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_softmax_kernel(const float* __restrict__ logits, int M, int E, int top_k, float rsf,
                     int32_t* __restrict__ ids, void* __restrict__ weights, int wdtype) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= M) return;
    int my_id;
    float my_w;
    route_token_softmax<SLOTS>(logits + static_cast<size_t>(t) * E, E, top_k, rsf, lane, my_id, my_w);
    if (lane < top_k) {
        const size_t o = static_cast<size_t>(t) * top_k + lane;
        ids[o] = my_id;
        store_from_f32(weights, o, my_w, wdtype);
    }
}

template <int SLOTS>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_sigmoid_grouped_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                             int M, int E, int top_k, int n_group, int topk_group, float rsf,
                             int32_t* __restrict__ ids, void* __restrict__ weights, int wdtype) {
    extern __shared__ float sh_b[];          // [kWarpsPerBlock][E] biased scores
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kWarpsPerBlock + warp;
    if (t >= M) return;                      // whole warps leave together
    int my_id;
    float my_w;
    route_token_sigmoid<SLOTS>(logits + static_cast<size_t>(t) * E, bias, E, top_k, n_group, topk_group, rsf,
                               lane, sh_b + warp * E, my_id, my_w);
    if (lane < top_k) {
        const size_t o = static_cast<size_t>(t) * top_k + lane;
        ids[o] = my_id;
        store_from_f32(weights, o, my_w, wdtype);
    }
}

__global__ void debug_sigmoid_kernel(const float* __restrict__ x, float* __restrict__ y, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) y[i] = sigmoid_spec(x[i]);
}

template <int SLOTS>
cudaError_t launch_route_slots(const float* logits, int M, int E, int top_k, int method,
                               const float* bias, int n_group, int topk_group, float rsf,
                               int32_t* ids, void* w, int wdtype, cudaStream_t s) {
    const dim3 grid(ceil_div(M, kWarpsPerBlock)), block(kWarpsPerBlock * 32);
    if (method == MOE_ROUTE_SOFTMAX_TOPK)
        return launch_pdl(route_softmax_kernel<SLOTS>, grid, block, 0, s, logits, M, E, top_k, rsf, ids, w,
                          wdtype);
    const size_t smem = sizeof(float) * kWarpsPerBlock * E;   // <= 32 KB for E <= 1024
    return launch_pdl(route_sigmoid_grouped_kernel<SLOTS>, grid, block, smem, s, logits, bias, M, E, top_k,
                      n_group, topk_group, rsf, ids, w, wdtype);
}

}  // namespace

cudaError_t launch_route(const float* logits, int M, int E, int top_k, int method,
                         const float* bias, int n_group, int topk_group, float rsf,
                         int32_t* ids, void* w, int wdtype, int* /*err*/, cudaStream_t s) {
    const int slots = ceil_div(E, 32);
    if (slots <= 1) return launch_route_slots<1>(logits, M, E, top_k, method, bias, n_group, topk_group, rsf, ids, w, wdtype, s);
    if (slots <= 2) return launch_route_slots<2>(logits, M, E, top_k, method, bias, n_group, topk_group, rsf, ids, w, wdtype, s);
    if (slots <= 4) return launch_route_slots<4>(logits, M, E, top_k, method, bias, n_group, topk_group, rsf, ids, w, wdtype, s);
    if (slots <= 8) return launch_route_slots<8>(logits, M, E, top_k, method, bias, n_group, topk_group, rsf, ids, w, wdtype, s);
    if (slots <= 16) return launch_route_slots<16>(logits, M, E, top_k, method, bias, n_group, topk_group, rsf, ids, w, wdtype, s);
    return launch_route_slots<32>(logits, M, E, top_k, method, bias, n_group, topk_group, rsf, ids, w, wdtype, s);
}

cudaError_t launch_debug_sigmoid(const float* x, float* y, int n, cudaStream_t s) {
    return launch_plain(debug_sigmoid_kernel, dim3(ceil_div(n, 256)), dim3(256), 0, s, x, y, n);
}

}  // namespace moe

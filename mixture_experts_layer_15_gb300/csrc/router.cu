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
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

// ---- the float32 sigmoid spec --------------------------------------------------
// exp(t) by Cody & Waite argument reduction and a Taylor polynomial, every
// step one IEEE float32 operation rounded to nearest. The __f*_rn intrinsics
// keep the compiler from contracting a multiply and an add into an FMA, so
// the result is reproducible bit for bit by any IEEE float32 implementation
// of the same steps:
//   t > 88 -> +inf;  t < -80 -> 0
//   n = rint(t * LOG2E);  r = (t - n*LN2_HI) - n*LN2_LO
//   p = Horner over c_i = fl32(1/i!), i = 7..0;  exp = p * 2^n
// LN2_HI is ln 2 cut to 16 significant bits (n*LN2_HI exact for |n| <= 256);
// LN2_LO is the float32 remainder.
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.62e4p-1f;
constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
constexpr float kC0 = 0x1p+0f;          // 1/0!
constexpr float kC1 = 0x1p+0f;          // 1/1!
constexpr float kC2 = 0x1p-1f;          // 1/2!
constexpr float kC3 = 0x1.555556p-3f;   // fl32(1/3!)
constexpr float kC4 = 0x1.555556p-5f;   // fl32(1/4!)
constexpr float kC5 = 0x1.111112p-7f;   // fl32(1/5!)
constexpr float kC6 = 0x1.6c16c2p-10f;  // fl32(1/6!)
constexpr float kC7 = 0x1.a01a02p-13f;  // fl32(1/7!)

__device__ __forceinline__ float exp_spec(float t) {
    if (isnan(t)) return t;
    if (t > 88.0f) return INFINITY;
    if (t < -80.0f) return 0.0f;
    const float n = rintf(__fmul_rn(t, kLog2e));
    float r = __fsub_rn(t, __fmul_rn(n, kLn2Hi));
    r = __fsub_rn(r, __fmul_rn(n, kLn2Lo));
    float p = kC7;
    p = __fadd_rn(__fmul_rn(p, r), kC6);
    p = __fadd_rn(__fmul_rn(p, r), kC5);
    p = __fadd_rn(__fmul_rn(p, r), kC4);
    p = __fadd_rn(__fmul_rn(p, r), kC3);
    p = __fadd_rn(__fmul_rn(p, r), kC2);
    p = __fadd_rn(__fmul_rn(p, r), kC1);
    p = __fadd_rn(__fmul_rn(p, r), kC0);
    const float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);
    return __fmul_rn(p, two_n);
}

__device__ __forceinline__ float sigmoid_spec(float x) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_spec(-x)));
}

// (key, id) order: a before b if a's key is larger, or equal with a lower id.
// id >= E marks "no candidate" and loses to any candidate.
__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib, int E) {
    if (ia >= E) return false;
    if (ib >= E) return true;
    return ka > kb || (ka == kb && ia < ib);
}

// Warp-wide arg-max of (key, id) with payload; every lane returns the winner.
__device__ __forceinline__ void warp_argmax(float& key, int& id, float& pay, int E) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float k2 = __shfl_xor_sync(0xffffffffu, key, off);
        const int i2 = __shfl_xor_sync(0xffffffffu, id, off);
        const float p2 = __shfl_xor_sync(0xffffffffu, pay, off);
        if (better(k2, i2, key, id, E)) { key = k2; id = i2; pay = p2; }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// top_k selection rounds over the lane's SLOTS candidates. `key[s]` is the
// selection key of expert lane + 32*s, `pay[s]` a value carried along,
// `allowed` a bit mask of eligible slots. Lane j < top_k ends with the j-th
// winner in (out_id, out_key, out_pay).
template <int SLOTS>
__device__ __forceinline__ void select_topk(const float (&key)[SLOTS], const float (&pay)[SLOTS],
                                            uint32_t allowed, int E, int top_k, int lane,
                                            int& out_id, float& out_key, float& out_pay) {
    uint32_t taken = 0;
    out_id = E; out_key = -INFINITY; out_pay = 0.0f;
    for (int j = 0; j < top_k; ++j) {
        float bk = -INFINITY, bp = 0.0f;
        int bi = E;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int id = lane + 32 * s;
            if (id < E && ((allowed >> s) & 1u) && !((taken >> s) & 1u) &&
                better(key[s], id, bk, bi, E)) {
                bk = key[s]; bi = id; bp = pay[s];
            }
        }
        warp_argmax(bk, bi, bp, E);
        if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) { out_id = bi; out_key = bk; out_pay = bp; }
    }
}

template <int SLOTS>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_softmax_kernel(const float* __restrict__ logits, int M, int E, int top_k, float rsf,
                     int32_t* __restrict__ ids, void* __restrict__ weights, int wdtype) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= M) return;
    const float* row = logits + static_cast<size_t>(t) * E;
    float key[SLOTS], pay[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int id = lane + 32 * s;
        key[s] = id < E ? __ldg(row + id) : -INFINITY;
        pay[s] = 0.0f;
    }
    int my_id; float my_key, my_pay;
    select_topk<SLOTS>(key, pay, 0xffffffffu, E, top_k, lane, my_id, my_key, my_pay);
    // The first winner holds the largest logit; the softmax restricted to the
    // selected experts and renormalised equals exp(l_j - l_max) / sum.
    const float lmax = __shfl_sync(0xffffffffu, my_key, 0);
    const float ex = lane < top_k ? expf(my_key - lmax) : 0.0f;
    const float denom = warp_sum(ex);
    if (lane < top_k) {
        const size_t o = static_cast<size_t>(t) * top_k + lane;
        ids[o] = my_id;
        store_from_f32(weights, o, ex / denom * rsf, wdtype);
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
    float* b_row = sh_b + warp * E;
    const float* row = logits + static_cast<size_t>(t) * E;
    float key[SLOTS], sc[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int id = lane + 32 * s;
        if (id < E) {
            sc[s] = sigmoid_spec(__ldg(row + id));
            key[s] = __fadd_rn(sc[s], __ldg(bias + id));
            b_row[id] = key[s];
        } else {
            sc[s] = 0.0f;
            key[s] = -INFINITY;
        }
    }
    __syncwarp();
    // group score: float32 sum of the group's two largest biased scores
    const int G = E / n_group;
    float gscore = -INFINITY;
    if (lane < n_group) {
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int i = 0; i < G; ++i) {
            const float v = b_row[lane * G + i];
            if (v > m1) { m2 = m1; m1 = v; }
            else if (v > m2) { m2 = v; }
        }
        gscore = __fadd_rn(m1, m2);
    }
    // keep the topk_group best groups (ties to the lower group id)
    uint32_t gtaken = 0;
    for (int j = 0; j < topk_group; ++j) {
        float k = (lane < n_group && !((gtaken >> lane) & 1u)) ? gscore : -INFINITY;
        int gi = (lane < n_group && !((gtaken >> lane) & 1u)) ? lane : n_group;
        float dummy = 0.0f;
        warp_argmax(k, gi, dummy, n_group);
        if (gi < n_group) gtaken |= 1u << gi;
    }
    uint32_t allowed = 0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int id = lane + 32 * s;
        if (id < E && ((gtaken >> (id / G)) & 1u)) allowed |= 1u << s;
    }
    int my_id; float my_key, my_s;
    select_topk<SLOTS>(key, sc, allowed, E, top_k, lane, my_id, my_key, my_s);
    const float sv = lane < top_k ? my_s : 0.0f;
    const float denom = warp_sum(sv);
    if (lane < top_k) {
        const size_t o = static_cast<size_t>(t) * top_k + lane;
        ids[o] = my_id;
        store_from_f32(weights, o, sv / denom * rsf, wdtype);
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
    debug_sigmoid_kernel<<<ceil_div(n, 256), 256, 0, s>>>(x, y, n);
    return cudaGetLastError();
}

}  // namespace moe

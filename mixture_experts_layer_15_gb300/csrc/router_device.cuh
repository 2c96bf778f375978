// Per-warp routing of one token, shared by the router kernels and the fused
// route+permute kernel (so both give the same bits). [Router] of
// vllm/model_executor/layers/fused_moe/modular_kernel.py (module header);
// the two methods are softmax -> top-k -> renormalise, and sigmoid +
// selection bias -> grouped top-k -> renormalise x scale (DeepSeek-V3's
// published routing rule).
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {
namespace route {

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

// 1/(1+e) correctly rounded: __frcp_rn gives the same bits as __fdiv_rn(1, .)
__device__ __forceinline__ float sigmoid_spec(float x) {
    return __frcp_rn(__fadd_rn(1.0f, exp_spec(-x)));
}

// Order-preserving 32-bit image of a float32 selection key: a > b (as floats)
// iff img(a) > img(b) (unsigned). -0.0 is folded onto +0.0 first, so the two
// compare equal as floats do; NaN maps to 0, below every other key.
__device__ __forceinline__ uint32_t key_image(float k) {
    if (isnan(k)) return 0u;
    const uint32_t u = __float_as_uint(__fadd_rn(k, 0.0f));       // -0.0 + 0.0 = +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// top_k selection rounds over the lane's SLOTS candidates. `key[s]` is the
// selection key of expert lane + 32*s, `pay[s]` a value carried along,
// `allowed` a bit mask of eligible slots. Order: larger key first, equal keys
// to the lower expert id. Each round takes the warp maximum of the key images
// (one redux), then the lowest expert id holding it: the lowest slot whose
// ballot is non-empty, and the lowest lane in that ballot. Lane j < top_k ends
// with the j-th winner in (out_id, out_key, out_pay).
template <int SLOTS>
__device__ __forceinline__ void select_topk(const float (&key)[SLOTS], const float (&pay)[SLOTS],
                                            uint32_t allowed, int E, int top_k, int lane,
                                            int& out_id, float& out_key, float& out_pay) {
    uint32_t img[SLOTS];
    uint32_t live = 0;                                   // slots still selectable
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        img[s] = key_image(key[s]);
        if (lane + 32 * s < E && ((allowed >> s) & 1u)) live |= 1u << s;
    }
    out_id = E; out_key = -INFINITY; out_pay = 0.0f;
    for (int j = 0; j < top_k; ++j) {
        uint32_t m = 0;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s)
            if (((live >> s) & 1u) && img[s] > m) m = img[s];
        const uint32_t any = __ballot_sync(0xffffffffu, live != 0);
        if (any == 0) break;                             // fewer candidates than top_k
        const uint32_t gmax = __reduce_max_sync(0xffffffffu, m);
        int win = -1;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const uint32_t b = __ballot_sync(0xffffffffu, ((live >> s) & 1u) && img[s] == gmax);
            if (win < 0 && b != 0) win = 32 * s + __ffs(b) - 1;
        }
        const int ws = win >> 5, wl = win & 31;
        float wk = 0.0f, wp = 0.0f;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s)
            if (s == ws) { wk = key[s]; wp = pay[s]; }
        wk = __shfl_sync(0xffffffffu, wk, wl);
        wp = __shfl_sync(0xffffffffu, wp, wl);
        if (lane == wl) live &= ~(1u << ws);
        if (lane == j) { out_id = win; out_key = wk; out_pay = wp; }
    }
}

// One warp routes one token (the logits row `row`): lane j < top_k returns
// the j-th selected expert and its weight.
template <int SLOTS>
__device__ __forceinline__ void route_token_softmax(const float* __restrict__ row, int E, int top_k, float rsf,
                                                    int lane, int& out_id, float& out_w) {
    float key[SLOTS], pay[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int id = lane + 32 * s;
        key[s] = id < E ? row[id] : -INFINITY;
        pay[s] = 0.0f;
    }
    int my_id; float my_key, my_pay;
    select_topk<SLOTS>(key, pay, 0xffffffffu, E, top_k, lane, my_id, my_key, my_pay);
    // The first winner holds the largest logit; the softmax restricted to the
    // selected experts and renormalised equals exp(l_j - l_max) / sum.
    const float lmax = __shfl_sync(0xffffffffu, my_key, 0);
    const float ex = lane < top_k ? expf(my_key - lmax) : 0.0f;
    const float denom = warp_sum(ex);
    out_id = my_id;
    out_w = ex / denom * rsf;
}

// Sigmoid + bias, grouped top-k. `b_row` is this warp's shared-memory scratch
// of E floats.
template <int SLOTS>
__device__ __forceinline__ void route_token_sigmoid(const float* __restrict__ row, const float* __restrict__ bias,
                                                    int E, int top_k, int n_group, int topk_group, float rsf,
                                                    int lane, float* b_row, int& out_id, float& out_w) {
    float key[SLOTS], sc[SLOTS];
    // every load first (one memory round trip for the token, not one per slot:
    // the sigmoid's branches would otherwise keep the later loads behind it)
    float lg[SLOTS], bs[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int id = lane + 32 * s;
        lg[s] = id < E ? __ldg(row + id) : 0.0f;
        bs[s] = id < E ? __ldg(bias + id) : 0.0f;
    }
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int id = lane + 32 * s;
        if (id < E) {
            sc[s] = sigmoid_spec(lg[s]);
            key[s] = __fadd_rn(sc[s], bs[s]);
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
    if (G == 32) {
        // group g is slot g (experts 32g .. 32g+31): its two largest keys by
        // warp reductions; the sum is of the same two floats as below
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            if (s >= n_group) break;
            const uint32_t im = key_image(key[s]);
            const uint32_t m1 = __reduce_max_sync(0xffffffffu, im);
            const uint32_t b1 = __ballot_sync(0xffffffffu, im == m1);
            const int l1 = __ffs(b1) - 1;
            const float f1 = __shfl_sync(0xffffffffu, key[s], l1);
            float f2;
            if (__popc(b1) >= 2) {
                f2 = f1;
            } else {
                const uint32_t m2 = __reduce_max_sync(0xffffffffu, lane == l1 ? 0u : im);
                const uint32_t b2 = __ballot_sync(0xffffffffu, lane != l1 && im == m2);
                f2 = __shfl_sync(0xffffffffu, key[s], __ffs(b2) - 1);
            }
            if (lane == s) gscore = __fadd_rn(f1, f2);
        }
    } else if (lane < n_group) {
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int i = 0; i < G; ++i) {
            const float v = b_row[lane * G + i];
            if (v > m1) { m2 = m1; m1 = v; }
            else if (v > m2) { m2 = v; }
        }
        gscore = __fadd_rn(m1, m2);
    }
    __syncwarp();
    // keep the topk_group best groups (ties to the lower group id); lane g < n_group
    // holds group g's score
    uint32_t gtaken = 0;
    {
        const uint32_t gimg = key_image(gscore);
        bool glive = lane < n_group;
        for (int j = 0; j < topk_group; ++j) {
            const uint32_t gmax = __reduce_max_sync(0xffffffffu, glive ? gimg : 0u);
            const uint32_t b = __ballot_sync(0xffffffffu, glive && gimg == gmax);
            if (b == 0) break;
            const int gi = __ffs(b) - 1;
            gtaken |= 1u << gi;
            if (lane == gi) glive = false;
        }
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
    out_id = my_id;
    out_w = sv / denom * rsf;
}

}  // namespace route
}  // namespace moe

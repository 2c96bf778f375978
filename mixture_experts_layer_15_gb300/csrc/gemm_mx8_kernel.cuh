// Grouped expert GEMMs with MXFP8 activations on the block-scaled tensor
// cores (tcgen05.mma kind::mxf8f6f4, E8M0 scales, one per 32 reduction
// elements of every row of both operands).
//
// The weights are MXFP4 (e2m1 codes + one E8M0 scale per 32, the recipe
// flashinfer_moe_ep.py ``FI_MOE_EP_BACKEND_SPECS`` names for the deep_gemm
// entry), the activations MXFP8 (E4M3 + E8M0 per 32), the ``quantize_input``
// step of build_fi_mega_config. Where the bf16-activation path decodes every
// weight tile to bf16 in shared memory, here the tensor core reads the codes
// and applies both scales itself:
//   A (weights, the MMA's M side): e2m1 codes by TMA with the
//     16U4_ALIGN16B data type -- every 8 bytes of codes land followed by 8
//     bytes of padding, the 4-bit operand layout of kind::mxf8f6f4 -- so a
//     k-block of 128 codes is a 128-byte row under the 128-byte swizzle;
//     HBM traffic stays at 64 bytes per row per k-block;
//   B (activations, the MMA's N side): E4M3 bytes, 128 per row per k-block;
//   scales: for each 128-row operand tile and k-block a 512-byte "atom",
//     row r's four scale bytes (its four 32-element chunks) at byte
//     (r % 32) * 16 + (r / 32) * 4; tcgen05.cp (32x128b, replicated to the
//     four TMEM subpartitions) moves an atom into four TMEM columns, where the
//     MMA of chunk j reads byte j (the descriptor's scale id) of row r's word
//     at lane r % 32, column r / 32. Weight atoms are written once by
//     moe_mx_prepare_scales; activation atoms by the quantiser (GEMM1's B)
//     and by GEMM1's epilogue (GEMM2's B), one atom per token tile of BT <=
//     128 rows and k-block, token n of the tile in atom row n.
//
// Units, split-K and the finalizing GEMM2 epilogue are those of the
// bf16-activation kernel (gemm_kernel.cuh); k-blocks are 128 elements. GEMM1
// units hold the gate tile and the up tile of the same 128 features, so the
// epilogue computes act(gate) * up per thread and quantises it at once: a
// warp's 32 lanes hold 32 consecutive features of a token, which is one MX
// block of GEMM2's reduction, so its scale is one warp max-reduction.
//
// CTA warps (persistent, one CTA per SM): warp 0 TMA producer; warps 1 and
// 2 the MMA issuers, one per A tile (warp 1 also allocates TMEM); warps
// 3..10 epilogue. One thread issuing every MMA and scale copy of a k-block
// bounds the kernel (its issue rate, not the tensor pipe, sets the pace at
// these tile shapes), so each A tile has its own issuing thread: it copies
// its A atom and its own copy of the B atom (a copy by one thread is not
// ordered before another thread's MMAs) and commits to the ring and
// accumulator barriers, which count both. TMEM holds the accumulators
// (double-buffered when they leave room) and, per ring stage and issuer,
// eight scale columns (its A atom, its B atom).
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "gemm_kernel.cuh"

namespace moe {
namespace gemm {

constexpr int kMxBK = 128;                     // reduction elements per k-block
constexpr int kAtom = 512;                     // bytes of one scale atom

template <int BT>
struct Cfg8 {
    static constexpr int EPI_WARPS = 8;
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    static constexpr int THREADS = 96 + EPI_THREADS;
    static constexpr int ISSUERS = 2;                      // MMA-issuing warps (one per A tile)
    static constexpr int A_BYTES = kBM * kMxBK;            // padded e2m1 tile in shared memory
    static constexpr int A_TX = kBM * kMxBK / 2;           // its transaction bytes (packed codes)
    static constexpr int B_BYTES = BT * kMxBK;
    static constexpr int OFF_SF = 2 * A_BYTES + B_BYTES;   // three atoms: A0, A1, B
    static constexpr int STAGE_BYTES = (OFF_SF + 3 * kAtom + 1023) / 1024 * 1024;
    static constexpr int STAGE_TX = 2 * A_TX + B_BYTES + 3 * kAtom;
    // the ring takes what the 227 KB a CTA may have leaves beside the rest of
    // the layout below (barriers, group tables, route table, alignment: < 16 KB)
    static constexpr int STAGES_FIT = (227 * 1024 - 16 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int SF_COLS = 16;                     // TMEM scale columns per stage (8 per issuer)
    static constexpr int ACC_COLS = 2 * BT;
    static constexpr int NBUF = (2 * ACC_COLS + STAGES * SF_COLS <= 512) ? 2 : 1;
    static constexpr int SF_BASE = NBUF * ACC_COLS;
    static constexpr int TMEM_NEED = SF_BASE + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64
                                   : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
    static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
    // full[S], empty[S], tfull[2], tempty[2], drain
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_PREFIX = OFF_MISC + 16;                     // [kMaxGroups+1] units
    static constexpr int OFF_TTP = OFF_PREFIX + (kMaxGroups + 1) * 4;    // [kMaxGroups+1] token tiles
    static constexpr int OFF_OFFS = OFF_TTP + (kMaxGroups + 1) * 4;      // [kMaxGroups+1]
    static constexpr int OFF_TMP = OFF_OFFS + (kMaxGroups + 1) * 4;      // [33]
    static constexpr int OFF_ROUTE = OFF_TMP + 36 * 4;                   // MODE_FINAL: [BT] token, [BT] scale
    static constexpr int SMEM_BYTES = OFF_ROUTE + 2 * BT * 4 + 1024;
    static_assert(STAGES >= 2, "ring too shallow");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(BT % 16 == 0 && BT >= 16 && BT <= 128, "token tile: one scale atom");
    static_assert(TMEM_NEED <= 512, "TMEM");
    static_assert(SF_BASE % 4 == 0 && OFF_SF % 16 == 0, "scale columns / atoms aligned");
};

// Arguments of one block-scaled GEMM. g: as for the other grouped GEMMs, with
// g.out = act codes [rows, N] (GEMM1) or y / the f32 output (GEMM2).
struct Mx8Args {
    GemmArgs g;
    const uint8_t* sfa;       // weight atoms [(groups * rows_per_group) / 128][kr / 128][512]
    const uint8_t* sfb;       // activation atoms [token tiles][kr / 128][512]
    uint8_t* sfb_out;         // GEMM1: act atoms for GEMM2 [token tiles][N / 128][512]
    int max_token_tiles;      // token tiles the atom buffers hold
};

// TT: tokens per token tile; HL: each token is two B rows (its hi and lo
// terms), so the tile's MMA N is twice its tokens (rounded up to 16).
__device__ __forceinline__ Unit decode_unit8(int u, const int* prefix, const int* offs, int TT, const GemmArgs& a,
                                             bool hl = false) {
    int lo = 0, hi = a.groups;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= u) lo = mid; else hi = mid;
    }
    Unit un;
    un.g = lo;
    int local = u - prefix[lo];
    un.s = local % a.splits;
    local /= a.splits;
    const int beg = offs[lo], end = offs[lo + 1];
    const int ntt = (end - beg + TT - 1) / TT;
    const int tt = local % ntt;
    un.wt = local / ntt;
    un.row0 = beg + tt * TT;
    un.row_end = min(end, a.rows_alloc);
    const int rows = min(TT, un.row_end - un.row0) * (hl ? 2 : 1);
    un.ncols = (rows + 15) & ~15;
    if (un.ncols < 16) un.ncols = 16;
    const int nkb = a.kr / kMxBK;
    un.kb0 = un.s * nkb / a.splits;
    un.kb1 = (un.s + 1) * nkb / a.splits;
    un.tile = u / a.splits;
    return un;
}

__device__ __forceinline__ int atom_byte(int n, int chunk) { return (n & 31) * 16 + ((n >> 5) << 2) + chunk; }

// MX block scale of a block whose largest magnitude has float32 bits `amax`:
// 2^(floor(log2 amax) - 8) as its E8M0 byte, kept in 1..254.
__device__ __forceinline__ uint32_t mx8_scale_byte(uint32_t amax_bits) {
    const int b = static_cast<int>((amax_bits >> 23) & 0xFFu) - 8;
    return static_cast<uint32_t>(b < 1 ? 1 : (b > 254 ? 254 : b));
}
// 1 / scale = 2^(127 - byte), a normal float for bytes 1..254 reachable here (<= 246)
__device__ __forceinline__ float mx8_inv_scale(uint32_t byte) { return __uint_as_float((254u - byte) << 23); }
__device__ __forceinline__ uint8_t e4m3_rn(float v) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// GEMM1 epilogue of 16 token columns: act = act(gate) * up, quantised in MX
// blocks of the warp's 32 features; codes to out[r, f], the block scale of
// each column to the act atom of (token tile, k-block wt) for GEMM2.
__device__ __forceinline__ void emit16_swiglu_mx8(const Unit& un, const Mx8Args& m, int q, int lane, int c0, int T,
                                                  const float (&v0)[16], const float (&v1)[16]) {
    const GemmArgs& a = m.g;
    uint8_t* out = static_cast<uint8_t*>(a.out);
    const int f = un.wt * kBM + q * 32 + lane;              // this lane's feature
    const size_t atom = (static_cast<size_t>(T) * (a.out_ld / kMxBK) + un.wt) * kAtom;
    float act[16];
    if (!act_is_plain(a.act, a.clamp)) {
#pragma unroll
        for (int i = 0; i < 16; ++i) act[i] = act_mul(v0[i], v1[i], a.act, a.clamp);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) act[i] = silu_mul(v0[i], v1[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(act[i]) & 0x7FFFFFFFu);
        const uint32_t sb = mx8_scale_byte(amax);
        const int r = un.row0 + c0 + i;
        if (r < un.row_end) {
            out[static_cast<size_t>(r) * a.out_ld + f] = e4m3_rn(act[i] * mx8_inv_scale(sb));
            if (lane == 0) m.sfb_out[atom + atom_byte(c0 + i, q)] = static_cast<uint8_t>(sb);
        }
    }
}

// ---- bf16 activations as two E4M3 terms (MOE_WEIGHTS_MXFP4_A16) -------------------
// A bf16 value x (8 significant bits) is split into hi + lo, each an E4M3 code
// (4 significant bits) times a per-32-block power-of-two scale:
//   hi = e4m3(x / s1) * s1,  lo = e4m3((x - hi) / s2) * s2,
// with s = the smallest power of two for which the block's largest magnitude
// is at most 448 * s (no code saturates). x - hi is exact in float32 and a
// multiple of x's ulp no larger than 8 ulp, so lo holds it exactly whenever
// it is a normal or subnormal E4M3 multiple of s2 -- every element within 2^14
// of its block's largest magnitude. The block-scaled MMA then computes the
// bf16-activation contraction as two e2m1 x E4M3 products summed in float32.

// Scale byte b (scale 2^(b-127)): smallest with amax <= 448 * 2^(b-127), in 1..254.
__device__ __forceinline__ uint32_t hl_scale_byte(uint32_t amax_bits) {
    const int e = static_cast<int>((amax_bits >> 23) & 0xFFu);
    const int b = e - 8 + ((amax_bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return static_cast<uint32_t>(b < 1 ? 1 : (b > 254 ? 254 : b));
}
__device__ __forceinline__ float e4m3_value(uint8_t code) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
    return __half2float(__half(h));
}

// GEMM1 epilogue of 16 accumulator columns = 8 tokens (hi and lo columns of a
// token summed): act = act(gate) * up, rounded to bf16, split into hi and lo
// over the warp's 32 features (one MX block of GEMM2's reduction); codes to
// act rows 2r (hi) and 2r + 1 (lo), block scales to the act atom.
__device__ __forceinline__ void emit16_swiglu_hl(const Unit& un, const Mx8Args& m, int q, int lane, int c0, int T,
                                                 const float (&v0)[16], const float (&v1)[16]) {
    const GemmArgs& a = m.g;
    uint8_t* out = static_cast<uint8_t*>(a.out);
    const int f = un.wt * kBM + q * 32 + lane;
    const size_t atom = (static_cast<size_t>(T) * (a.out_ld / kMxBK) + un.wt) * kAtom;
    const bool plain = act_is_plain(a.act, a.clamp);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float g = v0[2 * i] + v0[2 * i + 1], u = v1[2 * i] + v1[2 * i + 1];
        const float x = __bfloat162float(__float2bfloat16_rn(plain ? silu_mul(g, u) : act_mul(g, u, a.act, a.clamp)));
        const uint32_t b1 = hl_scale_byte(__reduce_max_sync(0xffffffffu, __float_as_uint(x) & 0x7FFFFFFFu));
        const uint8_t c1 = e4m3_rn(x * mx8_inv_scale(b1));
        const float r = x - e4m3_value(c1) * __uint_as_float(b1 << 23);      // exact
        const uint32_t b2 = hl_scale_byte(__reduce_max_sync(0xffffffffu, __float_as_uint(r) & 0x7FFFFFFFu));
        const uint8_t c2 = e4m3_rn(r * mx8_inv_scale(b2));
        const int row = un.row0 + c0 / 2 + i;
        if (row < un.row_end) {
            out[static_cast<size_t>(2 * row) * a.out_ld + f] = c1;
            out[static_cast<size_t>(2 * row + 1) * a.out_ld + f] = c2;
            if (lane == 0) {
                m.sfb_out[atom + atom_byte(c0 + 2 * i, q)] = static_cast<uint8_t>(b1);
                m.sfb_out[atom + atom_byte(c0 + 2 * i + 1, q)] = static_cast<uint8_t>(b2);
            }
        }
    }
}

// GEMM2 epilogues of 16 accumulator columns = 8 tokens: y = hi column + lo
// column, then as emit16 / emit16_final for token (not column) i.
template <typename OutT>
__device__ __forceinline__ void emit8_plain_hl(const Unit& un, const GemmArgs& a, int row_in_tile, int c0,
                                               const float (&v0)[16], const float (&v1)[16]) {
    OutT* out = static_cast<OutT*>(a.out);
    const int col = un.wt * a.wtile_rows + row_in_tile;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = un.row0 + c0 / 2 + i;
        if (r < un.row_end) {
            const size_t rb = static_cast<size_t>(r) * a.out_ld;
            store_out<OutT>(out + rb + col, v0[2 * i] + v0[2 * i + 1]);
            store_out<OutT>(out + rb + col + kBM, v1[2 * i] + v1[2 * i + 1]);
        }
    }
}

__device__ __forceinline__ void emit8_final_hl(const Unit& un, const GemmArgs& a, int row_in_tile, int c0,
                                               const int* tok, const float* scl, const float (&v0)[16],
                                               const float (&v1)[16]) {
    float* out = static_cast<float*>(a.out);
    const int col = un.wt * a.wtile_rows + row_in_tile;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = tok[c0 / 2 + i];
        if (t >= 0) {
            const float si = scl[c0 / 2 + i];
            float* o = out + static_cast<size_t>(t) * a.out_ld + col;
            atomicAdd(o, si * (v0[2 * i] + v0[2 * i + 1]));
            atomicAdd(o + kBM, si * (v1[2 * i] + v1[2 * i + 1]));
        }
    }
}

// BT: B rows per token tile (<= 128: one scale atom). HL: each token is two
// B rows (bf16 activations as two E4M3 terms), so a tile holds BT / 2 tokens.
template <int BT, int MODE, typename OutT, bool HL>
__global__ void __launch_bounds__(Cfg8<BT>::THREADS, 1)
grouped_gemm_mx8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const Mx8Args m) {
    using C = Cfg8<BT>;
    constexpr int TT = HL ? BT / 2 : BT;                   // tokens per token tile
    constexpr int kEpiThreads = C::EPI_THREADS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto full_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int b) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + b); };
    auto tempty_bar = [&](int b) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 2 + b); };
    const uint32_t drain_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
    int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
    int* ttp = reinterpret_cast<int*>(smem + C::OFF_TTP);
    int* offs = reinterpret_cast<int*>(smem + C::OFF_OFFS);
    int* tmp = reinterpret_cast<int*>(smem + C::OFF_TMP);
    int* route_tok = reinterpret_cast<int*>(smem + C::OFF_ROUTE);
    float* route_scl = reinterpret_cast<float*>(smem + C::OFF_ROUTE + 4 * BT);
    const GemmArgs& a = m.g;
    const int groups = a.groups;
    const int nkb_all = a.kr / kMxBK;

    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), C::ISSUERS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), C::ISSUERS);
            mbar_init(tempty_bar(b), kEpiThreads);
        }
        mbar_init(drain_bar, C::ISSUERS);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_trigger();
    for (int g = tid; g <= groups; g += C::THREADS) {
        int v = a.offsets != nullptr ? __ldg(a.offsets + g) : (g == 0 ? 0 : a.single_rows);
        if (v < 0 || v > a.rows_alloc) { set_error(a.err, MOE_ERR_DEVICE_INDEX); v = v < 0 ? 0 : a.rows_alloc; }
        offs[g] = v;
    }
    __syncthreads();
    for (int g = tid; g < groups; g += C::THREADS) {
        int cnt = offs[g + 1] - offs[g];
        if (cnt < 0) { set_error(a.err, MOE_ERR_DEVICE_INDEX); cnt = 0; }
        const int ntt = (cnt + TT - 1) / TT;
        prefix[g] = ntt * a.n_wtiles * a.splits;
        ttp[g] = ntt;
    }
    __syncthreads();
    int total_units = block_exclusive_scan(prefix, groups, tmp);
    const int ntiles = block_exclusive_scan(ttp, groups, tmp);
    if (ntiles > m.max_token_tiles) {                  // offsets not from a permute: touch nothing
        if (tid == 0) set_error(a.err, MOE_ERR_DEVICE_INDEX);
        total_units = 0;
    }
    if (tid == 0) prefix[groups] = total_units;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // global index of a unit's token tile: the row of its activation atoms
    auto tile_index = [&](const Unit& un) { return ttp[un.g] + (un.row0 - offs[un.g]) / TT; };

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
                const Unit un = decode_unit8(u, prefix, offs, TT, a, HL);
                const int a_row = un.g * a.rows_per_group + un.wt * a.wtile_rows;
                const uint8_t* sfa0 = m.sfa + static_cast<size_t>(a_row / kBM) * nkb_all * kAtom;
                const uint8_t* sfa1 = m.sfa + static_cast<size_t>((a_row + a.a1_offset) / kBM) * nkb_all * kAtom;
                const uint8_t* sfb = m.sfb + static_cast<size_t>(tile_index(un)) * nkb_all * kAtom;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
                    const uint32_t st = sbase + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(full_bar(stage), C::STAGE_TX);
                    tma_load_2d(st, &tmA, kb * kMxBK, a_row, full_bar(stage));
                    tma_load_2d(st + C::A_BYTES, &tmA, kb * kMxBK, a_row + a.a1_offset, full_bar(stage));
                    tma_load_2d(st + 2 * C::A_BYTES, &tmB, kb * kMxBK, HL ? 2 * un.row0 : un.row0, full_bar(stage));
                    bulk_load(st + C::OFF_SF, sfa0 + kb * kAtom, kAtom, full_bar(stage));
                    bulk_load(st + C::OFF_SF + kAtom, sfa1 + kb * kAtom, kAtom, full_bar(stage));
                    bulk_load(st + C::OFF_SF + 2 * kAtom, sfb + kb * kAtom, kAtom, full_bar(stage));
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                for (int s = 0; s < C::STAGES; ++s) {
                    if (!((issued >> s) & 1u)) continue;
                    const uint32_t p = (issued_phase >> s) & 1u;
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(full_bar(s), p) && globaltimer() - t0 < kWaitLimitNs) {}
                }
            }
        }
        __syncwarp();
    } else if (warp <= C::ISSUERS) {
        // ================= scale copies + MMA issuers (warp 1: A0, warp 2: A1) =================
        const int h = warp - 1;
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x, ++it) {
                const Unit un = decode_unit8(u, prefix, offs, TT, a, HL);
                const int buf = C::NBUF == 2 ? (it & 1) : 0;
                const uint32_t use = C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1);
                if (!wait_bar(tempty_bar(buf), use ^ 1u, abort_flag, a.err)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + buf * C::ACC_COLS + h * BT;
                // the chunk-kk instruction descriptor is idesc0 with scale id kk in both id fields
                const uint32_t idesc0 = idesc_mx(MX_E2M1, MX_E4M3, kBM, un.ncols, 0);
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!wait_bar(full_bar(stage), phase, abort_flag, a.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = sbase + stage * C::STAGE_BYTES;
                    // this issuer's columns: its A atom at sf, its copy of the B atom at sf + 4
                    const uint32_t sf = tmem_base + C::SF_BASE + stage * C::SF_COLS + 8 * h;
                    const uint64_t dsf = rows16_desc(st + C::OFF_SF);       // atoms 512 bytes apart: +32
                    tmem_copy_atom(sf, dsf + h * (kAtom / 16));             // A_h scales: columns sf .. sf+3
                    tmem_copy_atom(sf + 4, dsf + 2 * kAtom / 16);           // B scales
                    // chunk kk starts 32 bytes further into each 128-byte row: +2 in the
                    // descriptors' 16-byte address field
                    const uint64_t dA = sw128_kmajor_desc(st + h * C::A_BYTES);
                    const uint64_t dB = sw128_kmajor_desc(st + 2 * C::A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kMxBK / 32; ++kk) {
                        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(kk) << 4) | (static_cast<uint32_t>(kk) << 29);
                        const uint32_t acc = (kb > un.kb0 || kk > 0) ? 1u : 0u;
                        mma_mx(d, dA + 2 * kk, dB + 2 * kk, idesc, sf, sf + 4, acc);
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tfull_bar(buf));
            }
            mma_commit(drain_bar);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < kWaitLimitNs) {}
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 3..10) =================
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        const int etid = tid - 96;
        const int c_first = 16 * ((warp - 3) >> 2);
        constexpr int c_step = 16 * (C::EPI_WARPS / 4);
        auto emit = [&](const Unit& un, int c0, const float (&v0)[16], const float (&v1)[16]) {
            if constexpr (HL) {
                if constexpr (MODE == MODE_SWIGLU) emit16_swiglu_hl(un, m, q, lane, c0, tile_index(un), v0, v1);
                else if constexpr (MODE == MODE_FINAL)
                    emit8_final_hl(un, a, row_in_tile, c0, route_tok, route_scl, v0, v1);
                else emit8_plain_hl<OutT>(un, a, row_in_tile, c0, v0, v1);
            } else {
                if constexpr (MODE == MODE_SWIGLU) emit16_swiglu_mx8(un, m, q, lane, c0, tile_index(un), v0, v1);
                else if constexpr (MODE == MODE_FINAL)
                    emit16_final<2>(un, a, row_in_tile, c0, route_tok, route_scl, v0, v1);
                else emit16<2, MODE_PLAIN, OutT>(un, a, row_in_tile, c0, v0, v1);
            }
        };
        // a finalizing call's output start (written by its GEMM1 launch)
        if (a.init_out != nullptr) init_out_share(a, blockIdx.x, gridDim.x, etid, kEpiThreads);
        int it = 0;
        for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++it) {
            const Unit un = decode_unit8(u, prefix, offs, TT, a, HL);
            const int buf = C::NBUF == 2 ? (it & 1) : 0;
            const uint32_t use = C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1);
            if (MODE == MODE_FINAL) {
                named_bar_sync(1, kEpiThreads);
                // one table entry per token (HL: half the tile's columns)
                Unit ut = un;
                if (HL) ut.ncols = un.ncols / 2;
                load_route_table(ut, a, etid, kEpiThreads, route_tok, route_scl);
            }
            wait_bar(tfull_bar(buf), use, abort_flag, a.err);
            if (named_bar_or(1, kEpiThreads, *abort_flag != 0)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::ACC_COLS;
            const bool direct = a.splits == 1 || MODE == MODE_FINAL;
            if (direct) {
                // the quantising epilogue reduces across the warp: every lane of a
                // warp runs the same chunks
#pragma unroll 1
                for (int c0 = c_first; c0 < un.ncols; c0 += c_step) {
                    float v0[16], v1[16];
                    tmem_ld16x2(tb + c0, tb + BT + c0, v0, v1);
                    emit(un, c0, v0, v1);
                }
                tc_fence_before();
                mbar_arrive(tempty_bar(buf));
            } else {
                const size_t slot = static_cast<size_t>(2) * kBM * BT;
                const bool tile_ok = un.tile < a.max_tiles;
                float* part = a.partials + (static_cast<size_t>(un.tile) * a.splits + un.s) * slot;
#pragma unroll 1
                for (int c0 = c_first; c0 < un.ncols; c0 += c_step) {
                    float v0[16], v1[16];
                    tmem_ld16x2(tb + c0, tb + BT + c0, v0, v1);
                    if (tile_ok) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            part[static_cast<size_t>(c0 + i) * kBM + row_in_tile] = v0[i];
                            part[static_cast<size_t>(BT + c0 + i) * kBM + row_in_tile] = v1[i];
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(tempty_bar(buf));
                __threadfence();
                named_bar_sync(1, kEpiThreads);
                if (etid == 0) {
                    int last = 0;
                    if (tile_ok) {
                        const int old = atomicAdd(a.counters + un.tile, 1);
                        last = (old == a.splits - 1);
                        if (last) a.counters[un.tile] = 0;
                    } else {
                        set_error(a.err, MOE_ERR_DEVICE_INDEX);
                    }
                    *last_flag = last;
                }
                named_bar_sync(1, kEpiThreads);
                if (*last_flag) {
                    __threadfence();
                    const float* p0 = a.partials + static_cast<size_t>(un.tile) * a.splits * slot;
#pragma unroll 1
                    for (int c0 = c_first; c0 < un.ncols; c0 += c_step) {
                        float v0[16], v1[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) { v0[i] = 0.0f; v1[i] = 0.0f; }
                        for (int s = 0; s < a.splits; ++s) {
                            const float* ps = p0 + s * slot;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                v0[i] += __ldcg(ps + static_cast<size_t>(c0 + i) * kBM + row_in_tile);
                                v1[i] += __ldcg(ps + static_cast<size_t>(BT + c0 + i) * kBM + row_in_tile);
                            }
                        }
                        emit(un, c0, v0, v1);
                    }
                }
                named_bar_sync(1, kEpiThreads);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

template <int BT, int MODE, typename OutT, bool HL>
cudaError_t launch_mx8_kernel(const CUtensorMap& tA, const CUtensorMap& tB, const Mx8Args& m, int grid,
                              cudaStream_t s) {
    using C = Cfg8<BT>;
    auto kern = grouped_gemm_mx8_kernel<BT, MODE, OutT, HL>;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, s, tA, tB, m);
}

// bt: B rows per token tile (16, 32, 64 or 128; HL also 112).
template <int MODE, typename OutT, bool HL>
cudaError_t launch_mx8_bt(int bt, const CUtensorMap& tA, const CUtensorMap& tB, const Mx8Args& m, int grid,
                          cudaStream_t s) {
    switch (bt) {
        case 16: return launch_mx8_kernel<16, MODE, OutT, HL>(tA, tB, m, grid, s);
        case 32: return launch_mx8_kernel<32, MODE, OutT, HL>(tA, tB, m, grid, s);
        case 64: return launch_mx8_kernel<64, MODE, OutT, HL>(tA, tB, m, grid, s);
        case 112:
            if constexpr (HL) return launch_mx8_kernel<112, MODE, OutT, HL>(tA, tB, m, grid, s);
            else return cudaErrorInvalidValue;
        default: return launch_mx8_kernel<128, MODE, OutT, HL>(tA, tB, m, grid, s);
    }
}

// Defined in gemm_mx8.cu (hl = false: MXFP8 activations) and gemm_mx8_hl.cu
// (hl = true: bf16 activations as two E4M3 terms). mode: MODE_SWIGLU (GEMM1,
// act codes + atoms), MODE_PLAIN (GEMM2 into y of out_dtype) or MODE_FINAL
// (GEMM2 into the f32 out). bt: B rows per token tile.
cudaError_t launch_gemm_mx8(int mode, int bt, int out_dtype, const CUtensorMap& tA, const CUtensorMap& tB,
                            const Mx8Args& m, int grid, cudaStream_t s);
cudaError_t launch_gemm_mx8_hl(int mode, int bt, int out_dtype, const CUtensorMap& tA, const CUtensorMap& tB,
                               const Mx8Args& m, int grid, cudaStream_t s);

}  // namespace gemm
}  // namespace moe

// MXFP8 quantisation of activation rows and the scale layout of the
// block-scaled GEMMs.
//
// quantize_input (flashinfer_moe_ep.py, build_fi_mega_config), read as the
// MX recipe of the e2m1 + ue8m0-per-32 weights applied to the activations:
// every block of 32 consecutive values of a row shares the E8M0 scale
// 2^(floor(log2 amax) - 8) (8 = E4M3's largest exponent; the byte kept in
// 1..254), and each value becomes the E4M3 code nearest to value / scale
// (ties to even, saturated at 448) -- cvt.rn.satfinite.e4m3 on the exact
// power-of-two product. HBM-bound: one warp per row, 16-byte loads.
#include <cuda_fp8.h>

#include "common.cuh"
#include "gemm_mx8_kernel.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 256;

// ATOM = false: scales [rows, C/32] row-major. ATOM = true: the rows are
// grouped (offsets, `groups` groups) and cut into token tiles of `bt` rows
// per group; the scales go to the tile atoms the block-scaled GEMM reads
// (tile t, k-block kb: atom t * (C/128) + kb; row n of the tile, chunk j at
// byte (n % 32) * 16 + (n / 32) * 4 + j). Rows outside [offsets[0],
// offsets[groups]) are not touched; neither is anything when the groups need
// more than `max_tiles` tiles.
//
// HL: each row is split into two E4M3 terms, hi and lo, that sum to the bf16
// value (gemm_mx8_kernel.cuh, MOE_WEIGHTS_MXFP4_A16): row p's hi codes go to
// codes row 2p, its lo codes to row 2p + 1; in the tile atoms token n of a
// tile (bt tokens) has B rows 2n (hi) and 2n + 1 (lo), in the row-major scales
// rows 2p and 2p + 1.
//
// gather_inv (ATOM only, may be NULL): x holds the tokens in token order and
// row p reads token gather_inv[p] / gather_topk (the row gather of the permute,
// done here instead of through x_perm); an entry outside [0, rows_alloc) sets
// MOE_ERR_DEVICE_INDEX and the row is taken as zeros.
template <bool ATOM, bool HL>
__global__ void __launch_bounds__(kQThreads)
mxfp8_quantize_kernel(const __nv_bfloat16* __restrict__ x, int rows, int C, uint8_t* __restrict__ codes,
                      uint8_t* __restrict__ scales, const int32_t* __restrict__ offsets, int groups, int bt,
                      int rows_alloc, int max_tiles, int* err, const int32_t* __restrict__ gather_inv,
                      int gather_topk, int cpi) {
    __shared__ int s_offs[gemm::kMaxGroups + 1];
    __shared__ int s_ttp[gemm::kMaxGroups + 1];
    __shared__ int tmp[36];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int R = rows, p0 = 0;
    if (ATOM) {
        for (int g = tid; g <= groups; g += kQThreads) {
            int v = __ldg(offsets + g);
            if (v < 0 || v > rows_alloc) { set_error(err, MOE_ERR_DEVICE_INDEX); v = v < 0 ? 0 : rows_alloc; }
            s_offs[g] = v;
        }
        __syncthreads();
        for (int g = tid; g < groups; g += kQThreads) {
            const int cnt = s_offs[g + 1] - s_offs[g];
            s_ttp[g] = cnt > 0 ? (cnt + bt - 1) / bt : 0;
        }
        __syncthreads();
        const int ntiles = block_exclusive_scan(s_ttp, groups, tmp);
        p0 = s_offs[0];                                    // rows below the first group belong to none
        R = s_offs[groups];
        if (ntiles > max_tiles) {                          // offsets not from a permute: touch nothing
            if (tid == 0) set_error(err, MOE_ERR_DEVICE_INDEX);
            R = 0;
        }
    }
    const int nkb = C / gemm::kMxBK;
    const int nw = kQThreads / 32;
    // one warp per (row, group of cpi 256-column chunks): a row's groups go to
    // different warps, so a few rows still spread over many warps, and with
    // cpi = 4 a warp has the loads of its four chunks in flight at once
    // (cpi = 1 when the rows are too few to fill the GPU that way)
    const int chunks = (C + 255) / 256;
    const int ngr = (chunks + cpi - 1) / cpi;
    const long long items = static_cast<long long>(R > p0 ? R - p0 : 0) * ngr;
    for (long long it = static_cast<long long>(blockIdx.x) * nw + warp; it < items;
         it += static_cast<long long>(gridDim.x) * nw) {
        const int p = p0 + static_cast<int>(it / ngr);
        const int cbase = static_cast<int>(it % ngr) * 256 * cpi;
        int T = 0, n = 0;
        if (ATOM) {
            int lo = 0, hi = groups;                       // s_offs[lo] <= p < s_offs[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_offs[mid] <= p) lo = mid; else hi = mid;
            }
            const int local = p - s_offs[lo];
            T = s_ttp[lo] + local / bt;
            n = local % bt;
        }
        size_t src = static_cast<size_t>(p);
        bool zero = false;
        if (ATOM && gather_inv != nullptr) {
            const int e = __ldg(gather_inv + p);
            if (e < 0 || e >= rows_alloc) {
                if (lane == 0) set_error(err, MOE_ERR_DEVICE_INDEX);
                zero = true;
                src = 0;
            } else {
                src = static_cast<size_t>(e / gather_topk);
            }
        }
        const __nv_bfloat16* xr = x + src * C;
        uint8_t* cr = codes + static_cast<size_t>(p) * C;
        float vv[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = cbase + 256 * j + lane * 8;
            if (j < cpi && c < C && !zero) {
                Vec8<__nv_bfloat16>::load(xr + c, vv[j]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) vv[j][i] = 0.0f;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j >= cpi || cbase + 256 * j >= C) break;   // uniform over the warp
            const int c = cbase + 256 * j + lane * 8;
            const bool on = c < C;
            const float (&v)[8] = vv[j];
            float am = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(v[i]));
            // a block of 32 = 4 lanes x 8 values
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
            if (HL) {
                // hi = e4m3(v / s1) * s1, lo = e4m3((v - hi) / s2) * s2
                const uint32_t b1 = gemm::hl_scale_byte(__float_as_uint(am));
                const float inv1 = gemm::mx8_inv_scale(b1), s1 = __uint_as_float(b1 << 23);
                uint8_t c1[8];
                float r[8];
                float ar = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    c1[i] = gemm::e4m3_rn(v[i] * inv1);
                    r[i] = v[i] - gemm::e4m3_value(c1[i]) * s1;          // exact
                    ar = fmaxf(ar, fabsf(r[i]));
                }
                ar = fmaxf(ar, __shfl_xor_sync(0xffffffffu, ar, 1));
                ar = fmaxf(ar, __shfl_xor_sync(0xffffffffu, ar, 2));
                const uint32_t b2 = gemm::hl_scale_byte(__float_as_uint(ar));
                const float inv2 = gemm::mx8_inv_scale(b2);
                if (on) {
                    uint32_t h0 = 0, h1 = 0, l0 = 0, l1 = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        h0 |= static_cast<uint32_t>(c1[i]) << (8 * i);
                        h1 |= static_cast<uint32_t>(c1[4 + i]) << (8 * i);
                        l0 |= static_cast<uint32_t>(gemm::e4m3_rn(r[i] * inv2)) << (8 * i);
                        l1 |= static_cast<uint32_t>(gemm::e4m3_rn(r[4 + i] * inv2)) << (8 * i);
                    }
                    uint8_t* ch = codes + static_cast<size_t>(2 * p) * C;
                    *reinterpret_cast<uint2*>(ch + c) = make_uint2(h0, h1);
                    *reinterpret_cast<uint2*>(ch + C + c) = make_uint2(l0, l1);
                    if ((lane & 3) == 0) {
                        if (ATOM) {
                            uint8_t* at = scales + (static_cast<size_t>(T) * nkb + c / gemm::kMxBK) * gemm::kAtom;
                            const int jj = (c % gemm::kMxBK) / 32;
                            at[gemm::atom_byte(2 * n, jj)] = static_cast<uint8_t>(b1);
                            at[gemm::atom_byte(2 * n + 1, jj)] = static_cast<uint8_t>(b2);
                        } else {
                            uint8_t* sr = scales + static_cast<size_t>(2 * p) * (C / 32) + c / 32;
                            sr[0] = static_cast<uint8_t>(b1);
                            sr[C / 32] = static_cast<uint8_t>(b2);
                        }
                    }
                }
                continue;
            }
            const uint32_t sb = gemm::mx8_scale_byte(__float_as_uint(am));
            const float inv = gemm::mx8_inv_scale(sb);
            if (on) {
                uint32_t lo = 0, hi = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    lo |= static_cast<uint32_t>(gemm::e4m3_rn(v[i] * inv)) << (8 * i);
                    hi |= static_cast<uint32_t>(gemm::e4m3_rn(v[4 + i] * inv)) << (8 * i);
                }
                *reinterpret_cast<uint2*>(cr + c) = make_uint2(lo, hi);
                if ((lane & 3) == 0) {
                    if (ATOM)
                        scales[(static_cast<size_t>(T) * nkb + c / gemm::kMxBK) * gemm::kAtom +
                               gemm::atom_byte(n, (c % gemm::kMxBK) / 32)] = static_cast<uint8_t>(sb);
                    else
                        scales[static_cast<size_t>(p) * (C / 32) + c / 32] = static_cast<uint8_t>(sb);
                }
            }
        }
    }
}

// Scales [rows_total, cols/32] (row-major, one byte per 32 values) -> the
// atoms [rows_total/128][cols/128][512] of the block-scaled GEMM: row r of
// tile r/128, k-block kb: its four bytes (chunks 0..3) at byte
// (r % 32) * 16 + ((r % 128) / 32) * 4 of atom (r/128, kb).
__global__ void mx_prepare_scales_kernel(const uint8_t* __restrict__ sc, long long rows_total, int cols,
                                         uint8_t* __restrict__ out) {
    const int nkb = cols / gemm::kMxBK;
    const long long total = rows_total * nkb;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = i / nkb;
        const int kb = static_cast<int>(i % nkb);
        const uint32_t w = *reinterpret_cast<const uint32_t*>(sc + row * (cols / 32) + kb * 4);
        const int r = static_cast<int>(row % gemm::kBM);
        *reinterpret_cast<uint32_t*>(out + ((row / gemm::kBM) * nkb + kb) * gemm::kAtom + (r & 31) * 16 +
                                     ((r >> 5) << 2)) = w;
    }
}

}  // namespace

namespace {
// CTAs for rows x groups of four 256-column chunks, one warp per item, at
// most 8 per SM.
// Chunks per work item: 4, unless the rows give fewer items of four chunks
// than one CTA's warps per SM (then 1: four times the warps, each a quarter
// of the dependent work).
int quantize_cpi(int rows, int C, const DeviceInfo& dev) {
    const long long items4 = static_cast<long long>(rows) * ((C + 1023) / 1024);
    return items4 < static_cast<long long>(kQThreads / 32) * (dev.sm_count > 0 ? dev.sm_count : 152) ? 1 : 4;
}

int quantize_grid(int rows, int C, const DeviceInfo& dev) {
    const int cpi = quantize_cpi(rows, C, dev);
    const long long items = static_cast<long long>(rows) * ((C + 256 * cpi - 1) / (256 * cpi));
    const int nw = kQThreads / 32;
    long long grid = (items + nw - 1) / nw;
    const long long cap = 8LL * (dev.sm_count > 0 ? dev.sm_count : 152);
    if (grid > cap) grid = cap;
    return grid < 1 ? 1 : static_cast<int>(grid);
}
}  // namespace

cudaError_t launch_mxfp8_quantize(const void* x, int rows, int C, uint8_t* codes, uint8_t* scales, int* err,
                                  const DeviceInfo& dev, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int grid = quantize_grid(rows, C, dev);
    return launch_pdl(mxfp8_quantize_kernel<false, false>, dim3(grid), dim3(kQThreads), 0, s,
                      static_cast<const __nv_bfloat16*>(x), rows, C, codes, scales,
                      static_cast<const int32_t*>(nullptr), 0, 1, rows, 0, err, static_cast<const int32_t*>(nullptr),
                      1, quantize_cpi(rows, C, dev));
}

cudaError_t launch_e4m3_split(const void* x, int rows, int C, uint8_t* codes, uint8_t* scales, int* err,
                              const DeviceInfo& dev, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int grid = quantize_grid(rows, C, dev);
    return launch_pdl(mxfp8_quantize_kernel<false, true>, dim3(grid), dim3(kQThreads), 0, s,
                      static_cast<const __nv_bfloat16*>(x), rows, C, codes, scales,
                      static_cast<const int32_t*>(nullptr), 0, 1, rows, 0, err, static_cast<const int32_t*>(nullptr),
                      1, quantize_cpi(rows, C, dev));
}

cudaError_t launch_mxfp8_quantize_tiles(const void* x, int rows_alloc, int C, const int32_t* offsets, int groups,
                                        int bt, int max_tiles, uint8_t* codes, uint8_t* atoms, int* err,
                                        const DeviceInfo& dev, cudaStream_t s, bool hl, const int32_t* gather_inv,
                                        int gather_topk) {
    const int grid = quantize_grid(rows_alloc, C, dev);
    auto kern = hl ? mxfp8_quantize_kernel<true, true> : mxfp8_quantize_kernel<true, false>;
    return launch_pdl(kern, dim3(grid), dim3(kQThreads), 0, s, static_cast<const __nv_bfloat16*>(x), rows_alloc, C,
                      codes, atoms, offsets, groups, bt, rows_alloc, max_tiles, err, gather_inv,
                      gather_topk > 0 ? gather_topk : 1, quantize_cpi(rows_alloc, C, dev));
}

cudaError_t launch_mx_prepare_scales(const uint8_t* scales, long long rows_total, int cols, uint8_t* out,
                                     const DeviceInfo& dev, cudaStream_t s) {
    const long long total = rows_total * (cols / gemm::kMxBK);
    if (total == 0) return cudaSuccess;
    long long grid = (total + 255) / 256;
    if (grid > 16LL * dev.sm_count) grid = 16LL * dev.sm_count;
    return launch_plain(mx_prepare_scales_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, scales, rows_total,
                        cols, out);
}

}  // namespace moe

// Device helpers shared by the kernels of the MoE library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "moe_internal.h"

namespace moe {

// ---- device error word -------------------------------------------------------
// Kernels never trap: a detected problem records its status code here (first
// writer wins) and the kernel skips the offending item.
__device__ __forceinline__ void set_error(int* err, int code) {
    if (err != nullptr) atomicCAS(err, 0, code);
}

// ---- programmatic dependent launch --------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialisation, so it may start while the previous kernel of the stream is
// still finishing. It may only do local set-up (shared memory, TMEM, barrier
// initialisation) before pdl_wait(), which returns once every earlier kernel
// of the stream has completed and its writes are visible; all global-memory
// reads and writes come after it. pdl_trigger() lets the next kernel start
// its own set-up; it is issued right after pdl_wait() by every CTA, so a
// dependent grid can only start once every CTA of this grid is resident (no
// CTA of this grid can then be starved of an SM by the waiting dependents).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Plain (stream-ordered) launch that returns the launch's own error code, so
// no earlier, unrelated error of the caller is read or cleared.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_plain(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// PDL launch of a kernel in thread-block clusters of `cluster` CTAs along x
// (grid.x a multiple of it). Falls back to a plain cluster launch if the two
// attributes cannot be combined.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster,
                                      cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess) {
        cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, args...);
    }
    return e;
}

// ---- thread-block clusters ---------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster must reach this: it orders the
// shared-memory writes before it with the reads after it, cluster-wide.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The int at the same shared-memory offset as `local` in CTA `rank` of the cluster.
__device__ __forceinline__ int ld_cluster_i32(const int* local, uint32_t rank) {
    const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
    return v;
}

// ---- dtype helpers -------------------------------------------------------------
__device__ __forceinline__ float load_as_f32(const void* p, size_t i, int dtype) {
    if (dtype == MOE_DTYPE_F32) return static_cast<const float*>(p)[i];
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

__device__ __forceinline__ void store_from_f32(void* p, size_t i, float v, int dtype) {
    if (dtype == MOE_DTYPE_F32) static_cast<float*>(p)[i] = v;
    else static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

// 8 consecutive elements as float (16-byte aligned source for bf16, 32 for f32).
template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
        uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};
template <> struct Vec8<float> {
    static __device__ __forceinline__ void load(const float* p, float (&v)[8]) {
        float4 a = reinterpret_cast<const float4*>(p)[0];
        float4 b = reinterpret_cast<const float4*>(p)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    static __device__ __forceinline__ void store(float* p, const float (&v)[8]) {
        reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
};

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Block-wide in-place exclusive scan of data[0..n); returns the total.
// `tmp` holds >= 33 ints. Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(int* data, int n, int* tmp) {
    const int nt = blockDim.x, tid = threadIdx.x;
    const int per = (n + nt - 1) / nt;
    const int b = tid * per, e = min(n, b + per);
    int local = 0;
    for (int i = b; i < e; ++i) local += data[i];
    // inclusive warp scan of the per-thread sums
    const int lane = tid & 31, warp = tid >> 5;
    int v = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
    }
    if (lane == 31) tmp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        const int nw = nt >> 5;
        int w = lane < nw ? tmp[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += u;
        }
        if (lane < nw) tmp[lane] = w;            // inclusive warp totals
        if (lane == 31) tmp[32] = w;             // block total
    }
    __syncthreads();
    int run = v - local + (warp > 0 ? tmp[warp - 1] : 0);
    for (int i = b; i < e; ++i) {
        const int d = data[i];
        data[i] = run;
        run += d;
    }
    const int total = tmp[32];
    __syncthreads();
    return total;
}


}  // namespace moe

// moe_permute_noalloc: the permute for callers that cannot allocate device
// memory -- code that runs while a CUDA graph is being captured into a
// pre-sized memory pool, an embedding runtime whose allocator is off limits
// to libraries, or a real-time path that must never reach cudaMalloc. It
// computes exactly what moe_permute computes, but the per-chunk expert
// histograms that moe_permute keeps in the caller's workspace live in a
// fixed array inside this library instead.
//
// The array is a file-scope static __device__ buffer of
// kNoAllocScratchInts ints (1 MiB). Every GPU that loads the library holds
// one copy of it until the process exits. Host code never names the array
// as an address: on the first call on a device, with that device current,
// cudaGetSymbolAddress gives the device pointer, which is cached per device
// and passed to the kernels.
//
// The permute writes every scratch entry it later reads (the count kernel
// fills the histograms before the scan reads them), so nothing has to be
// cleared between calls. All calls on a device share the one array: two
// calls whose kernels overlap on the GPU (different streams without
// ordering, or concurrent graph launches) race on it and give wrong maps.
#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.h"

namespace {

constexpr size_t kNoAllocScratchInts = 262144;   // 1 MiB

static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
    std::once_flag once;
    int32_t* ptr = nullptr;
};
ScratchSlot g_scratch[kMaxDevices];

// Device pointer of this device's scratch array (set up once per device).
int32_t* scratch_for_current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
    ScratchSlot* s = &g_scratch[d];
    std::call_once(s->once, [s] {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) == cudaSuccess) s->ptr = static_cast<int32_t*>(p);
        else cudaGetLastError();
    });
    return s->ptr;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_permute_noalloc(const int32_t* topk_ids, int M, int top_k, int E,
                                          const int32_t* expert_map, int E_local, const void* x, int K,
                                          int32_t* expert_offsets, int32_t* expanded_idx_to_permuted_idx,
                                          int32_t* permuted_to_expanded, void* x_perm, cudaStream_t stream) {
    if (M < 0 || top_k <= 0 || E < 1 || E_local < 1 || E_local > 1024 || top_k > E) return MOE_ERR_INVALID_ARG;
    if (expert_map == nullptr && E_local != E) return MOE_ERR_INVALID_ARG;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    if (x_perm != nullptr) {
        if (x == nullptr || K <= 0) return MOE_ERR_INVALID_ARG;
        if (K % 8 != 0 || !aligned16(x) || !aligned16(x_perm)) return MOE_ERR_ALIGNMENT;
    }
    if (expert_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (M > 0 && (topk_ids == nullptr || expanded_idx_to_permuted_idx == nullptr ||
                  permuted_to_expanded == nullptr))
        return MOE_ERR_INVALID_ARG;
    // the fixed scratch bounds the problem size
    if (M > 0 && moe::permute_workspace_bytes(M, top_k, E_local) > kNoAllocScratchInts * sizeof(int32_t))
        return MOE_ERR_WORKSPACE;
    moe::DeviceInfo info;
    if (!moe::current_device_info(&info)) return MOE_ERR_CUDA;
    if (info.cc_major != 10 || info.cc_minor != 3) return MOE_ERR_UNSUPPORTED_ARCH;
    int32_t* scratch = scratch_for_current_device();
    if (scratch == nullptr) return MOE_ERR_CUDA;
    if (M == 0) {
        return cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E_local + 1), stream) == cudaSuccess
                   ? MOE_OK : MOE_ERR_CUDA;
    }
    const cudaError_t e = moe::launch_permute(topk_ids, M, top_k, E, expert_map, E_local, x, K, expert_offsets,
                                              expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm, scratch,
                                              moe::device_error_word(), info, stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

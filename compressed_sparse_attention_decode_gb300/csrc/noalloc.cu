// csa2_reindex_noalloc: the Reindex entry point for callers that cannot hand
// the library a workspace.  Some callers cannot call cudaMalloc at all: a
// plug-in running inside a host application that owns and budgets every byte
// of device memory, or a real-time decode loop that must never hit the
// implicit device-wide synchronisation of cudaMalloc / cudaFree.  This variant
// takes its scratch from a fixed array in the library's own device memory
// instead, so the caller only passes inputs and outputs.
//
// The array below is part of the library image: every GPU that loads the
// library holds CSA2_NOALLOC_SCRATCH_BYTES of device memory until the process
// exits, whether or not this entry point is called.
#include <mutex>

#include "common.cuh"

#define CSA2_NOALLOC_SCRATCH_BYTES (8u << 20)

namespace csa2 {
csa2_status check_cache(const csa2_cache* c, bool need_ikey);
size_t reindex_ws(int batch, int n_q, int64_t pool_len);
cudaError_t launch_reindex(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales, const float* iq_raw,
                           const float* w_head, int n_q, int H, const int32_t* pool, int pool_len, int k,
                           int32_t* idx_out, void* ws, cudaStream_t st);
}  // namespace csa2

// Shared by every call on a device; it keeps whatever the last call left in it.
static __device__ __align__(256) unsigned char g_reindex_scratch[CSA2_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in, so
// the kernels must be given this address, never the symbol itself.  The cached
// address belongs to the device's current context: after cudaDeviceReset it
// is stale, so the library must not be used across a device reset.
cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_reindex_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" csa2_status csa2_reindex_noalloc(const csa2_cache* cache, const uint8_t* iq_codes,
                                            const uint8_t* iq_scales, const float* w_head, int32_t n_q,
                                            int32_t n_heads, const int32_t* pool, int32_t pool_len, int32_t k,
                                            int32_t* idx_out, void* stream) {
    using namespace csa2;
    // the same cache checks as csa2_reindex
    const csa2_status cs = check_cache(cache, true);
    if (cs != CSA2_OK) return cs;
    if (n_q < 1 || k < 1 || k > MAX_K || n_heads < 1 || n_heads > MAX_IDX_HEADS || pool_len < 1 ||
        pool_len > 16384)
        return CSA2_ERR_INVALID_ARG;
    if (!iq_codes || !iq_scales || !w_head || !pool || !idx_out || !aligned_to(iq_codes, 4) ||
        !aligned_to(w_head, 4) || !aligned_to(pool, 4) || !aligned_to(idx_out, 4))
        return CSA2_ERR_INVALID_ARG;
    // the request must fit the fixed scratch array
    if (reindex_ws(cache->batch, n_q, pool_len) > CSA2_NOALLOC_SCRATCH_BYTES) return CSA2_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return CSA2_ERR_CUDA;
    // Nothing in the scratch has to start at zero: every byte a Reindex call
    // reads there was written earlier in the same call.
    cudaError_t e = launch_reindex(*cache, iq_codes, iq_scales, nullptr, w_head, n_q, n_heads, pool, pool_len, k, idx_out,
                                   scratch, (cudaStream_t)stream);
    return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

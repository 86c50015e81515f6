// The C ABI of libcsa2: host-side validation, workspace sizing and launches.
// Every check runs before anything is enqueued, so a rejected call leaves the
// stream and all buffers untouched.
#include <cmath>

#include "common.cuh"

namespace csa2 {
cudaError_t launch_cache_write(const csa2_cache& c, const uint16_t* h, int64_t entry0, int n_ent, const float* w0,
                               const float* w1, const uint16_t* ikey_raw, cudaStream_t st);
cudaError_t launch_cache_write_proj(const csa2_cache& c, const uint16_t* h, int64_t entry0, int n_ent, const float* w0,
                                    const float* w1, const uint8_t* wik_codes, const uint8_t* wik_scales,
                                    cudaStream_t st);
cudaError_t launch_quantize_fp4(const float* x, int64_t n_rows, int d, uint8_t* codes, uint8_t* scales,
                                cudaStream_t st);
cudaError_t launch_indexer_full(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                                const float* w_head, int n_q, const int64_t* q_pos, int H, int k, int32_t* idx_out,
                                int pool_blocks, int bs, int32_t* pool_out, void* ws, cudaStream_t st);
cudaError_t launch_reindex(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales, const float* iq_raw,
                           const float* w_head, int n_q, int H, const int32_t* pool, int pool_len, int k,
                           int32_t* idx_out, void* ws, cudaStream_t st);
cudaError_t launch_reuse(const int32_t* prev, int32_t* out, int64_t n, cudaStream_t st);
cudaError_t launch_sparse_attn(const csa2_cache& c, const uint16_t* q, int n_q, int H, const int64_t* q_pos,
                               const int32_t* idx, int k, const uint16_t* swa, int64_t swa_pos0, int swa_len,
                               float scale, float* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t st);
size_t sparse_attn_ws(int batch, int n_q, int H, int k);
size_t indexer_full_ws(int batch, int n_q, int64_t capacity);
size_t reindex_ws(int batch, int n_q, int64_t pool_len);
cudaError_t launch_selftest_wait(uint32_t max_polls, int* err, cudaStream_t st);
}  // namespace csa2

#include <atomic>

namespace csa2 {
static std::atomic<long long> g_launches{0};
void note_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace csa2

using namespace csa2;

namespace {
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

namespace csa2 {
// The cache checks of every entry point (the no-workspace Reindex too).
csa2_status check_cache(const csa2_cache* c, bool need_ikey) {
    if (!c) return CSA2_ERR_INVALID_ARG;
    if (c->batch < 1 || c->capacity < 1) return CSA2_ERR_INVALID_ARG;
    if (c->d_lat != D_LAT) return CSA2_ERR_UNSUPPORTED;
    if (c->d_idx != 64 && c->d_idx != 128) return CSA2_ERR_UNSUPPORTED;
    if (c->ratio != 1 && c->ratio != 2) return CSA2_ERR_INVALID_ARG;
    if (!c->lat_codes || !c->lat_scales || !aligned(c->lat_codes, 16) || !aligned(c->lat_scales, 16))
        return CSA2_ERR_INVALID_ARG;
    // indexer-key scale rows are d_idx/16 bytes: that is all the alignment their loads need
    if (need_ikey && (!c->ikey_codes || !c->ikey_scales || !aligned(c->ikey_codes, 16) ||
                      !aligned(c->ikey_scales, (size_t)(c->d_idx / 16))))
        return CSA2_ERR_INVALID_ARG;
    return CSA2_OK;
}
}  // namespace csa2

namespace {
csa2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

}  // namespace

extern "C" {

int32_t csa2_abi_version(void) { return 200; }

int64_t csa2_launch_count(void) { return (int64_t)g_launches.load(std::memory_order_relaxed); }

const char* csa2_status_string(csa2_status s) {
    switch (s) {
        case CSA2_OK: return "ok";
        case CSA2_ERR_INVALID_ARG: return "invalid argument";
        case CSA2_ERR_UNSUPPORTED: return "unsupported configuration";
        case CSA2_ERR_CUDA: return "CUDA error";
        case CSA2_ERR_WORKSPACE: return "workspace missing or too small";
        case CSA2_ERR_TIMEOUT: return "a kernel gave up on a bounded wait";
    }
    return "unknown status";
}

size_t csa2_workspace_size(int32_t op, int32_t batch, int32_t n_q, int32_t n_heads, int32_t k, int64_t capacity) {
    if (batch < 1 || n_q < 1 || capacity < 0) return 0;
    switch (op) {
        case CSA2_OP_INDEXER_TOPK: return indexer_full_ws(batch, n_q, capacity);
        case CSA2_OP_REINDEX: return reindex_ws(batch, n_q, capacity);
        case CSA2_OP_SPARSE_ATTN: return sparse_attn_ws(batch, n_q, n_heads, k);
    }
    return 0;
}

csa2_status csa2_poll_error(void* workspace, size_t ws_bytes, void* stream) {
    if (!workspace || ws_bytes < 16 || !aligned(workspace, 16)) return CSA2_ERR_INVALID_ARG;
    const cudaStream_t st = (cudaStream_t)stream;
    int word = 0;
    CSA2_CUDA_TRY(cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, st));
    CSA2_CUDA_TRY(cudaStreamSynchronize(st));
    if (word == 0) return CSA2_OK;
    CSA2_CUDA_TRY(cudaMemsetAsync(workspace, 0, sizeof(int), st));
    CSA2_CUDA_TRY(cudaStreamSynchronize(st));
    return CSA2_ERR_TIMEOUT;
}

csa2_status csa2_selftest_wait_timeout(uint32_t max_polls, void* workspace, size_t ws_bytes, void* stream) {
    if (max_polls < 1 || !workspace || ws_bytes < 16 || !aligned(workspace, 16)) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_selftest_wait(max_polls, reinterpret_cast<int*>(workspace), (cudaStream_t)stream));
}

// the checks shared by both cache writes (ratio 2 merges pairs of positions)
static csa2_status check_cache_write(const csa2_cache* cache, const uint16_t* h, int64_t pos0, int32_t n_pos,
                                     const float* w0, const float* w1, bool need_ikey) {
    csa2_status s = check_cache(cache, need_ikey);
    if (s != CSA2_OK) return s;
    if (!h || !aligned(h, 16)) return CSA2_ERR_INVALID_ARG;
    if (pos0 < 0 || n_pos < 0) return CSA2_ERR_INVALID_ARG;
    if (cache->ratio == 2) {
        if (!w0 || !w1 || !aligned(w0, 16) || !aligned(w1, 16)) return CSA2_ERR_INVALID_ARG;
        if ((pos0 & 1) || (n_pos & 1)) return CSA2_ERR_INVALID_ARG;
    }
    if (pos0 / cache->ratio + n_pos / cache->ratio > cache->capacity) return CSA2_ERR_INVALID_ARG;
    return CSA2_OK;
}

csa2_status csa2_cache_write(const csa2_cache* cache, const uint16_t* h, int64_t pos0, int32_t n_pos,
                             const float* w0, const float* w1, const uint16_t* ikey_raw, void* stream) {
    csa2_status s = check_cache_write(cache, h, pos0, n_pos, w0, w1, ikey_raw != nullptr);
    if (s != CSA2_OK) return s;
    if (ikey_raw && !aligned(ikey_raw, 16)) return CSA2_ERR_INVALID_ARG;
    const int r = cache->ratio;
    return from_cuda(launch_cache_write(*cache, h, pos0 / r, n_pos / r, w0, w1, ikey_raw, (cudaStream_t)stream));
}

csa2_status csa2_cache_write_projected(const csa2_cache* cache, const uint16_t* h, int64_t pos0, int32_t n_pos,
                                       const float* w0, const float* w1, const uint8_t* wik_codes,
                                       const uint8_t* wik_scales, void* stream) {
    csa2_status s = check_cache_write(cache, h, pos0, n_pos, w0, w1, true);
    if (s != CSA2_OK) return s;
    if (!wik_codes || !wik_scales || !aligned(wik_codes, 16) || !aligned(wik_scales, 4)) return CSA2_ERR_INVALID_ARG;
    const int r = cache->ratio;
    return from_cuda(launch_cache_write_proj(*cache, h, pos0 / r, n_pos / r, w0, w1, wik_codes, wik_scales,
                                             (cudaStream_t)stream));
}

csa2_status csa2_quantize_fp4(const float* x, int64_t n_rows, int32_t d, uint8_t* codes, uint8_t* scales,
                              void* stream) {
    if (n_rows < 0 || d <= 0 || d % 16) return CSA2_ERR_INVALID_ARG;
    if (n_rows == 0) return CSA2_OK;
    if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 8)) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_quantize_fp4(x, n_rows, d, codes, scales, (cudaStream_t)stream));
}

csa2_status csa2_indexer_topk(const csa2_cache* cache, const uint8_t* iq_codes, const uint8_t* iq_scales,
                              const float* w_head, int32_t n_q, const int64_t* q_pos, int32_t n_heads, int32_t k,
                              int32_t* idx_out, int32_t pool_blocks, int32_t pool_block_size, int32_t* pool_out,
                              void* workspace, size_t ws_bytes, void* stream) {
    csa2_status s = check_cache(cache, true);
    if (s != CSA2_OK) return s;
    if (!iq_codes || !iq_scales || !w_head || !q_pos || !idx_out) return CSA2_ERR_INVALID_ARG;
    if (!aligned(iq_codes, 16) || !aligned(w_head, 4) || !aligned(q_pos, 8) || !aligned(idx_out, 4))
        return CSA2_ERR_INVALID_ARG;
    if (n_q < 1 || n_heads < 1 || n_heads > MAX_IDX_HEADS || k < 1 || k > MAX_K) return CSA2_ERR_INVALID_ARG;
    if (pool_blocks < 0) return CSA2_ERR_INVALID_ARG;
    if (pool_blocks > 0) {
        // pool_block_size 0: the pure pool of the pool_blocks best entries
        if (pool_block_size < 0 || pool_blocks > MAX_K || (int64_t)pool_blocks * pool_block_size > 16384 ||
            !pool_out || !aligned(pool_out, 4))
            return CSA2_ERR_INVALID_ARG;
    }
    size_t need = indexer_full_ws(cache->batch, n_q, cache->capacity);
    if (!workspace || ws_bytes < need || !aligned(workspace, 16)) return CSA2_ERR_WORKSPACE;
    return from_cuda(launch_indexer_full(*cache, iq_codes, iq_scales, w_head, n_q, q_pos, n_heads, k, idx_out,
                                         pool_blocks, pool_block_size, pool_blocks > 0 ? pool_out : nullptr,
                                         workspace, (cudaStream_t)stream));
}

csa2_status csa2_reindex(int32_t mode, const csa2_cache* cache, const uint8_t* iq_codes, const uint8_t* iq_scales,
                         const float* w_head, int32_t n_q, int32_t n_heads, const int32_t* pool, int32_t pool_len,
                         const int32_t* prev_idx, int32_t k, int32_t* idx_out, void* workspace, size_t ws_bytes,
                         void* stream) {
    if (mode != CSA2_REINDEX && mode != CSA2_REUSE) return CSA2_ERR_INVALID_ARG;
    csa2_status s = check_cache(cache, mode == CSA2_REINDEX);
    if (s != CSA2_OK) return s;
    if (n_q < 1 || k < 1 || k > MAX_K || !idx_out || !aligned(idx_out, 4)) return CSA2_ERR_INVALID_ARG;
    if (mode == CSA2_REUSE) {
        if (!prev_idx || !aligned(prev_idx, 4)) return CSA2_ERR_INVALID_ARG;
        return from_cuda(launch_reuse(prev_idx, idx_out, (int64_t)cache->batch * n_q * k, (cudaStream_t)stream));
    }
    if (!iq_codes || !iq_scales || !w_head || !pool || !aligned(iq_codes, 4) || !aligned(w_head, 4) ||
        !aligned(pool, 4))
        return CSA2_ERR_INVALID_ARG;
    if (n_heads < 1 || n_heads > MAX_IDX_HEADS || pool_len < 1 || pool_len > 16384) return CSA2_ERR_INVALID_ARG;
    size_t need = reindex_ws(cache->batch, n_q, pool_len);
    if (!workspace || ws_bytes < need || !aligned(workspace, 16)) return CSA2_ERR_WORKSPACE;
    return from_cuda(launch_reindex(*cache, iq_codes, iq_scales, nullptr, w_head, n_q, n_heads, pool, pool_len, k, idx_out,
                                    workspace, (cudaStream_t)stream));
}

csa2_status csa2_reindex_f32(const csa2_cache* cache, const float* iq, const float* w_head, int32_t n_q,
                             int32_t n_heads, const int32_t* pool, int32_t pool_len, int32_t k, int32_t* idx_out,
                             void* workspace, size_t ws_bytes, void* stream) {
    csa2_status s = check_cache(cache, true);
    if (s != CSA2_OK) return s;
    if (n_q < 1 || k < 1 || k > MAX_K || !idx_out || !aligned(idx_out, 4)) return CSA2_ERR_INVALID_ARG;
    if (!iq || !w_head || !pool || !aligned(iq, 16) || !aligned(w_head, 4) || !aligned(pool, 4))
        return CSA2_ERR_INVALID_ARG;
    if (n_heads < 1 || n_heads > MAX_IDX_HEADS || pool_len < 1 || pool_len > 16384) return CSA2_ERR_INVALID_ARG;
    size_t need = reindex_ws(cache->batch, n_q, pool_len);
    if (!workspace || ws_bytes < need || !aligned(workspace, 16)) return CSA2_ERR_WORKSPACE;
    return from_cuda(launch_reindex(*cache, nullptr, nullptr, iq, w_head, n_q, n_heads, pool, pool_len, k, idx_out,
                                    workspace, (cudaStream_t)stream));
}

csa2_status csa2_sparse_attn(const csa2_cache* cache, const uint16_t* q, int32_t n_q, int32_t n_heads,
                             const int64_t* q_pos, const int32_t* idx, int32_t k, const uint16_t* swa,
                             int64_t swa_pos0, int32_t swa_len, float scale, float* out, float* lse,
                             void* workspace, size_t ws_bytes, void* stream) {
    csa2_status s = check_cache(cache, false);
    if (s != CSA2_OK) return s;
    if (!q || !q_pos || !out || !aligned(q, 16) || !aligned(q_pos, 8) || !aligned(out, 16)) return CSA2_ERR_INVALID_ARG;
    if (n_q < 1 || n_heads < 1 || n_heads > 128 || k < 0 || k > MAX_K || swa_len < 0 || swa_pos0 < 0)
        return CSA2_ERR_INVALID_ARG;
    if (k > 0 && (!idx || !aligned(idx, 4))) return CSA2_ERR_INVALID_ARG;
    if (swa_len > 0 && (!swa || !aligned(swa, 16))) return CSA2_ERR_INVALID_ARG;
    if (lse && !aligned(lse, 4)) return CSA2_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return CSA2_ERR_INVALID_ARG;
    size_t need = sparse_attn_ws(cache->batch, n_q, n_heads, k);
    if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 16))) return CSA2_ERR_WORKSPACE;
    return from_cuda(launch_sparse_attn(*cache, q, n_q, n_heads, q_pos, idx, k, swa, swa_pos0, swa_len, scale, out,
                                        lse, workspace, ws_bytes, (cudaStream_t)stream));
}

}  // extern "C"

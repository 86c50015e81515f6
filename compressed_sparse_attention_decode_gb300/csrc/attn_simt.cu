// Sparse attention over the top-k entries plus the sliding window, CUDA-core
// version ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる", §2.3.1: every
// query attends to its selected entries and to the local SWA KV; §1.1: all
// heads read one shared 512-dim latent, used as key and as value).
//
// One block of 8 warps per (sequence, query, 8 heads); warp = head.  Key rows
// are staged 32 at a time into shared memory as fp32 (FP4 rows dequantised,
// window rows widened from bf16), then every warp runs an online softmax over
// them: lane l owns dims l, l+32, ..., l+480 of the output.  This is the
// simple path kept for shapes the tensor-core kernel does not take.
#include "common.cuh"

namespace csa2 {

constexpr int SIMT_HEADS = 8;
constexpr int SIMT_TILE = 32;

__device__ __forceinline__ void window_range(int64_t p, int64_t swa_pos0, int swa_len, int64_t& lo, int& nwin) {
    lo = p - (WINDOW - 1);
    if (lo < 0) lo = 0;
    if (lo < swa_pos0) lo = swa_pos0;
    int64_t hi = p;
    if (hi > swa_pos0 + swa_len - 1) hi = swa_pos0 + swa_len - 1;
    nwin = hi >= lo ? (int)(hi - lo + 1) : 0;
}

__device__ __forceinline__ float e2m1_to_f32(uint32_t nib) {
    // magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} for codes 0..7, sign in bit 3
    uint32_t m = nib & 7u;
    float mag = (m < 2u) ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1u)) * ((m & 1u) ? 1.5f : 1.0f);
    return (nib & 8u) ? -mag : mag;
}

__global__ void __launch_bounds__(256) k_sparse_attn_simt(
    const uint8_t* __restrict__ lat_codes, const uint8_t* __restrict__ lat_scales, int capacity,
    const uint16_t* __restrict__ q, int n_q, int H, const int64_t* __restrict__ q_pos, const int32_t* __restrict__ idx,
    int k, const uint16_t* __restrict__ swa, int64_t swa_pos0, int swa_len, float scale, float* __restrict__ out,
    float* __restrict__ lse) {
    pdl_wait();
    pdl_launch_next();
    extern __shared__ float sm[];
    float* qs = sm;                                  // [8][512]
    float* tile = qs + SIMT_HEADS * D_LAT;           // [32][512]
    int* rowok = reinterpret_cast<int*>(tile + SIMT_TILE * D_LAT);
    const int b = blockIdx.z, qi = blockIdx.y, h0 = blockIdx.x * SIMT_HEADS;
    const int64_t gq = (int64_t)b * n_q + qi;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < SIMT_HEADS * D_LAT; i += blockDim.x) {
        int hh = h0 + i / D_LAT;
        qs[i] = hh < H ? bf16_bits_to_f32(q[(gq * H + hh) * D_LAT + i % D_LAT]) : 0.0f;
    }
    const int64_t p = q_pos[gq];
    int64_t wlo;
    int nwin;
    window_range(p, swa_pos0, swa_len, wlo, nwin);
    const int n_slots = k + nwin;
    const int32_t* ids = idx + gq * k;

    float m_run = -INFINITY, l_run = 0.0f, o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = 0.0f;

    for (int s0 = 0; s0 < n_slots; s0 += SIMT_TILE) {
        __syncthreads();
        {   // stage 32 rows: thread -> (row, 64-dim part)
            const int r = threadIdx.x >> 3, part = threadIdx.x & 7;
            const int s = s0 + r;
            float* dst = tile + r * D_LAT + part * 64;
            int ok = 0;
            if (s < k) {
                int j = ids[s];
                if (j >= 0 && j < capacity) {
                    ok = 1;
                    const int64_t row = (int64_t)b * capacity + j;
                    const uint4* cp = reinterpret_cast<const uint4*>(lat_codes + row * (D_LAT / 2) + part * 32);
                    uint4 c0 = __ldg(cp), c1 = __ldg(cp + 1);
                    uint32_t sc = __ldg(reinterpret_cast<const uint32_t*>(lat_scales + row * (D_LAT / 16) + part * 4));
                    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        float sv = e4m3_to_f32((sc >> (8 * (w >> 1))) & 255u);
#pragma unroll
                        for (int t = 0; t < 8; ++t) dst[w * 8 + t] = e2m1_to_f32((cw[w] >> (4 * t)) & 15u) * sv;
                    }
                }
            } else if (s < n_slots) {
                ok = 1;
                const int64_t wr = (int64_t)b * swa_len + (wlo + (s - k) - swa_pos0);
                const uint4* wp = reinterpret_cast<const uint4*>(swa + wr * D_LAT + part * 64);
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    uint4 u = __ldg(wp + v);
                    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        dst[v * 8 + 2 * t] = bf16_bits_to_f32(uw[t] & 0xffffu);
                        dst[v * 8 + 2 * t + 1] = bf16_bits_to_f32(uw[t] >> 16);
                    }
                }
            }
            if (part == 0) rowok[r] = ok;
        }
        __syncthreads();
        if (h0 + warp >= H) continue;
        const float* qh = qs + warp * D_LAT;
        for (int r = 0; r < SIMT_TILE; ++r) {
            if (!rowok[r]) continue;
            const float* kr = tile + r * D_LAT;
            float dot = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) dot = fmaf(qh[lane + 32 * i], kr[lane + 32 * i], dot);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const float s = dot * scale;
            if (s > m_run) {
                const float corr = __expf(m_run - s);
                l_run *= corr;
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] *= corr;
                m_run = s;
            }
            const float pexp = __expf(s - m_run);
            l_run += pexp;
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = fmaf(pexp, kr[lane + 32 * i], o[i]);
        }
    }
    if (h0 + warp >= H) return;
    const int hh = h0 + warp;
    const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    float* op = out + (gq * H + hh) * D_LAT;
#pragma unroll
    for (int i = 0; i < 16; ++i) op[lane + 32 * i] = o[i] * inv;
    if (lse != nullptr && lane == 0) lse[gq * H + hh] = l_run > 0.0f ? m_run + logf(l_run) : -INFINITY;
}

cudaError_t launch_sparse_attn_simt(const csa2_cache& c, const uint16_t* q, int n_q, int H, const int64_t* q_pos,
                                    const int32_t* idx, int k, const uint16_t* swa, int64_t swa_pos0, int swa_len,
                                    float scale, float* out, float* lse, cudaStream_t st) {
    const size_t smem = (SIMT_HEADS * D_LAT + SIMT_TILE * D_LAT) * sizeof(float) + SIMT_TILE * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(k_sparse_attn_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((H + SIMT_HEADS - 1) / SIMT_HEADS, n_q, c.batch);
    launch_k(k_sparse_attn_simt, grid, 256, smem, st, c.lat_codes, c.lat_scales, c.capacity, q, n_q, H, q_pos, idx, k, swa,
                                                swa_pos0, swa_len, scale, out, lse);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa2

namespace csa2 {

bool attn_tc_supported(int H);
size_t attn_tc_ws(int batch, int n_q, int H, int k);
cudaError_t launch_sparse_attn_tc(const csa2_cache& c, const uint16_t* q, int n_q, int H, const int64_t* q_pos,
                                  const int32_t* idx, int k, const uint16_t* swa, int64_t swa_pos0, int swa_len,
                                  float scale, float* out, float* lse, void* ws, cudaStream_t st);

bool attn_pair_supported(int H);
size_t attn_pair_ws(int batch, int n_q);
cudaError_t launch_sparse_attn_pair(const csa2_cache& c, const uint16_t* q, int n_q, const int64_t* q_pos,
                                    const int32_t* idx, int k, const uint16_t* swa, int64_t swa_pos0, int swa_len,
                                    float scale, float* out, float* lse, void* ws, cudaStream_t st);

size_t sparse_attn_ws(int batch, int n_q, int H, int k) {
    if (attn_pair_supported(H)) return attn_pair_ws(batch, n_q);
    return attn_tc_supported(H) ? attn_tc_ws(batch, n_q, H, k) : 0;
}

// 64 heads: the CTA-pair tensor-core kernel; other head counts the tensor-core
// tiles take (multiples of 16 up to 64, of 64 up to 128): the per-tile kernel
// with a combine pass; anything else: the CUDA-core kernel
cudaError_t launch_sparse_attn(const csa2_cache& c, const uint16_t* q, int n_q, int H, const int64_t* q_pos,
                               const int32_t* idx, int k, const uint16_t* swa, int64_t swa_pos0, int swa_len,
                               float scale, float* out, float* lse, void* ws, size_t, cudaStream_t st) {
    if (attn_pair_supported(H))
        return launch_sparse_attn_pair(c, q, n_q, q_pos, idx, k, swa, swa_pos0, swa_len, scale, out, lse, ws, st);
    if (attn_tc_supported(H))
        return launch_sparse_attn_tc(c, q, n_q, H, q_pos, idx, k, swa, swa_pos0, swa_len, scale, out, lse, ws, st);
    return launch_sparse_attn_simt(c, q, n_q, H, q_pos, idx, k, swa, swa_pos0, swa_len, scale, out, lse, st);
}

}  // namespace csa2

// Cache write: the encoder's 2:1 channel-wise merge fused with FP4
// quantisation ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる", §1.1
// sequence dimension and §2.3.1 compressor without overlap / position
// embedding), the decoder's one entry per position (§2.3.3), the indexer key
// projected from the entry (§2.3.1), plus the FP4 quantiser used for indexer
// queries.
//
// One warp per entry: lane g owns channels 16g..16g+15, i.e. one FP4 scale
// group, so the merge, the group max, the scale and the 8 code bytes stay in
// registers.  A warp reads 2 KB of bf16 hidden states and writes 256 + 32
// bytes, all coalesced.
#include "common.cuh"

namespace csa2 {

// The 16 latent values of channel group `lane` of entry i (of this call):
// ratio 2 merges raw positions 2i and 2i+1 (e = fmaf(w1, h1, float(w0 * h0))),
// ratio 1 takes raw position i as it is.
__device__ __forceinline__ void entry_latent(const uint16_t* __restrict__ h, int b, int n_ent, int i, int ratio,
                                             const float* __restrict__ w0, const float* __restrict__ w1, int lane,
                                             float* x) {
    const uint16_t* h0 = h + ((int64_t)b * n_ent * ratio + (int64_t)ratio * i) * D_LAT + lane * 16;
    uint4 a0 = __ldg(reinterpret_cast<const uint4*>(h0));
    uint4 a1 = __ldg(reinterpret_cast<const uint4*>(h0) + 1);
    const uint32_t hw0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    if (ratio == 1) {
#pragma unroll
        for (int c = 0; c < 16; ++c) x[c] = bf16_bits_to_f32((c & 1) ? (hw0[c >> 1] >> 16) : (hw0[c >> 1] & 0xffffu));
        return;
    }
    const uint16_t* h1 = h0 + D_LAT;
    uint4 c0 = __ldg(reinterpret_cast<const uint4*>(h1));
    uint4 c1 = __ldg(reinterpret_cast<const uint4*>(h1) + 1);
    const uint32_t hw1[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        float4 p = __ldg(reinterpret_cast<const float4*>(w0 + lane * 16) + v);
        float4 q = __ldg(reinterpret_cast<const float4*>(w1 + lane * 16) + v);
        const float pw[4] = {p.x, p.y, p.z, p.w};
        const float qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            int c = v * 4 + t;
            uint32_t b0 = (c & 1) ? (hw0[c >> 1] >> 16) : (hw0[c >> 1] & 0xffffu);
            uint32_t b1 = (c & 1) ? (hw1[c >> 1] >> 16) : (hw1[c >> 1] & 0xffffu);
            // e = fmaf(w1, h1, float(w0 * h0)): one rounded product, one fused multiply-add
            x[c] = __fmaf_rn(qw[t], bf16_bits_to_f32(b1), __fmul_rn(pw[t], bf16_bits_to_f32(b0)));
        }
    }
}

__global__ void __launch_bounds__(256) k_cache_write(uint8_t* __restrict__ lat_codes, uint8_t* __restrict__ lat_scales,
                                                     uint8_t* __restrict__ ik_codes, uint8_t* __restrict__ ik_scales,
                                                     int capacity, int d_idx, const uint16_t* __restrict__ h,
                                                     int64_t entry0, int n_ent, int ratio, const float* __restrict__ w0,
                                                     const float* __restrict__ w1,
                                                     const uint16_t* __restrict__ ikey_raw) {
    pdl_wait();
    pdl_launch_next();
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int b = blockIdx.y;
    if (i >= n_ent) return;
    const int64_t e = entry0 + i;
    const int64_t row = (int64_t)b * capacity + e;
    float x[16];
    entry_latent(h, b, n_ent, i, ratio, w0, w1, lane, x);
    uint32_t q0, q1, sb;
    quant_group16(x, q0, q1, sb);
    reinterpret_cast<uint2*>(lat_codes + row * (D_LAT / 2))[lane] = make_uint2(q0, q1);
    lat_scales[row * (D_LAT / 16) + lane] = (uint8_t)sb;

    if (ikey_raw != nullptr && lane < d_idx / 16) {
        const uint16_t* kr = ikey_raw + ((int64_t)b * n_ent + i) * d_idx + lane * 16;
        uint4 k0 = __ldg(reinterpret_cast<const uint4*>(kr));
        uint4 k1 = __ldg(reinterpret_cast<const uint4*>(kr) + 1);
        const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int c = 0; c < 16; ++c)
            x[c] = bf16_bits_to_f32((c & 1) ? (kw[c >> 1] >> 16) : (kw[c >> 1] & 0xffffu));
        quant_group16(x, q0, q1, sb);
        reinterpret_cast<uint2*>(ik_codes + row * (d_idx / 2))[lane] = make_uint2(q0, q1);
        ik_scales[row * (d_idx / 16) + lane] = (uint8_t)sb;
    }
}

// E4M3 value times 2^9 (an integer below 2^18: the smallest E4M3 value is 2^-9)
__device__ __forceinline__ int cw_e4m3_x512(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    return e ? (int)((8u + m) << (e - 1u)) : (int)m;
}

// Cache write with the indexer key projected from the entry itself
// ("DeepSeek-v4.1 Flash" §2.3.1: the indexer K is a projection of the main KV
// entry).  Per entry (one warp; lane g owns latent group g): the latent as in
// k_cache_write, then k[d] = sum_c W[d][c] L[c] over the stored (dequantised)
// latent L and the FP4 projection W.  With doubled E2M1 values and 2^9-scaled
// E4M3 scales, a group's term is G4 * SW * SL * 2^-20 with the integer group
// sum G4 (dp4a) and |G4 * SW * SL| < 2^48, so the 32 group terms add up
// exactly in int64 (below 2^53); the sum is rounded once to fp32 and the d_idx
// values are quantised with the same codec (lane q: group q).  W sits in
// shared memory as doubled int8 words, one pad word per row so that the 32
// lanes of a warp (32 rows) hit 32 different banks.
constexpr int CWP_EPW = 8;                     // entries per warp
constexpr int CWP_WS = 129;                    // words per W row in shared memory

template <int DI>
__global__ void __launch_bounds__(256) k_cache_write_proj(uint8_t* __restrict__ lat_codes,
                                                          uint8_t* __restrict__ lat_scales,
                                                          uint8_t* __restrict__ ik_codes,
                                                          uint8_t* __restrict__ ik_scales, int capacity,
                                                          const uint16_t* __restrict__ h, int64_t entry0, int n_ent,
                                                          int ratio, const float* __restrict__ w0,
                                                          const float* __restrict__ w1,
                                                          const uint8_t* __restrict__ wik_codes,
                                                          const uint8_t* __restrict__ wik_scales) {
    pdl_wait();
    pdl_launch_next();
    extern __shared__ int smw[];
    int* Wq = smw;                                   // [DI][CWP_WS] doubled E2M1 values, int8 x4
    int* Ws = Wq + DI * CWP_WS;                      // [DI][33] scales x 2^9 (one pad word per row)
    int* Lq = Ws + DI * 33;                          // per warp: 128 words of the entry's codes, 32 scales
    float* Kf = reinterpret_cast<float*>(Lq + 8 * 160);   // per warp: the DI projected values
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.y;
    for (int i = tid; i < DI * 128; i += 256) {
        const int d = i >> 7, w = i & 127;
        Wq[d * CWP_WS + w] = (int)unpack4_int8(reinterpret_cast<const uint16_t*>(wik_codes + (int64_t)d * (D_LAT / 2))[w]);
    }
    for (int i = tid; i < DI * 32; i += 256) Ws[(i >> 5) * 33 + (i & 31)] = cw_e4m3_x512(wik_scales[i]);
    __syncthreads();
    int* Lw = Lq + warp * 160;
    float* Kw = Kf + warp * DI;
    for (int jj = 0; jj < CWP_EPW; ++jj) {
        const int i = (blockIdx.x * 8 + warp) * CWP_EPW + jj;
        if (i >= n_ent) break;                          // warp-uniform
        const int64_t row = (int64_t)b * capacity + entry0 + i;
        float x[16];
        entry_latent(h, b, n_ent, i, ratio, w0, w1, lane, x);
        uint32_t q0, q1, sb;
        quant_group16(x, q0, q1, sb);
        reinterpret_cast<uint2*>(lat_codes + row * (D_LAT / 2))[lane] = make_uint2(q0, q1);
        lat_scales[row * (D_LAT / 16) + lane] = (uint8_t)sb;
        Lw[4 * lane] = (int)unpack4_int8(q0 & 0xffffu);
        Lw[4 * lane + 1] = (int)unpack4_int8(q0 >> 16);
        Lw[4 * lane + 2] = (int)unpack4_int8(q1 & 0xffffu);
        Lw[4 * lane + 3] = (int)unpack4_int8(q1 >> 16);
        Lw[128 + lane] = cw_e4m3_x512(sb);
        __syncwarp();
#pragma unroll
        for (int t = 0; t < DI / 32; ++t) {
            const int d = lane + 32 * t;
            long long D = 0;
#pragma unroll 8
            for (int g = 0; g < 32; ++g) {
                const int G4 = group_dot4(Wq + d * CWP_WS + 4 * g, reinterpret_cast<const uint32_t*>(Lw + 4 * g));
                D += (long long)(G4 * Ws[d * 33 + g]) * Lw[128 + g];
            }
            Kw[d] = __ll2float_rn(D) * 0x1p-20f;        // one rounding; the power of two is exact
        }
        __syncwarp();
        if (lane < DI / 16) {
            float kx[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) kx[c] = Kw[16 * lane + c];
            quant_group16(kx, q0, q1, sb);
            reinterpret_cast<uint2*>(ik_codes + row * (DI / 2))[lane] = make_uint2(q0, q1);
            ik_scales[row * (DI / 16) + lane] = (uint8_t)sb;
        }
        __syncwarp();
    }
}

// one thread per 16-value group
__global__ void __launch_bounds__(256) k_quantize_fp4(const float* __restrict__ x, int64_t n_groups,
                                                      uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    pdl_wait();
    pdl_launch_next();
    int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n_groups) return;
    float v[16];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        float4 p = __ldg(reinterpret_cast<const float4*>(x + g * 16) + t);
        v[4 * t] = p.x;
        v[4 * t + 1] = p.y;
        v[4 * t + 2] = p.z;
        v[4 * t + 3] = p.w;
    }
    uint32_t q0, q1, sb;
    quant_group16(v, q0, q1, sb);
    reinterpret_cast<uint2*>(codes)[g] = make_uint2(q0, q1);
    scales[g] = (uint8_t)sb;
}

cudaError_t launch_cache_write(const csa2_cache& c, const uint16_t* h, int64_t entry0, int n_ent, const float* w0,
                               const float* w1, const uint16_t* ikey_raw, cudaStream_t st) {
    if (n_ent == 0) return cudaSuccess;
    dim3 grid((n_ent + 7) / 8, c.batch);
    launch_k(k_cache_write, grid, 256, 0, st, c.lat_codes, c.lat_scales, c.ikey_codes, c.ikey_scales, c.capacity, c.d_idx,
                                        h, entry0, n_ent, (int)c.ratio, w0, w1, ikey_raw);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_cache_write_proj(const csa2_cache& c, const uint16_t* h, int64_t entry0, int n_ent, const float* w0,
                                    const float* w1, const uint8_t* wik_codes, const uint8_t* wik_scales,
                                    cudaStream_t st) {
    if (n_ent == 0) return cudaSuccess;
    dim3 grid((n_ent + 8 * CWP_EPW - 1) / (8 * CWP_EPW), c.batch);
    auto kern = c.d_idx == 128 ? k_cache_write_proj<128> : k_cache_write_proj<64>;
    const size_t smem = ((size_t)c.d_idx * (CWP_WS + 33) + 8 * 160 + 8 * c.d_idx) * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    launch_k(kern, grid, 256, smem, st, c.lat_codes, c.lat_scales, c.ikey_codes, c.ikey_scales, c.capacity, h, entry0,
             n_ent, (int)c.ratio, w0, w1, wik_codes, wik_scales);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp4(const float* x, int64_t n_rows, int d, uint8_t* codes, uint8_t* scales,
                                cudaStream_t st) {
    int64_t n_groups = n_rows * (d / 16);
    if (n_groups == 0) return cudaSuccess;
    launch_k(k_quantize_fp4, (unsigned)((n_groups + 255) / 256), 256, 0, st, x, n_groups, codes, scales);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa2

// Cache write: the encoder's 2:1 channel-wise merge fused with FP4
// quantisation ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる", §1.1
// sequence dimension and §2.3.1 compressor without overlap / position
// embedding), plus the FP4 quantiser used for indexer queries.
//
// One warp per entry: lane g owns channels 16g..16g+15, i.e. one FP4 scale
// group, so the merge, the group max, the scale and the 8 code bytes stay in
// registers.  A warp reads 2 KB of bf16 hidden states and writes 256 + 32
// bytes, all coalesced.
#include "common.cuh"

namespace csa2 {

__global__ void __launch_bounds__(256) k_cache_write(uint8_t* __restrict__ lat_codes, uint8_t* __restrict__ lat_scales,
                                                     uint8_t* __restrict__ ik_codes, uint8_t* __restrict__ ik_scales,
                                                     int capacity, int d_idx, const uint16_t* __restrict__ h,
                                                     int64_t entry0, int n_ent, const float* __restrict__ w0,
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

    const uint16_t* h0 = h + ((int64_t)b * n_ent * 2 + 2 * (int64_t)i) * D_LAT + lane * 16;
    const uint16_t* h1 = h0 + D_LAT;
    uint4 a0 = __ldg(reinterpret_cast<const uint4*>(h0));
    uint4 a1 = __ldg(reinterpret_cast<const uint4*>(h0) + 1);
    uint4 c0 = __ldg(reinterpret_cast<const uint4*>(h1));
    uint4 c1 = __ldg(reinterpret_cast<const uint4*>(h1) + 1);
    const uint32_t hw0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t hw1[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    float x[16];
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
                                        h, entry0, n_ent, w0, w1, ikey_raw);
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

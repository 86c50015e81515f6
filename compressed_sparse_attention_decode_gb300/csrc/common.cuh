// Shared device helpers of the CUDA path (FP4/E4M3 codec, key orderings,
// exact indexer group sums).  Nothing here is shared with the CPU oracle.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp8.h>

#include "../../include/csa2.h"

namespace csa2 {

// ---------------------------------------------------------------- launches
// Every kernel of the library is launched with programmatic stream
// serialisation: a kernel waits at its top until its predecessor has completed
// and that grid's memory is visible, then lets its own successor be scheduled,
// so a successor overlaps only its immediate predecessor (and may do work that
// needs nothing the stream produced before it waits).  Outside such a launch
// both instructions do nothing.
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// (d0, d1) = (a0 b0 + d0, a1 b1 + d1), each rounded once as by fmaf, in one packed instruction
__device__ __forceinline__ void fma2_rn(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rd, {%0, %1};\n"
        " fma.rn.f32x2 rd, ra, rb, rd;\n mov.b64 {%0, %1}, rd;\n}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// square root, approximate: callers leave room for its error (far below 2^-20 relative)
__device__ __forceinline__ float sqrt_approx(float x) {
    float y;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr int D_LAT = 512;
constexpr int WINDOW = 128;
constexpr int MAX_K = 2048;
constexpr int MAX_IDX_HEADS = 32;

// ---------------------------------------------------------------- formats

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// E4M3 byte -> float: exponent 0 is subnormal m * 2^-9, else (8+m) * 2^(e-10).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0x1p-9f;
    return (b & 0x80u) ? -mag : mag;
}

// float >= 0 -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float v) {
    return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// E2M1 code of x for scale s > 0, by comparing |x| with the exact midpoints
// t*s (t has at most 3 significant bits and s at most 4, so t*s is exact in
// fp32).  Strict / non-strict comparisons put every tie on the even code.
__device__ __forceinline__ uint32_t e2m1_code(float x, float s) {
    float a = fabsf(x);
    uint32_t m = (a > 0.25f * s) + (a >= 0.75f * s) + (a > 1.25f * s) + (a >= 1.75f * s) +
                 (a > 2.5f * s) + (a >= 3.5f * s) + (a > 5.0f * s);
    return m | ((x < 0.0f && m) ? 8u : 0u);
}

// Quantise 16 floats: scale byte = E4M3(amax/6) (IEEE division), two words of
// packed codes (element 2i in the low nibble of byte i).
__device__ __forceinline__ void quant_group16(const float* x, uint32_t& w0, uint32_t& w1, uint32_t& sbyte) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    sbyte = f32_to_e4m3_satfinite(__fdiv_rn(amax, 6.0f));
    float s = e4m3_to_f32(sbyte);
    w0 = 0u;
    w1 = 0u;
    if (s > 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) w0 |= e2m1_code(x[i], s) << (4 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i) w1 |= e2m1_code(x[8 + i], s) << (4 * i);
    }
}

// ---------------------------------------------------------------- orderings

// order-preserving maps float -> uint (larger float -> larger uint); -0 == +0
__device__ __forceinline__ uint32_t f32_key(float f) {
    uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ unsigned long long f64_key(double f) {
    unsigned long long u = (unsigned long long)__double_as_longlong(f + 0.0);
    return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// ---------------------------------------------------------------- indexer group sums

// Split 4 E2M1 codes (16 bits, code i in nibble i) into two words of int8
// magnitudes times two, one word for the positive codes and one for the
// negative ones (zeros elsewhere).  prmt's default mode selects byte
// (nibble & 7) of the table {0,1,2,3,4,6,8,12} and, when the nibble's bit 3
// is set, replaces it by its sign (0x00 for these non-negative bytes).
__device__ __forceinline__ void unpack4_signed(uint32_t nib16, uint32_t& pos, uint32_t& neg) {
    const uint32_t lo = 0x03020100u, hi = 0x0C080604u;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(pos) : "r"(lo), "r"(hi), "r"(nib16));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(neg) : "r"(lo), "r"(hi), "r"(nib16 ^ 0x8888u));
}

// 4 * (sum over a 16-group of q_i * k_i) for E2M1 values, exact in int32:
// q and k as doubled values in signed int8 x4 words (|.| <= 12)
__device__ __forceinline__ int group_dot4(const int* q, const uint32_t* k) {
    int acc = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) acc = __dp4a(q[w], (int)k[w], acc);
    return acc;
}

// four E2M1 codes (16 bits) -> their doubled values as signed int8 x4
__device__ __forceinline__ uint32_t unpack4_int8(uint32_t nib16) {
    uint32_t p, n;
    unpack4_signed(nib16, p, n);
    return __vsub4(p, n);
}

// process-wide count of kernel launches enqueued by the library
void note_launch(int n = 1);

}  // namespace csa2

#define CSA2_CUDA_TRY(expr)                                   \
    do {                                                      \
        cudaError_t _e = (expr);                              \
        if (_e != cudaSuccess) return CSA2_ERR_CUDA;          \
    } while (0)

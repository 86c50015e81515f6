// Sparse attention on the tensor cores (tcgen05, TMEM accumulators)
// ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる", §2.3.1: each query
// attends to its top-k entries and its local window; §1.1: one shared 512-dim
// latent is both key and value for every head, i.e. MQA).
//
// One CTA per (query, 128-key tile, group of <= 64 heads):
//   L  [128 keys x 512] fp16 in shared memory (FP4 rows dequantised exactly:
//      E2M1 x E4M3 has at most 7 significant bits and lies in [2^-10, 2688];
//      window rows converted from bf16), 128B-swizzled K-major slabs of 64 dims
//   Q  [heads x 512] fp16, same layout
//   S^T = L . Q^T            M = 128 keys, N = heads, K = 512   (TMEM)
//   P   = exp2(S^T*c - m_h)  per-head column max over the tile  (fp16, smem)
//   O^T = L^T . P            M = 4 x 128 dims, N = heads, K = 128 keys: L read
//                            through an MN-major descriptor, no copy
//   l   = 1^T . P            column sums from the same rounded P
// Keys sit on the MMA's M side so every MMA is a full M = 128 one even though
// there are only 64 heads.  The per-tile (m, l, O) partials are merged by
// k_attn_combine.
#include "common.cuh"
#include "umma.cuh"

namespace csa2 {

constexpr int TC_TILE = 128;
constexpr int TC_HG = 64;
constexpr int TC_THREADS = 256;
constexpr uint32_t SM_Q = 0;                         // 8 slabs x HG x 128 B   (<= 64 KB)
constexpr uint32_t SM_L = 64 * 1024;                 // 8 slabs x 128 x 128 B (128 KB)
constexpr uint32_t SM_P = SM_L + 128 * 1024;         // 128 x 128 B            (16 KB)
constexpr uint32_t SM_ONES = SM_P + 16 * 1024;       // 128 x 16 fp16 ones     (4 KB)
constexpr uint32_t SM_RED = SM_ONES + 4 * 1024;      // 4 warps x 64 floats    (1 KB)
constexpr uint32_t SM_DYN = SM_RED + 1024 + 1024;    // + slack for 1024-B alignment
constexpr uint32_t SLAB_L = TC_TILE * 128;           // bytes per 64-dim slab of L
// MN-major views: stride between 64-wide MN atoms / between 8-row K groups
constexpr uint32_t MN_A_LBO = SLAB_L, MN_A_SBO = 1024;
constexpr uint32_t MN_B_LBO = 8192, MN_B_SBO = 1024;
// TMEM columns
constexpr uint32_t TM_S = 0, TM_O = 64, TM_L = 320, TM_COLS = 512;
constexpr int ATTN_QCHUNK = 256;

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 8 E2M1 codes (one word, code i in nibble i) -> 4 f16x2 words, value order kept
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t* o) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, __half2 s) {
    __half2 x = *reinterpret_cast<__half2*>(&a);
    x = __hmul2(x, s);
    return *reinterpret_cast<uint32_t*>(&x);
}

__device__ __forceinline__ uint32_t f32_order(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float f32_unorder(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int HG>
__global__ void __launch_bounds__(TC_THREADS, 1) k_sparse_attn_tc(
    const uint8_t* __restrict__ lat_codes, const uint8_t* __restrict__ lat_scales, int capacity,
    const uint16_t* __restrict__ q, int n_q, int q0, int H, const int64_t* __restrict__ q_pos,
    const int32_t* __restrict__ idx, int k, const uint16_t* __restrict__ swa, int64_t swa_pos0, int swa_len,
    float scale_log2e, int n_tiles, float* __restrict__ part_o, float2* __restrict__ part_ml, int* __restrict__ err) {
    pdl_wait();
    pdl_launch_next();
    extern __shared__ uint8_t dyn[];
    __shared__ __align__(8) unsigned long long mbar;
    __shared__ uint32_t tmem_base;
    __shared__ int rowok[TC_TILE];

    const uint32_t raw = umma::smem_u32(dyn);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = dyn + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x % n_tiles, hg = blockIdx.x / n_tiles;
    const int qi = q0 + blockIdx.y, b = blockIdx.z;
    const int nqc = gridDim.y;
    const int64_t gq = (int64_t)b * n_q + qi;
    const uint32_t mb = umma::smem_u32(&mbar);

    if (tid == 0) {
        umma::mbar_init(mb, 1);
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(umma::smem_u32(&tmem_base), TM_COLS);

    // ---- Q: heads hg*HG .. +HG, bf16 -> fp16, swizzled K-major.  All of a
    // thread's loads are issued before any conversion, so the CTA pays one
    // memory round trip for Q rather than one per chunk.
    {
        constexpr int QCH = HG * 64 / TC_THREADS;           // 16-byte chunks per thread
        uint4 qv[QCH];
#pragma unroll
        for (int u = 0; u < QCH; ++u) {
            const int i = tid + u * TC_THREADS, h = i >> 6, c = i & 63;
            qv[u] = __ldg(reinterpret_cast<const uint4*>(q + ((gq * H + hg * HG + h) * D_LAT + c * 8)));
        }
#pragma unroll
        for (int u = 0; u < QCH; ++u) {
            const int i = tid + u * TC_THREADS, h = i >> 6, c = i & 63;
            const uint4 v = qv[u];
            uint4 o = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
            *reinterpret_cast<uint4*>(sm + SM_Q + (c >> 3) * (HG * 128) + swz(h, c & 7)) = o;
        }
    }
    // ---- ones (fp16 1.0) for the column sums
    reinterpret_cast<uint4*>(sm + SM_ONES)[tid] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);

    // ---- L tile: thread -> (row r, half of the 512 dims)
    {
        const int r = tid & 127, half = tid >> 7;
        const int slot = tile * TC_TILE + r;
        const int64_t p = q_pos[gq];
        int64_t wlo = p - (WINDOW - 1);
        if (wlo < 0) wlo = 0;
        if (wlo < swa_pos0) wlo = swa_pos0;
        int64_t whi = p;
        if (whi > swa_pos0 + swa_len - 1) whi = swa_pos0 + swa_len - 1;
        const int nwin = whi >= wlo ? (int)(whi - wlo + 1) : 0;
        int kind = 0;  // 0 empty, 1 FP4 entry, 2 window row
        int64_t row = 0;
        if (slot < k) {
            int j = idx[gq * k + slot];
            if (j >= 0 && j < capacity) {
                kind = 1;
                row = (int64_t)b * capacity + j;
            }
        } else if (slot < k + nwin) {
            kind = 2;
            row = (int64_t)b * swa_len + (wlo + (slot - k) - swa_pos0);
        }
        uint8_t* dst = sm + SM_L;
        if (kind == 1) {
            const uint4* cp = reinterpret_cast<const uint4*>(lat_codes + row * (D_LAT / 2) + half * 128);
            uint4 sc = __ldg(reinterpret_cast<const uint4*>(lat_scales + row * (D_LAT / 16) + half * 16));
            uint4 cw[8];
#pragma unroll
            for (int v = 0; v < 8; ++v) cw[v] = __ldg(cp + v);
            const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
            for (int v = 0; v < 8; ++v) {           // 32 dims = 2 scale groups
                const uint32_t words[4] = {cw[v].x, cw[v].y, cw[v].z, cw[v].w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {       // 8 dims = one 16-byte chunk
                    const int g = 2 * v + (t >> 1);  // scale group within this half
                    const float sf = e4m3_to_f32((sw[g >> 2] >> (8 * (g & 3))) & 255u);
                    const __half2 s2 = __float2half2_rn(sf);
                    uint32_t f[4];
                    e2m1x8_to_f16(words[t], f);
                    uint4 o = make_uint4(hmul2_u32(f[0], s2), hmul2_u32(f[1], s2), hmul2_u32(f[2], s2),
                                         hmul2_u32(f[3], s2));
                    const int c = half * 32 + v * 4 + t;     // 8-dim chunk index 0..63
                    *reinterpret_cast<uint4*>(dst + (c >> 3) * SLAB_L + swz(r, c & 7)) = o;
                }
            }
        } else if (kind == 2) {
            const uint4* wp = reinterpret_cast<const uint4*>(swa + row * D_LAT + half * 256);
#pragma unroll
            for (int part = 0; part < 2; ++part) {          // two batches of 16 loads
                uint4 wv[16];
#pragma unroll
                for (int v = 0; v < 16; ++v) wv[v] = __ldg(wp + part * 16 + v);
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    const uint4 u = wv[v];
                    uint4 o = make_uint4(bf16x2_to_f16x2(u.x), bf16x2_to_f16x2(u.y), bf16x2_to_f16x2(u.z),
                                         bf16x2_to_f16x2(u.w));
                    const int c = half * 32 + part * 16 + v;
                    *reinterpret_cast<uint4*>(dst + (c >> 3) * SLAB_L + swz(r, c & 7)) = o;
                }
            }
        } else {
#pragma unroll 8
            for (int v = 0; v < 32; ++v) {
                const int c = half * 32 + v;
                *reinterpret_cast<uint4*>(dst + (c >> 3) * SLAB_L + swz(r, c & 7)) = make_uint4(0, 0, 0, 0);
            }
        }
        if (half == 0) rowok[r] = kind != 0;
    }
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = tmem_base;
    if (warp >= 4) return;           // loaders are done; warps 0-3 own the TMEM lanes

    // ---- S^T = L . Q^T
    if (tid == 0) {
        const uint32_t id1 = umma::idesc_f16(128, HG, 0, 0);
#pragma unroll 4
        for (int ks = 0; ks < 32; ++ks) {
            uint64_t a = umma::desc(base + SM_L + (ks >> 2) * SLAB_L + (ks & 3) * 32, 16, 1024, umma::LAYOUT_SW128);
            uint64_t bq = umma::desc(base + SM_Q + (ks >> 2) * (HG * 128) + (ks & 3) * 32, 16, 1024,
                                     umma::LAYOUT_SW128);
            umma::mma_f16(tmem + TM_S, a, bq, id1, ks > 0);
        }
        umma::commit(mb);
    }
    bool ok = umma::mbar_wait(mb, 0);
    umma::fence_after();
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float* red = reinterpret_cast<float*>(sm + SM_RED);
    float x[TC_HG];
    const bool valid = rowok[tid] != 0;
    for (int c = 0; c < HG; c += 16) umma::tmem_ld16(lane_base + TM_S + c, x + c);
    umma::tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < TC_HG; ++h) {
        if (h < HG) {
            x[h] = valid ? x[h] * scale_log2e : -INFINITY;
            uint32_t mk = __reduce_max_sync(0xffffffffu, f32_order(x[h]));
            if (lane == 0) red[warp * TC_HG + h] = f32_unorder(mk);
        }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    // ---- P = exp2(x - m) as fp16, rows = keys (MN-major B operand of the second GEMM)
    uint32_t prow[TC_HG / 2];
#pragma unroll
    for (int h = 0; h < TC_HG; h += 2) {
        if (h < HG) {
            float m0 = fmaxf(fmaxf(red[h], red[TC_HG + h]), fmaxf(red[2 * TC_HG + h], red[3 * TC_HG + h]));
            float m1 = fmaxf(fmaxf(red[h + 1], red[TC_HG + h + 1]), fmaxf(red[2 * TC_HG + h + 1], red[3 * TC_HG + h + 1]));
            float p0 = (m0 == -INFINITY) ? 0.0f : umma::ex2(x[h] - m0);
            float p1 = (m1 == -INFINITY) ? 0.0f : umma::ex2(x[h + 1] - m1);
            __half2 hp = __floats2half2_rn(p0, p1);
            prow[h / 2] = *reinterpret_cast<uint32_t*>(&hp);
        }
    }
    for (int c = 0; c < HG / 8; ++c)
        *reinterpret_cast<uint4*>(sm + SM_P + swz(tid, c)) =
            make_uint4(prow[4 * c], prow[4 * c + 1], prow[4 * c + 2], prow[4 * c + 3]);
    const int64_t slab_id = (((int64_t)b * nqc + blockIdx.y) * n_tiles + tile);
    if (tid < HG) {
        float m = fmaxf(fmaxf(red[tid], red[TC_HG + tid]), fmaxf(red[2 * TC_HG + tid], red[3 * TC_HG + tid]));
        part_ml[slab_id * H + hg * HG + tid].x = m;
    }
    umma::fence_proxy_async();
    umma::fence_before();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    umma::fence_after();

    // ---- O^T = L^T . P (4 M-tiles of 128 dims) and l = 1^T . P
    if (tid == 0) {
        const uint32_t id2 = umma::idesc_f16(128, HG, 1, 1);
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint64_t a = umma::desc(base + SM_L + (2 * mt) * SLAB_L + ks * 2048, MN_A_LBO, MN_A_SBO,
                                        umma::LAYOUT_SW128);
                uint64_t bp = umma::desc(base + SM_P + ks * 2048, MN_B_LBO, MN_B_SBO, umma::LAYOUT_SW128);
                umma::mma_f16(tmem + TM_O + 64 * mt, a, bp, id2, ks > 0);
            }
        }
        const uint32_t id3 = umma::idesc_f16(128, HG, 0, 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint64_t a = umma::desc(base + SM_ONES, 128, 256, umma::LAYOUT_NONE);
            uint64_t bp = umma::desc(base + SM_P + ks * 2048, MN_B_LBO, MN_B_SBO, umma::LAYOUT_SW128);
            umma::mma_f16(tmem + TM_L, a, bp, id3, ks > 0);
        }
        umma::commit(mb);
    }
    ok = umma::mbar_wait(mb, 1) && ok;
    umma::fence_after();
    if (!ok && tid == 0) atomicExch(err, 1);

    // ---- epilogue: partial O (unnormalised, relative to m), l
    float* po = part_o + slab_id * (int64_t)H * D_LAT;
    for (int mt = 0; mt < 4; ++mt) {
        float o[TC_HG];
        for (int c = 0; c < HG; c += 16) umma::tmem_ld16(lane_base + TM_O + 64 * mt + c, o + c);
        umma::tmem_wait_ld();
        const int d = mt * 128 + tid;
#pragma unroll
        for (int h = 0; h < TC_HG; ++h)
            if (h < HG) po[(int64_t)(hg * HG + h) * D_LAT + d] = ok ? o[h] : __int_as_float(0x7fc00000);
    }
    if (warp == 0) {
        float l[TC_HG];
        for (int c = 0; c < HG; c += 16) umma::tmem_ld16(lane_base + TM_L + c, l + c);
        umma::tmem_wait_ld();
        if (lane == 0)
            for (int h = 0; h < HG; ++h) part_ml[slab_id * H + hg * HG + h].y = l[h];
    }
    umma::fence_before();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (warp == 0) {
        umma::fence_after();
        umma::tmem_dealloc(tmem, TM_COLS);
    }
}

// merge the per-tile partials of one (query, head): m in log2 units
__global__ void __launch_bounds__(128) k_attn_combine(const float* __restrict__ part_o,
                                                      const float2* __restrict__ part_ml, int n_q, int q0, int H,
                                                      int n_tiles, float* __restrict__ out, float* __restrict__ lse) {
    pdl_wait();
    pdl_launch_next();
    const int h = blockIdx.x, ql = blockIdx.y, b = blockIdx.z;
    const int nqc = gridDim.y;
    const int64_t s0 = ((int64_t)b * nqc + ql) * n_tiles;
    float M = -INFINITY;
    for (int t = 0; t < n_tiles; ++t) M = fmaxf(M, part_ml[(s0 + t) * H + h].x);
    float L = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t = 0; t < n_tiles; ++t) {
        float2 ml = part_ml[(s0 + t) * H + h];
        if (ml.x == -INFINITY) continue;
        float w = umma::ex2(ml.x - M);
        L += w * ml.y;
        float4 v = reinterpret_cast<const float4*>(part_o + ((s0 + t) * H + h) * D_LAT)[threadIdx.x];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    const int64_t gq = (int64_t)b * n_q + q0 + ql;
    reinterpret_cast<float4*>(out + (gq * H + h) * D_LAT)[threadIdx.x] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (lse != nullptr && threadIdx.x == 0)
        lse[gq * H + h] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

bool attn_tc_supported(int H) { return H == 16 || H == 32 || H == 48 || H == 64 || (H > 64 && H % 64 == 0 && H <= 128); }

static int n_tiles_of(int k) { return (k + WINDOW + TC_TILE - 1) / TC_TILE; }

size_t attn_tc_ws(int batch, int n_q, int H, int k) {
    const int qc = n_q < ATTN_QCHUNK ? n_q : ATTN_QCHUNK;
    const size_t slabs = (size_t)batch * qc * n_tiles_of(k);
    return 256 + slabs * H * (D_LAT * sizeof(float) + sizeof(float2));
}

cudaError_t launch_sparse_attn_tc(const csa2_cache& c, const uint16_t* q, int n_q, int H, const int64_t* q_pos,
                                  const int32_t* idx, int k, const uint16_t* swa, int64_t swa_pos0, int swa_len,
                                  float scale, float* out, float* lse, void* ws, cudaStream_t st) {
    const int HG = H <= TC_HG ? H : TC_HG;
    const int n_tiles = n_tiles_of(k);
    const int qc = n_q < ATTN_QCHUNK ? n_q : ATTN_QCHUNK;
    int* err = reinterpret_cast<int*>(ws);
    float2* part_ml = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(ws) + 256);
    float* part_o = reinterpret_cast<float*>(part_ml + (size_t)c.batch * qc * n_tiles * H);
    auto kern = HG == 64 ? k_sparse_attn_tc<64> : (HG == 32 ? k_sparse_attn_tc<32> : (HG == 48 ? k_sparse_attn_tc<48> : k_sparse_attn_tc<16>));
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM_DYN);
    if (e != cudaSuccess) return e;
    const float scale_log2e = scale * 1.4426950408889634f;
    for (int q0 = 0; q0 < n_q; q0 += qc) {
        const int nqc = (n_q - q0) < qc ? (n_q - q0) : qc;
        dim3 g1(n_tiles * (H / HG), nqc, c.batch);
        launch_k(kern, g1, TC_THREADS, SM_DYN, st, c.lat_codes, c.lat_scales, c.capacity, q, n_q, q0, H, q_pos, idx, k,
                                             swa, swa_pos0, swa_len, scale_log2e, n_tiles, part_o, part_ml, err);
        note_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        dim3 g2(H, nqc, c.batch);
        launch_k(k_attn_combine, g2, 128, 0, st, part_o, part_ml, n_q, q0, H, n_tiles, out, lse);
        note_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace csa2

// Sparse attention, 64 heads, one CTA pair (thread-block cluster of 2) per
// query ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる", §2.3.1 top-k
// entries plus the local window; §1.1 one 512-dim latent shared by every head).
//
// CTA r of the pair owns latent dims [256r, 256r+256).  Per 128-key tile:
//   S_r = L[:, dims_r] . Q[:, dims_r]^T   (tcgen05, M = 128 keys, N = 64 heads,
//                                          K = 256, fp32 in TMEM)
//   each CTA sends its partial scores to the other with asynchronous remote
//   stores counted on the receiver's mbarrier, and adds the other's
//   (S = S_0 + S_1, the same bits in both CTAs); an online softmax with a lazy
//   running max (a max reduction runs only when some score rises more than 2^8
//   above the running max) writes P (fp16), and both CTAs accumulate their own
//   output dims: O_r^T += L[:, dims_r]^T . P, l += 1^T . P (TMEM, across all
//   tiles).  One thread per CTA waits on the barriers the peer fills (cluster
//   scope) and passes them on through a named barrier of the softmax warps.
// The query's top-k indices are staged in shared memory at the start and every
// row the CTA will read is prefetched into L2, so the tile gathers that follow
// (double-buffered, overlapping the MMAs and softmax) are single L2 round trips.
//
// Warps: 0-7 softmax / epilogue (warp w reads TMEM lanes 32(w%4).. = key rows,
// later output dims, for heads 32(w/4)..+31), warp 8 issues the MMAs, warps
// 9-15 gather rows.  Tiles 0.. hold the selected FP4 entries, the last tile the
// window rows (bf16).
#include "common.cuh"
#include "umma.cuh"

namespace csa2 {

constexpr int AP_TILE = 128;
constexpr int AP_H = 64;
constexpr int AP_THREADS = 512;
constexpr int AP_SMW = 8;                            // softmax warps 0-7: lane quadrant x head half
constexpr int AP_SMT = AP_SMW * 32;
constexpr int AP_MMAW = 8;                           // warp 8 issues the MMAs
constexpr int AP_LOADERS = 224;                      // warps 9-15
constexpr uint32_t AP_SLAB = AP_TILE * 128;          // 64 dims x 128 keys x fp16
constexpr uint32_t AP_SQ = 0;                        // Q half: 4 slabs x 64 heads x 128 B = 32 KB
constexpr uint32_t AP_SL = 32 * 1024;                // 2 buffers x 4 slabs (128 KB)
constexpr uint32_t AP_LBUF = 4 * AP_SLAB;
constexpr uint32_t AP_SP = AP_SL + 2 * AP_LBUF;      // P: 128 keys x 64 heads fp16 (16 KB)
constexpr uint32_t AP_SONES = AP_SP + 16 * 1024;     // ones, 128 x 16 fp16 (4 KB)
constexpr uint32_t AP_SX = AP_SONES + 4 * 1024;      // the peer's partial scores, 128 x 64 f32 (32 KB)
constexpr uint32_t AP_SIDX = AP_SX + 32 * 1024;      // the query's indices, MAX_K ints
constexpr uint32_t AP_RED = AP_SIDX + MAX_K * 4;     // column maxima / row sums, 4 quadrants x 64
constexpr uint32_t AP_MISC = AP_RED + 1024;          // m_run[64], fac[64], flags
constexpr uint32_t AP_DYN = AP_MISC + 1024 + 1024;
constexpr uint32_t AP_XBYTES = AP_TILE * AP_H * 4;   // partial scores one CTA sends per tile
constexpr uint32_t APT_S = 0, APT_O = 128, APT_L = 256, APT_COLS = 512;
constexpr float AP_LAZY = 8.0f;                      // log2 headroom before the running max is raised

__device__ __forceinline__ uint32_t apswz(uint32_t row, uint32_t chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

__device__ __forceinline__ uint32_t ap_bf16x2_to_f16x2(uint32_t v) {
    __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void ap_e2m1x8(uint32_t w, uint32_t* o) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}
// two E4M3 bytes (low byte -> low half) to fp16x2, exactly
__device__ __forceinline__ __half2 ap_e4m3x2(uint32_t two) {
    uint32_t r;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(r) : "r"(two));
    return *reinterpret_cast<__half2*>(&r);
}
__device__ __forceinline__ uint32_t ap_hmul2(uint32_t a, __half2 s) {
    __half2 x = __hmul2(*reinterpret_cast<__half2*>(&a), s);
    return *reinterpret_cast<uint32_t*>(&x);
}
__device__ __forceinline__ uint32_t ap_ord(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ap_unord(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(AP_THREADS, 1) k_sparse_attn_pair(
    const uint8_t* __restrict__ lat_codes, const uint8_t* __restrict__ lat_scales, int capacity,
    const uint16_t* __restrict__ q, int n_q, int q0, const int64_t* __restrict__ q_pos,
    const int32_t* __restrict__ idx, int k, const uint16_t* __restrict__ swa, int64_t swa_pos0, int swa_len,
    float scale_log2e, float* __restrict__ out, float* __restrict__ lse, int* __restrict__ err) {
    extern __shared__ uint8_t dyn[];
    __shared__ __align__(8) unsigned long long b_lfull[2], b_lfree[2], b_sfull[2], b_sfree[2], b_pfull, b_odone, b_xfull,
        b_xfree;
    __shared__ uint32_t tmem_base;
    __shared__ int rowok[2][AP_TILE];

    const uint32_t raw = umma::smem_u32(dyn);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = dyn + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = umma::cluster_rank();
    const uint32_t peer = rank ^ 1u;
    const int d0 = (int)rank * 256;
    const int qi = q0 + blockIdx.y, b = blockIdx.z;
    const int64_t gq = (int64_t)b * n_q + qi;

    // window of this query (clipped to the rows present) and tile count
    const int64_t p = q_pos[gq];
    int64_t wlo = p - (WINDOW - 1);
    if (wlo < 0) wlo = 0;
    if (wlo < swa_pos0) wlo = swa_pos0;
    int64_t whi = p;
    if (whi > swa_pos0 + swa_len - 1) whi = swa_pos0 + swa_len - 1;
    const int nwin = whi >= wlo ? (int)(whi - wlo + 1) : 0;
    const int T = 1 + (k + AP_TILE - 1) / AP_TILE;

    auto sa = [&](const void* x) { return umma::smem_u32(x); };
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            umma::mbar_init(sa(&b_lfull[i]), AP_LOADERS);
            umma::mbar_init(sa(&b_lfree[i]), 1);
            umma::mbar_init(sa(&b_sfull[i]), 1);
            umma::mbar_init(sa(&b_sfree[i]), AP_SMW);
        }
        umma::mbar_init(sa(&b_pfull), AP_SMW);
        umma::mbar_init(sa(&b_odone), 1);
        umma::mbar_init(sa(&b_xfull), 1);          // armed by this CTA, filled by the peer's stores
        umma::mbar_init(sa(&b_xfree), 1);          // the peer's thread 0, once it has read the scores
        umma::fence_mbar_init();
        umma::mbar_arrive_expect_tx(sa(&b_xfull), AP_XBYTES);
    }
    if (warp == 0) umma::tmem_alloc(sa(&tmem_base), APT_COLS);
    // ---- Q half: 64 heads x 256 dims, bf16 -> fp16, one round of loads
    {
        uint4 qv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = tid + u * AP_THREADS, h = i >> 5, c = i & 31;
            qv[u] = __ldg(reinterpret_cast<const uint4*>(q + ((gq * AP_H + h) * D_LAT + d0 + c * 8)));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = tid + u * AP_THREADS, h = i >> 5, c = i & 31;
            const uint4 v = qv[u];
            *reinterpret_cast<uint4*>(sm + AP_SQ + (c >> 3) * (AP_H * 128) + apswz(h, c & 7)) =
                make_uint4(ap_bf16x2_to_f16x2(v.x), ap_bf16x2_to_f16x2(v.y), ap_bf16x2_to_f16x2(v.z),
                           ap_bf16x2_to_f16x2(v.w));
        }
    }
    if (tid < 256) reinterpret_cast<uint4*>(sm + AP_SONES)[tid] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    float* m_run = reinterpret_cast<float*>(sm + AP_MISC);
    float* fac = m_run + AP_H;
    int* flag = reinterpret_cast<int*>(fac + AP_H);
    if (tid < AP_H) m_run[tid] = -INFINITY;
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    umma::cluster_sync();              // both CTAs' barriers exist before any remote store or arrive
    umma::fence_after();
    const uint32_t tmem = tmem_base;
    bool ok = true;

    if (warp > AP_MMAW) {
        // ================= loaders
        const int lt = tid - (AP_MMAW + 1) * 32;
        int* sidx = reinterpret_cast<int*>(sm + AP_SIDX);
        const uint8_t* codes_b = lat_codes + (int64_t)b * capacity * (D_LAT / 2) + d0 / 2;
        const uint8_t* scales_b = lat_scales + (int64_t)b * capacity * (D_LAT / 16) + d0 / 16;
        const uint16_t* win_b = swa + ((int64_t)b * swa_len + (wlo - swa_pos0)) * D_LAT + d0;
        for (int s = lt; s < k; s += AP_LOADERS) {
            const int j = idx[gq * k + s];
            sidx[s] = (j >= 0 && j < capacity) ? j : -1;
        }
        umma::bar_named(2, AP_LOADERS);
        // every row this CTA reads, into L2 now: the gathers below then hit L2
        for (int s = lt; s < k; s += AP_LOADERS) {
            const int j = sidx[s];
            if (j >= 0) {
                umma::prefetch_l2(codes_b + (int64_t)j * (D_LAT / 2));
                umma::prefetch_l2(scales_b + (int64_t)j * (D_LAT / 16));
            }
        }
        for (int u = lt; u < nwin * 4; u += AP_LOADERS) umma::prefetch_l2(win_b + (int64_t)(u >> 2) * D_LAT + (u & 3) * 64);
        for (int t = 0; t < T; ++t) {
            const int buf = t & 1;
            if (t >= 2) ok &= umma::mbar_wait(sa(&b_lfree[buf]), ((t >> 1) - 1) & 1);
            uint8_t* L = sm + AP_SL + buf * AP_LBUF;
            if (t == T - 1) {
                // window rows: 128 rows x 32 chunks of 8 dims (bf16 -> fp16), 8 loads in flight per thread
                for (int u0 = lt; u0 < AP_TILE * 32; u0 += AP_LOADERS * 8) {
                    uint4 wv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int u = u0 + i * AP_LOADERS, r = u >> 5, c = u & 31;
                        wv[i] = make_uint4(0, 0, 0, 0);
                        if (u < AP_TILE * 32 && r < nwin)
                            wv[i] = __ldg(reinterpret_cast<const uint4*>(win_b + (int64_t)r * D_LAT + c * 8));
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int u = u0 + i * AP_LOADERS, r = u >> 5, c = u & 31;
                        if (u < AP_TILE * 32) {
                            const uint4 v = wv[i];
                            *reinterpret_cast<uint4*>(L + (c >> 3) * AP_SLAB + apswz(r, c & 7)) =
                                make_uint4(ap_bf16x2_to_f16x2(v.x), ap_bf16x2_to_f16x2(v.y),
                                           ap_bf16x2_to_f16x2(v.z), ap_bf16x2_to_f16x2(v.w));
                            if (c == 0) rowok[buf][r] = r < nwin;
                        }
                    }
                }
            } else {
                // selected FP4 rows: 128 rows x 8 units of 32 dims (16 B of codes + 2 scale bytes)
                constexpr int NU = (AP_TILE * 8 + AP_LOADERS - 1) / AP_LOADERS;
                uint4 cw[NU];
                uint32_t sc[NU];
#pragma unroll
                for (int i = 0; i < NU; ++i) {
                    const int u = lt + i * AP_LOADERS, r = u >> 3, c = u & 7;
                    const int slot = t * AP_TILE + r;
                    cw[i] = make_uint4(0, 0, 0, 0);
                    sc[i] = 0u;
                    if (u < AP_TILE * 8 && slot < k) {
                        const int j = sidx[slot];
                        if (j >= 0) {
                            cw[i] = __ldg(reinterpret_cast<const uint4*>(codes_b + (int64_t)j * (D_LAT / 2)) + c);
                            sc[i] = __ldg(reinterpret_cast<const uint16_t*>(scales_b + (int64_t)j * (D_LAT / 16)) + c);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < NU; ++i) {
                    const int u = lt + i * AP_LOADERS, r = u >> 3, c = u & 7;
                    if (u < AP_TILE * 8) {
                        const int slot = t * AP_TILE + r;
                        const bool valid = slot < k && sidx[slot] >= 0;
                        const uint32_t words[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
                        // an empty slot has zero codes and zero scales, so it expands to zeros
                        const __half2 sp = ap_e4m3x2(sc[i]);
                        const __half2 s_lo = __low2half2(sp), s_hi = __high2half2(sp);
#pragma unroll
                        for (int w = 0; w < 4; ++w) {        // 8 dims per word; scale group 2c + w/2
                            const __half2 s2 = (w >> 1) ? s_hi : s_lo;
                            uint32_t f[4];
                            ap_e2m1x8(words[w], f);
                            const uint4 o = make_uint4(ap_hmul2(f[0], s2), ap_hmul2(f[1], s2), ap_hmul2(f[2], s2),
                                                       ap_hmul2(f[3], s2));
                            const int cc = c * 4 + w;                // 8-dim chunk 0..31
                            *reinterpret_cast<uint4*>(L + (cc >> 3) * AP_SLAB + apswz(r, cc & 7)) = o;
                        }
                        if (c == 0) rowok[buf][r] = valid;
                    }
                }
            }
            umma::fence_proxy_async();
            umma::mbar_arrive(sa(&b_lfull[buf]));
        }
    } else if (warp == AP_MMAW) {
        // ================= MMA issuer
        if (lane == 0) {
            const uint32_t id1 = umma::idesc_f16(128, AP_H, 0, 0);
            const uint32_t id2 = umma::idesc_f16(128, AP_H, 1, 1);
            const uint32_t id3 = umma::idesc_f16(128, AP_H, 0, 1);
            // Two independent streams: GEMM1 of tile t needs its half rows loaded
            // (lfull) and its score buffer released (sfree of tile t-2); GEMM2 of
            // tile t needs P (pfull).  Serve whichever is ready, so a slow load of
            // tile t+1 never holds back the value GEMM of tile t.
            int n1 = 0, n2 = 0;
            uint32_t spins = 0;
            while (n2 < T) {
                bool progressed = false;
                if (n1 < T && n1 <= n2 + 1) {
                    const int buf = n1 & 1;
                    if (umma::mbar_test(sa(&b_lfull[buf]), (n1 >> 1) & 1) &&
                        (n1 < 2 || umma::mbar_test(sa(&b_sfree[buf]), ((n1 >> 1) - 1) & 1))) {
                        umma::fence_after();
                        const uint32_t Lb = base + AP_SL + buf * AP_LBUF;
#pragma unroll
                        for (int ks = 0; ks < 16; ++ks) {
                            const uint64_t a = umma::desc(Lb + (ks >> 2) * AP_SLAB + (ks & 3) * 32, 16, 1024,
                                                          umma::LAYOUT_SW128);
                            const uint64_t bq = umma::desc(base + AP_SQ + (ks >> 2) * (AP_H * 128) + (ks & 3) * 32, 16,
                                                           1024, umma::LAYOUT_SW128);
                            umma::mma_f16(tmem + APT_S + 64 * buf, a, bq, id1, ks > 0);
                        }
                        umma::commit(sa(&b_sfull[buf]));
                        ++n1;
                        progressed = true;
                    }
                }
                if (n2 < n1 && umma::mbar_test(sa(&b_pfull), n2 & 1)) {
                    umma::fence_after();
                    const int buf = n2 & 1;
                    const uint32_t Lb = base + AP_SL + buf * AP_LBUF;
                    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint64_t a = umma::desc(Lb + (2 * mt) * AP_SLAB + ks * 2048, AP_SLAB, 1024,
                                                          umma::LAYOUT_SW128);
                            const uint64_t bp = umma::desc(base + AP_SP + ks * 2048, 8192, 1024, umma::LAYOUT_SW128);
                            umma::mma_f16(tmem + APT_O + 64 * mt, a, bp, id2, (n2 > 0 || ks > 0) ? 1u : 0u);
                        }
                    }
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t a = umma::desc(base + AP_SONES, 128, 256, umma::LAYOUT_NONE);
                        const uint64_t bp = umma::desc(base + AP_SP + ks * 2048, 8192, 1024, umma::LAYOUT_SW128);
                        umma::mma_f16(tmem + APT_L, a, bp, id3, (n2 > 0 || ks > 0) ? 1u : 0u);
                    }
                    umma::commit(sa(&b_odone));
                    umma::commit(sa(&b_lfree[buf]));
                    ++n2;
                    progressed = true;
                }
                if (progressed) {
                    spins = 0;
                } else if (++spins > (1u << 26)) {     // nothing moved for far too long: give up
                    ok = false;
                    break;
                }
            }
        }
    } else if (warp < AP_SMW) {
        // ================= softmax: thread = key row 32*(warp%4)+lane, heads hh*32 .. +31
        const int qd = warp & 3, hh = warp >> 2;
        const int row = qd * 32 + lane;
        const int hc = hh * 32;
        const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
        const uint32_t sx_peer = umma::mapa(base + AP_SX, peer);
        const uint32_t xfull_peer = umma::mapa(sa(&b_xfull), peer);
        const uint32_t xfree_peer = umma::mapa(sa(&b_xfree), peer);
        float* red = reinterpret_cast<float*>(sm + AP_RED);           // [4 quadrants][64 heads]
        const float* sx = reinterpret_cast<const float*>(sm + AP_SX);
        for (int t = 0; t < T; ++t) {
            const int buf = t & 1;
            float x[32];
            ok &= umma::mbar_wait(sa(&b_sfull[buf]), (t >> 1) & 1);
            umma::fence_after();
            umma::tmem_ld16(lane_base + APT_S + 64 * buf + hc, x);
            umma::tmem_ld16(lane_base + APT_S + 64 * buf + hc + 16, x + 16);
            umma::tmem_wait_ld();
            umma::fence_before();
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(sa(&b_sfree[buf]));
            // send the partial scores to the peer (16-byte chunks swizzled by row
            // to spread banks), once it has read the previous ones
            if (t >= 1) {
                if (tid == 0) ok &= umma::mbar_wait_cluster(sa(&b_xfree), (t - 1) & 1);
                umma::bar_named(1, AP_SMT);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
                umma::st_async_v4(sx_peer + row * 256 + (((hh * 8 + c) ^ (row & 15)) << 4), x[4 * c], x[4 * c + 1],
                                  x[4 * c + 2], x[4 * c + 3], xfull_peer);
            if (tid == 0) {
                ok &= umma::mbar_wait_cluster(sa(&b_xfull), t & 1);
                if (t + 1 < T) umma::mbar_arrive_expect_tx(sa(&b_xfull), AP_XBYTES);   // arm the next tile
            }
            umma::bar_named(1, AP_SMT);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 v = *reinterpret_cast<const float4*>(sx + row * 64 + (((hh * 8 + c) ^ (row & 15)) << 2));
                // S = S_0 + S_1 in both CTAs (addition is commutative, so the bits agree)
                x[4 * c] += v.x;
                x[4 * c + 1] += v.y;
                x[4 * c + 2] += v.z;
                x[4 * c + 3] += v.w;
            }
            // row validity was written by the loaders of this buffer: observe their barrier too
            ok &= umma::mbar_wait(sa(&b_lfull[buf]), (t >> 1) & 1);
            const bool valid = rowok[buf][row] != 0;
            bool exceed = false;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 mm = *reinterpret_cast<const float4*>(m_run + hc + 4 * q4);
                const float mv[4] = {mm.x, mm.y, mm.z, mm.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = 4 * q4 + e;
                    x[h] = valid ? x[h] * scale_log2e : -INFINITY;
                    exceed |= x[h] > mv[e] + AP_LAZY;
                }
            }
            // both CTAs hold the same scores, so they take the same branch
            const bool raise = umma::bar_red_or(1, AP_SMT, exceed);
            if (raise) {
                // new running max for the heads that rose too far: column maxima of the tile
#pragma unroll
                for (int h = 0; h < 32; ++h) {
                    const uint32_t mk = __reduce_max_sync(0xffffffffu, ap_ord(x[h]));
                    if (lane == 0) red[qd * AP_H + hc + h] = ap_unord(mk);
                }
                umma::bar_named(1, AP_SMT);
                if (tid < AP_H) {
                    const float mt = fmaxf(fmaxf(red[tid], red[AP_H + tid]), fmaxf(red[2 * AP_H + tid], red[3 * AP_H + tid]));
                    const float mo = m_run[tid];
                    float f = 1.0f;
                    if (mt > -INFINITY && (mo == -INFINITY || mt > mo + AP_LAZY)) {
                        f = (mo == -INFINITY) ? 0.0f : umma::ex2(mo - mt);
                        m_run[tid] = mt;
                    }
                    fac[tid] = f;
                    const unsigned any = __ballot_sync(0xffffffffu, f != 1.0f);
                    if (lane == 0) flag[warp] = any != 0;
                }
                if (t >= 1) ok &= umma::mbar_wait(sa(&b_odone), (t - 1) & 1);   // previous P and O are settled
                umma::bar_named(1, AP_SMT);
                umma::fence_after();
                if (t >= 1 && (flag[0] | flag[1])) {
                    // rescale O^T (both dim tiles) and l in this thread's 32 head columns
#pragma unroll 1
                    for (int blk = 0; blk < 3; ++blk) {
                        const uint32_t col0 = (blk < 2 ? APT_O + 64 * blk : APT_L) + hc;
#pragma unroll
                        for (int c = 0; c < 32; c += 16) {
                            float v[16];
                            umma::tmem_ld16(lane_base + col0 + c, v);
                            umma::tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] *= fac[hc + c + i];
                            umma::tmem_st16(lane_base + col0 + c, v);
                        }
                    }
                    umma::tmem_wait_st();
                }
            } else if (t >= 1) {
                ok &= umma::mbar_wait(sa(&b_odone), (t - 1) & 1);             // GEMM2 of t-1 has read P
            }
            // P = exp2(x - m_run), fp16, row = key (MN-major B operand), this thread's 4 chunks
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[4];
                const float4 ma = *reinterpret_cast<const float4*>(m_run + hc + 8 * c);
                const float4 mb = *reinterpret_cast<const float4*>(m_run + hc + 8 * c + 4);
                const float mv[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = 8 * c + 2 * e;
                    const float m0 = mv[2 * e], m1 = mv[2 * e + 1];
                    const float p0 = (x[h] == -INFINITY || m0 == -INFINITY) ? 0.0f : umma::ex2(x[h] - m0);
                    const float p1 = (x[h + 1] == -INFINITY || m1 == -INFINITY) ? 0.0f : umma::ex2(x[h + 1] - m1);
                    const __half2 hp = __floats2half2_rn(p0, p1);
                    w[e] = *reinterpret_cast<const uint32_t*>(&hp);
                }
                *reinterpret_cast<uint4*>(sm + AP_SP + apswz(row, hh * 4 + c)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            umma::fence_proxy_async();
            umma::fence_before();
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(sa(&b_pfull));
            // every warp read the peer's scores before the barrier above: let it send the next ones
            if (tid == 0) umma::mbar_arrive_remote(xfree_peer);
        }
        // ================= epilogue: thread = output dim 32*(warp%4)+lane of each 128-dim tile, its 32 heads
        ok &= umma::mbar_wait(sa(&b_odone), (T - 1) & 1);
        umma::fence_after();
        float inv[32];
        umma::tmem_ld16(lane_base + APT_L + hc, inv);
        umma::tmem_ld16(lane_base + APT_L + hc + 16, inv + 16);
        umma::tmem_wait_ld();
        if (lse != nullptr && rank == 0 && qd == 0 && lane == 0)
#pragma unroll
            for (int h = 0; h < 32; ++h)
                lse[gq * AP_H + hc + h] =
                    inv[h] > 0.0f ? (m_run[hc + h] + log2f(inv[h])) * 0.69314718055994531f : -INFINITY;
#pragma unroll
        for (int h = 0; h < 32; ++h) inv[h] = inv[h] > 0.0f ? 1.0f / inv[h] : 0.0f;
        for (int mt = 0; mt < 2; ++mt) {
            float* op = out + (gq * AP_H + hc) * D_LAT + d0 + mt * 128 + row;
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                float o[16];
                umma::tmem_ld16(lane_base + APT_O + 64 * mt + hc + c, o);
                umma::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    op[(int64_t)(c + i) * D_LAT] = ok ? o[i] * inv[c + i] : __int_as_float(0x7fc00000);
            }
        }
    }
    if (!ok) atomicExch(err, 1);
    umma::fence_before();
    __syncthreads();
    umma::cluster_sync();              // the peer is done with this CTA's shared memory
    if (warp == 0) {
        umma::fence_after();
        umma::tmem_dealloc(tmem, APT_COLS);
    }
}

bool attn_pair_supported(int H) { return H == AP_H; }

cudaError_t launch_sparse_attn_pair(const csa2_cache& c, const uint16_t* q, int n_q, const int64_t* q_pos,
                                    const int32_t* idx, int k, const uint16_t* swa, int64_t swa_pos0, int swa_len,
                                    float scale, float* out, float* lse, int* err, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(k_sparse_attn_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)AP_DYN);
    if (e != cudaSuccess) return e;
    const float scale_log2e = scale * 1.4426950408889634f;
    for (int q0 = 0; q0 < n_q; q0 += 65535) {
        const int nqc = (n_q - q0) < 65535 ? (n_q - q0) : 65535;
        dim3 grid(2, nqc, c.batch);
        k_sparse_attn_pair<<<grid, AP_THREADS, AP_DYN, st>>>(c.lat_codes, c.lat_scales, c.capacity, q, n_q, q0, q_pos,
                                                             idx, k, swa, swa_pos0, swa_len, scale_log2e, out, lse, err);
        note_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace csa2

// Sparse attention, 64 heads, one CTA pair (thread-block cluster of 2) per
// query ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる", §2.3.1 top-k
// entries plus the local window; §1.1 one 512-dim latent shared by every head).
//
// The pair splits the keys: CTA r takes the 64-key tiles r, r+2, .. of the
// selected FP4 entries and window rows [64r, 64r+64), with all 512 latent
// dims.  Per tile:
//   S^T = Q . L^T        (tcgen05, M = 64 heads, N = 64 keys, K = 512, fp32 in
//                         TMEM: head h in lane 32(h/16) + h%16)
//   an online softmax in which each thread owns one head and 32 of the tile's
//   keys (two threads per head): the running max is checked per thread and
//   raised only when a score rises more than 2^8 above it (then O is rescaled
//   in TMEM); P^T goes to shared memory in fp16 and its row sums stay in
//   registers;
//   O^T += L^T . P       (M = 128 dims x 4, N = 64 heads, K = 64 keys)
// Tiles are double-buffered (L, S, P), so the gather and dequantisation of the
// next tile overlap the MMAs and softmax of this one.  At the end the two CTAs
// swap their per-head running max and row sum through distributed shared
// memory (asynchronous remote stores counted on an mbarrier of the receiver:
// point to point, no cluster-wide barrier) and scale their partial O to the
// common max and normaliser; each
// sends its share of the other CTA's half of the output dims into that CTA's
// (now idle) Q area with asynchronous remote stores counted on an mbarrier,
// and stores its own half once, its share plus the one received.
//
// Warps: 0-7 softmax / epilogue (warp w: TMEM lane quarter w%4, key half
// w/4), warps 8 and 9 issue the score MMAs (K = dims 0-255 and 256-511 into
// two TMEM partials that the softmax adds; the first half starts as soon as
// its dims are expanded), warps 10 and 11 the output MMAs (dim tiles 0-1 and
// 2-3): one thread issues about one MMA per 55 cycles, two keep the tensor
// pipe busy.  Warps 12-19 gather rows (four 32-dim units of a tile per
// thread; the expansion sits on the tiles' critical path, and eight warps do it
// in four even rounds).  Q (loaded and converted to fp16 by warps 0-11, one
// head per warp at a time) and tile 0, the CTA's window rows
// (contiguous: one bulk copy), come first; the FP4 tiles follow, their rows
// prefetched into L2 one tile ahead, so the gathers are single L2 round trips.  Everything before
// the indices (Q, the window tile, TMEM and barriers) overlaps the preceding
// kernel of the stream (programmatic launch); only the loaders wait for it.
//
// Range: fp16 operands hold every FP4 latent value exactly, and bf16 q and
// window values exactly as long as they lie in [2^-14, 65504].  Any finite
// bf16 input is taken: a head of q whose largest magnitude falls outside
// [2^-10, 2^15) is scaled by a power of two into [2^14, 2^15) and its scores
// scaled back (exact); the same holds for the CTA's window rows, whose
// contribution to O is brought back to the common scale before the first FP4
// tile's values are added (or in the final scale when there is none).
#include "common.cuh"
#include "umma.cuh"

namespace csa2 {

constexpr int AP_TILE = 64;                          // keys per tile
constexpr int AP_H = 64;
constexpr int AP_THREADS = 640;
constexpr int AP_SMW = 8;                            // softmax warps 0-7
constexpr int AP_SMT = AP_SMW * 32;
constexpr int AP_MMAW = 8;                           // warps 8, 9 issue the score MMAs (GEMM1), dims 0-255 / 256-511
constexpr int AP_MMA2 = 10;                          // warps 10, 11 issue the output MMAs (GEMM2), dim tiles 0-1 / 2-3
constexpr int AP_LOADW = 12;                         // warps 12-19 gather rows
constexpr int AP_LOADERS = 256;
constexpr uint32_t AP_QSLAB = AP_H * 128;            // 64 heads x 64 dims fp16
constexpr uint32_t AP_LSLAB = AP_TILE * 128;         // 64 keys x 64 dims fp16
constexpr uint32_t AP_SQ = 0;                        // Q: 8 slabs (64 KB)
constexpr uint32_t AP_SL = 8 * AP_QSLAB;             // L: 2 buffers x 8 slabs (128 KB)
constexpr uint32_t AP_LBUF = 8 * AP_LSLAB;
constexpr uint32_t AP_SP = AP_SL + 2 * AP_LBUF;      // P^T: 2 buffers x 64 heads x 64 keys fp16
constexpr uint32_t AP_PBUF = AP_H * 128;
constexpr uint32_t AP_SIDX = AP_SP + 2 * AP_PBUF;    // the query's indices, MAX_K ints
constexpr uint32_t AP_RED = AP_SIDX + MAX_K * 4;     // per key half x 64 heads (max, then row sums)
constexpr uint32_t AP_MISC = AP_RED + 1024;          // m_run[64], fac[64], flags[8], own m/l, peer m/l, scale
constexpr uint32_t AP_DYN = AP_MISC + 3072 + 1024;
constexpr uint32_t APT_S = 0, APT_O = 256, APT_COLS = 512;   // S^T partial p of buffer b at APT_S + 64 (2b + p)
constexpr float AP_LAZY = 8.0f;                      // log2 headroom before the running max is raised

__device__ __forceinline__ uint32_t apswz(uint32_t row, uint32_t chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

__device__ __forceinline__ uint32_t ap_bf16x2_to_f16x2(uint32_t v) {
    __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    return *reinterpret_cast<uint32_t*>(&h);
}
// bf16 pair -> fp16 pair after scaling by d (a power of two): exact unless a value leaves fp16's range
__device__ __forceinline__ uint32_t ap_bf16x2_to_f16x2_scaled(uint32_t v, float d) {
    __half2 h = __floats2half2_rn(__uint_as_float(v << 16) * d, __uint_as_float(v & 0xffff0000u) * d);
    return *reinterpret_cast<uint32_t*>(&h);
}
// the largest bf16 magnitude (as bits, sign cleared) of the eight values in v
__device__ __forceinline__ uint32_t ap_absmax4(const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
    return m;
}
// 2^e as a float, for -126 <= e <= 127
__device__ __forceinline__ float ap_pow2(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }
// The power-of-two exponent E by which values whose largest magnitude has bf16 bits `mx` are
// divided before they go to fp16: 0 while that magnitude lies in [2^-10, 2^15) (or is 0), else
// the E that brings it into [2^14, 2^15), kept within [-100, 100].
__device__ __forceinline__ int ap_range_exp(uint32_t mx) {
    if (mx == 0u) return 0;
    const int e = (int)((mx >> 7) & 0xffu) - 127;          // largest magnitude in [2^e, 2^(e+1))
    if (e >= -10 && e < 15) return 0;
    return max(-100, min(100, e - 14));
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
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(AP_THREADS, 1) k_sparse_attn_pair(
    const uint8_t* __restrict__ lat_codes, const uint8_t* __restrict__ lat_scales, int capacity,
    const uint16_t* __restrict__ q, int n_q, int q0, const int64_t* __restrict__ q_pos,
    const int32_t* __restrict__ idx, int k, const uint16_t* __restrict__ swa, int64_t swa_pos0, int swa_len,
    float scale_log2e, float* __restrict__ out, float* __restrict__ lse, int* __restrict__ err) {
    // Programmatic launch: everything up to the indices (Q, the window rows and their tile, the
    // TMEM and barrier set-up) overlaps the preceding kernel; only the loaders wait for it, before
    // they read idx, and only then let the successor be scheduled, so that the successor overlaps
    // this kernel alone.  Nothing this kernel writes is read by that kernel.
    extern __shared__ uint8_t dyn[];
    __shared__ __align__(8) unsigned long long b_lhalf[2], b_lfull[2], b_lfree[2], b_sfull[2], b_sfree[2], b_pfull[2],
        b_odone[2], b_wfull, b_xch, b_ml;
    __shared__ uint32_t tmem_base;
    __shared__ __align__(16) uint8_t rowok[2][AP_TILE];

    const uint32_t raw = umma::smem_u32(dyn);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = dyn + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = umma::cluster_rank();
    const uint32_t peer = rank ^ 1u;
    const int qi = q0 + blockIdx.y, b = blockIdx.z;
    const int64_t gq = (int64_t)b * n_q + qi;

    // window of this query (clipped to the rows present); this CTA's tiles:
    // FP4 tiles rank, rank+2, .. of the T4 tiles of k entries, then its half of the window
    const int64_t p = q_pos[gq];
    int64_t wlo = p - (WINDOW - 1);
    if (wlo < 0) wlo = 0;
    if (wlo < swa_pos0) wlo = swa_pos0;
    int64_t whi = p;
    if (whi > swa_pos0 + swa_len - 1) whi = swa_pos0 + swa_len - 1;
    const int nwin = whi >= wlo ? (int)(whi - wlo + 1) : 0;
    const int nwr = max(0, min(AP_TILE, nwin - (int)rank * AP_TILE));   // window rows of this CTA
    const int T4 = (k + AP_TILE - 1) / AP_TILE;
    const int n4 = (T4 + 1 - (int)rank) / 2;
    const int T = n4 + 1;

    float* m_run = reinterpret_cast<float*>(sm + AP_MISC);          // [64]
    float* fac = m_run + AP_H;                                       // [64] running-max factor
    int* flag = reinterpret_cast<int*>(fac + AP_H);                  // [8]
    float* own_ml = reinterpret_cast<float*>(flag + 8);              // m[64], l[64]
    float* peer_ml = own_ml + 2 * AP_H;                              // written by the peer
    float* fown = peer_ml + 2 * AP_H;                                // this CTA's final scale per head
    float* ofac = fown + AP_H;                                       // [64] factor applied to O
    unsigned int* qmax = reinterpret_cast<unsigned int*>(ofac + AP_H);   // [64] exponent E of each head of q
    int* wexp = reinterpret_cast<int*>(qmax + AP_H);                 // [0] window exponent, [1] largest |window| bits
    float* red = reinterpret_cast<float*>(sm + AP_RED);              // [2 halves][64 heads]

    auto sa = [&](const void* x) { return umma::smem_u32(x); };
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            umma::mbar_init(sa(&b_lhalf[i]), AP_LOADERS / 32);   // dims 0-255 of the tile expanded (per warp)
            umma::mbar_init(sa(&b_lfull[i]), AP_LOADERS / 32);   // all of it
            umma::mbar_init(sa(&b_lfree[i]), 2);              // both GEMM2 issuers done with the tile
            umma::mbar_init(sa(&b_sfull[i]), 2);              // both K halves of the scores
            umma::mbar_init(sa(&b_sfree[i]), AP_SMW);
            umma::mbar_init(sa(&b_pfull[i]), AP_SMW);
            umma::mbar_init(sa(&b_odone[i]), 2);
        }
        umma::mbar_init(sa(&b_wfull), 1);
        umma::mbar_init(sa(&b_xch), 1);
        umma::mbar_init(sa(&b_ml), 1);
        umma::fence_mbar_init();
        // the peer's share of this CTA's half of the output arrives here (64 heads x 256 dims fp32)
        umma::mbar_arrive_expect_tx(sa(&b_xch), AP_H * 256 * 4);
        // and the peer's per-head running max and row sum (64 + 64 floats)
        umma::mbar_arrive_expect_tx(sa(&b_ml), 2 * AP_H * 4);
        // the window's largest magnitude starts at 0 before the loaders (past b_wfull) add to it
        wexp[1] = 0;
        // this CTA's window rows are contiguous: one bulk copy, raw bf16, into L buffer 1
        umma::mbar_arrive_expect_tx(sa(&b_wfull), (uint32_t)nwr * 1024u);
        if (nwr > 0)
            umma::bulk_g2s(base + AP_SL + AP_LBUF,
                           swa + ((int64_t)b * swa_len + (wlo - swa_pos0) + (int64_t)rank * AP_TILE) * D_LAT,
                           (uint32_t)nwr * 1024u, sa(&b_wfull));
    }
    // The loaders wait only for the barrier set-up (named barrier 3, with warp 0) and start on the
    // first tile at once; warps 0-11 stage Q and allocate TMEM among themselves (barrier 4).
    constexpr uint32_t AP_QT = AP_LOADW * 32;
    if (warp == 0) {
        __syncwarp();
        umma::bar_arrive(3, 32 + AP_LOADERS);
        umma::tmem_alloc(sa(&tmem_base), APT_COLS);
    }
    umma::cluster_arrive_relaxed();    // waited for before the first access to the peer's shared memory
    bool ok = true;
    uint32_t tmem = 0;
    if (warp >= AP_LOADW) {
        umma::bar_named(3, 32 + AP_LOADERS);
        {
            // tile 0 = the window rows: bf16 rows from L buffer 1 (bulk copy) to fp16 slabs in buffer 0;
            // their largest magnitude is tracked on the way, and should it lie outside
            // [2^-10, 2^15) each thread converts its own units again, scaled by 2^-E
            const int lt = tid - (int)AP_QT;
            ok &= umma::mbar_wait_fast(sa(&b_wfull), 0);
            const uint8_t* R = sm + AP_SL + AP_LBUF;
            uint8_t* L = sm + AP_SL;
            uint32_t mx = 0u;
            auto convert_window = [&](int ew) {
                const float wdown = ap_pow2(-ew);
                for (int u0 = lt; u0 < AP_TILE * 64; u0 += AP_LOADERS * 8) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int u = u0 + i * AP_LOADERS, r = u >> 6, c = u & 63;
                        if (u < AP_TILE * 64) {
                            uint4 v = make_uint4(0, 0, 0, 0);
                            if (r < nwr) v = *reinterpret_cast<const uint4*>(R + r * 1024 + c * 16);
                            uint4 o;
                            if (ew == 0) {
                                o = make_uint4(ap_bf16x2_to_f16x2(v.x), ap_bf16x2_to_f16x2(v.y),
                                               ap_bf16x2_to_f16x2(v.z), ap_bf16x2_to_f16x2(v.w));
                                mx = max(mx, ap_absmax4(v));
                            } else {
                                o = make_uint4(ap_bf16x2_to_f16x2_scaled(v.x, wdown), ap_bf16x2_to_f16x2_scaled(v.y, wdown),
                                               ap_bf16x2_to_f16x2_scaled(v.z, wdown), ap_bf16x2_to_f16x2_scaled(v.w, wdown));
                            }
                            *reinterpret_cast<uint4*>(L + (c >> 3) * AP_LSLAB + apswz(r, c & 7)) = o;
                            if (c == 0) rowok[0][r] = r < nwr ? 1 : 0;
                        }
                    }
                }
            };
            convert_window(0);
            mx = __reduce_max_sync(0xffffffffu, mx);
            if (lane == 0 && mx) atomicMax(reinterpret_cast<unsigned int*>(&wexp[1]), mx);
            umma::bar_named(2, AP_LOADERS);
            const int ew = ap_range_exp((uint32_t)wexp[1]);
            if (lt == 0) wexp[0] = ew;
            if (ew != 0) convert_window(ew);
            // each thread orders its own writes for the tensor core, then one arrival per warp
            umma::fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                umma::mbar_arrive(sa(&b_lhalf[0]));
                umma::mbar_arrive(sa(&b_lfull[0]));
            }
        }
        // the indices are the preceding kernel's output
        pdl_wait();
        pdl_launch_next();
        int* sidx = reinterpret_cast<int*>(sm + AP_SIDX);
        for (int u = tid - (int)AP_QT; u < n4 * AP_TILE; u += AP_LOADERS) {
            const int s = (2 * (u / AP_TILE) + (int)rank) * AP_TILE + u % AP_TILE;
            if (s < k) {
                const int j = idx[gq * k + s];
                sidx[s] = (j >= 0 && j < capacity) ? j : -1;
            }
        }
        umma::bar_named(2, AP_LOADERS);          // sidx staged; buffer 1 read in full before tile 1 overwrites it
    } else {
        // ---- Q: 64 heads x 512 dims, bf16 -> fp16, K-major slabs of 64 dims (A operand), by warps
        // 0-11: warp w takes heads w, w+12, .. (lane l: 16-byte chunks l and l+32 of each), all
        // loads in flight at once; a head whose largest magnitude lies outside [2^-10, 2^15) is
        // scaled by 2^-E on the way (the warp sees the whole head)
        constexpr int QW = AP_LOADW;                                   // warps staging Q
        constexpr int QHPW = (AP_H + QW - 1) / QW;                     // heads per warp (at most)
        uint4 qv[QHPW][2];
        const uint4* qsrc = reinterpret_cast<const uint4*>(q + gq * AP_H * D_LAT);
#pragma unroll
        for (int r = 0; r < QHPW; ++r) {
            const int h = warp + QW * r;
            if (h < AP_H) {
                qv[r][0] = __ldg(qsrc + h * 64 + lane);
                qv[r][1] = __ldg(qsrc + h * 64 + 32 + lane);
            }
        }
#pragma unroll
        for (int r = 0; r < QHPW; ++r) {
            const int h = warp + QW * r;
            if (h < AP_H) {                      // warp-uniform
                const uint32_t mx = __reduce_max_sync(0xffffffffu, max(ap_absmax4(qv[r][0]), ap_absmax4(qv[r][1])));
                const int eh = ap_range_exp(mx);
                const float d = ap_pow2(-eh);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int c = lane + 32 * hh;
                    const uint4 v = qv[r][hh];
                    uint4 o;
                    if (eh == 0)
                        o = make_uint4(ap_bf16x2_to_f16x2(v.x), ap_bf16x2_to_f16x2(v.y), ap_bf16x2_to_f16x2(v.z),
                                       ap_bf16x2_to_f16x2(v.w));
                    else
                        o = make_uint4(ap_bf16x2_to_f16x2_scaled(v.x, d), ap_bf16x2_to_f16x2_scaled(v.y, d),
                                       ap_bf16x2_to_f16x2_scaled(v.z, d), ap_bf16x2_to_f16x2_scaled(v.w, d));
                    *reinterpret_cast<uint4*>(sm + AP_SQ + (c >> 3) * AP_QSLAB + apswz(h, c & 7)) = o;
                }
                if (lane == 0) qmax[h] = (uint32_t)eh;     // the head's exponent
            }
        }
        if (tid < AP_H) m_run[tid] = -INFINITY;
        umma::fence_proxy_async();
        umma::fence_before();
        umma::bar_named(4, AP_QT);
        umma::fence_after();
        tmem = tmem_base;
    }

    if (warp >= AP_LOADW) {
        // ================= loaders
        const int lt = tid - (int)AP_QT;
        int* sidx = reinterpret_cast<int*>(sm + AP_SIDX);
        const uint8_t* codes_b = lat_codes + (int64_t)b * capacity * (D_LAT / 2);
        const uint8_t* scales_b = lat_scales + (int64_t)b * capacity * (D_LAT / 16);
        // the rows of FP4 tile f into L2, one tile ahead of the gathers: the gathers then hit L2,
        // and DRAM serves the tiles in the order they are needed
        auto prefetch_tile = [&](int f) {
            if (f < n4)
                for (int u = lt; u < AP_TILE; u += AP_LOADERS) {
                    const int s = (2 * f + (int)rank) * AP_TILE + u;
                    const int j = s < k ? sidx[s] : -1;
                    if (j >= 0) {
                        umma::prefetch_l2(codes_b + (int64_t)j * (D_LAT / 2));
                        umma::prefetch_l2(codes_b + (int64_t)j * (D_LAT / 2) + 128);
                        umma::prefetch_l2(scales_b + (int64_t)j * (D_LAT / 16));
                    }
                }
        };
        prefetch_tile(0);
        for (int t = 1; t < T; ++t) {
            const int buf = t & 1;
            uint8_t* L = sm + AP_SL + buf * AP_LBUF;
            {
                // selected FP4 rows: 64 rows x 16 units of 32 dims (16 B of codes + 2 scale bytes),
                // fetched before waiting for the buffer so that the round trip overlaps the wait
                constexpr int NU = (AP_TILE * 16 + AP_LOADERS - 1) / AP_LOADERS;
                const int f = t - 1;                        // FP4 tile f of this CTA
                const int slot0 = (2 * f + (int)rank) * AP_TILE;
                uint4 cw[NU];
                uint32_t sc[NU];
                // unit u of the tile (row r, 32-dim unit c): a warp takes 4 rows x 8 units, so that
                // one load instruction touches four whole 128-byte lines of codes (the gather is
                // paced by the lines looked up per instruction, not the bytes), and the 8 threads
                // of a quarter warp (4 rows, 2 units) write 8 different bank groups of the swizzled slab
                auto unit_rc = [](int u, int& r, int& c) {
                    const int q = u >> 5, l = u & 31;
                    r = 4 * (q & 15) + (l & 3);
                    c = 8 * (q >> 4) + (l >> 2);
                };
#pragma unroll
                for (int i = 0; i < NU; ++i) {
                    const int u = lt + i * AP_LOADERS;
                    int r, c;
                    unit_rc(u, r, c);
                    const int slot = slot0 + r;
                    cw[i] = make_uint4(0, 0, 0, 0);
                    sc[i] = 0u;
                    if (u < AP_TILE * 16 && slot < k) {
                        const int j = sidx[slot];
                        if (j >= 0) {
                            cw[i] = __ldg(reinterpret_cast<const uint4*>(codes_b + (int64_t)j * (D_LAT / 2)) + c);
                            sc[i] = __ldg(reinterpret_cast<const uint16_t*>(scales_b + (int64_t)j * (D_LAT / 16)) + c);
                        }
                    }
                }
                prefetch_tile(f + 1);
                if (t >= 2) ok &= umma::mbar_wait_fast(sa(&b_lfree[buf]), ((t >> 1) - 1) & 1);
                // units u < 512 hold dims 0-255 (c < 8): expanded first, so that the first half of
                // the score MMAs can start while the second half is expanded
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                for (int i = 0; i < NU; ++i) {
                    const int u = lt + i * AP_LOADERS;
                    int r, c;
                    unit_rc(u, r, c);
                    if (u < AP_TILE * 16 && (u >= AP_TILE * 8) == (hf == 1)) {
                        const int slot = slot0 + r;
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
                            const int cc = c * 4 + w;                // 8-dim chunk 0..63
                            *reinterpret_cast<uint4*>(L + (cc >> 3) * AP_LSLAB + apswz(r, cc & 7)) = o;
                        }
                        if (c == 0) rowok[buf][r] = valid ? 1 : 0;
                    }
                }
                if (hf == 0) {
                    umma::fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) umma::mbar_arrive(sa(&b_lhalf[buf]));
                }
                }
            }
            umma::fence_proxy_async();
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(sa(&b_lfull[buf]));
        }
    } else if (warp == AP_MMAW || warp == AP_MMAW + 1) {
        // ================= GEMM1 issuers: warp 8 + p takes dims 256p .. 256p+255 of S^T of tile t
        // into its own TMEM partial once those dims are expanded (lhalf / lfull) and the softmax
        // has read the scores of tile t-2 out of the same buffer (sfree)
        if (lane == 0) {
            const int part = warp - AP_MMAW;
            const uint32_t id1 = umma::idesc_f16(64, AP_TILE, 0, 0);
            const uint64_t qd0 = umma::desc(base + AP_SQ, 16, 1024, umma::LAYOUT_SW128);
            unsigned long long* ready = part == 0 ? b_lhalf : b_lfull;
            for (int t = 0; t < T && ok; ++t) {
                const int buf = t & 1;
                ok &= umma::mbar_wait_fast(sa(&ready[buf]), (t >> 1) & 1);
                if (t >= 2) ok &= umma::mbar_wait_fast(sa(&b_sfree[buf]), ((t >> 1) - 1) & 1);
                if (!ok) break;
                umma::fence_after();
                const uint64_t ld0 = umma::desc(base + AP_SL + buf * AP_LBUF, 16, 1024, umma::LAYOUT_SW128);
                // K-step ks: 16 dims at byte (ks/4) * slab + (ks%4) * 32 of both operands (Q and L
                // slabs have the same size), i.e. a constant added to the descriptors' address field
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const int ks = 16 * part + kk;
                    const uint64_t off = (uint64_t)(((ks >> 2) * AP_QSLAB + (ks & 3) * 32) >> 4);
                    umma::mma_f16(tmem + APT_S + 64 * (2 * buf + part), qd0 + off, ld0 + off, id1, kk > 0);
                }
                umma::commit(sa(&b_sfull[buf]));
            }
        }
    } else if (warp == AP_MMA2 || warp == AP_MMA2 + 1) {
        // ================= GEMM2 issuers: warp 10 + p adds dim tiles 2p, 2p+1 of O^T += L^T . P of
        // tile t once P is written (pfull); the completion of both releases the L buffer (lfree)
        // and the P buffer (odone)
        if (lane == 0) {
            const int part = warp - AP_MMA2;
            const uint32_t id2 = umma::idesc_f16(128, AP_H, 1, 0);
            for (int t = 0; t < T && ok; ++t) {
                const int buf = t & 1;
                ok &= umma::mbar_wait_fast(sa(&b_pfull[buf]), (t >> 1) & 1);
                if (!ok) break;
                umma::fence_after();
                const uint64_t la0 = umma::desc(base + AP_SL + buf * AP_LBUF, AP_LSLAB, 1024, umma::LAYOUT_SW128);
                const uint64_t pb0 = umma::desc(base + AP_SP + buf * AP_PBUF, 16, 1024, umma::LAYOUT_SW128);
#pragma unroll
                for (int mt = 2 * part; mt < 2 * part + 2; ++mt) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t offa = (uint64_t)(((2 * mt) * AP_LSLAB + ks * 2048) >> 4);
                        const uint64_t offp = (uint64_t)((ks * 32) >> 4);
                        umma::mma_f16(tmem + APT_O + 64 * mt, la0 + offa, pb0 + offp, id2, (t > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                umma::commit(sa(&b_odone[buf]));
                umma::commit(sa(&b_lfree[buf]));
            }
        }
    } else {
        // ================= softmax: warp w reads the 16 score rows (heads) of TMEM lane
        // quarter w%4 with the 16x64b shape, for keys 32(w/4) .. +31 of each tile: lane t
        // holds head 16(w%4) + t/4 + 8(t%2) and the keys of parity par = (t/2)%2
        const int qd = warp & 3, half = warp >> 2;
        const int h = qd * 16 + (lane >> 2) + 8 * (lane & 1);
        const int par = (lane >> 1) & 1;
        const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
        const float hmul = scale_log2e * ap_pow2((int)qmax[h]);   // times this head's q exponent
        float lsum = 0.0f;                   // sum of P over this thread's keys, all tiles so far
        int ew = 0;                          // exponent of the window rows (known once tile 0 is in)
        for (int t = 0; t < T; ++t) {
            const int buf = t & 1;
            float x[16];                     // keys 32*half + par + 2i
            ok &= umma::mbar_wait_fast(sa(&b_sfull[buf]), (t >> 1) & 1);
            umma::fence_after();
            {
                float x1[16];
                umma::tmem_ld16x64b_x16(lane_base + APT_S + 64 * (2 * buf) + 32 * half, x);
                umma::tmem_ld16x64b_x16(lane_base + APT_S + 64 * (2 * buf + 1) + 32 * half, x1);
                umma::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] += x1[i];
            }
            umma::fence_before();
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(sa(&b_sfree[buf]));
            // key validity was written by the loaders of this buffer: observe their barrier too
            ok &= umma::mbar_wait_fast(sa(&b_lfull[buf]), (t >> 1) & 1);
            if (t == 0) ew = wexp[0];
            const float mul = t == 0 ? hmul * ap_pow2(ew) : hmul;
            // the window tile's part of O is brought to the common scale before tile 1 adds to it
            const bool force = t == 1 && ew != 0;
            const float mh = m_run[h];
            bool exceed = false;
            {
                const uint4 v0 = *reinterpret_cast<const uint4*>(&rowok[buf][32 * half]);
                const uint4 v1 = *reinterpret_cast<const uint4*>(&rowok[buf][32 * half + 16]);
                const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int key = par + 2 * i;                       // within the half
                    const bool valid = (vw[key >> 2] >> (8 * (key & 3))) & 0xffu;
                    x[i] = valid ? x[i] * mul : -INFINITY;
                    exceed |= x[i] > mh + AP_LAZY;
                }
            }
            const bool raise = umma::bar_red_or(1, AP_SMT, exceed);
            if (raise || force) {
                // new running max for the heads that rose too far: max over the head's four threads
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < 16; ++i) mx = fmaxf(mx, x[i]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                if (par == 0) red[half * AP_H + h] = mx;
                umma::bar_named(1, AP_SMT);
                if (half == 0) {
                    float f = 1.0f;
                    if (par == 0) {
                        const float mt = fmaxf(red[h], red[AP_H + h]);
                        const float mo = m_run[h];
                        if (mt > -INFINITY && (mo == -INFINITY || mt > mo + AP_LAZY)) {
                            f = (mo == -INFINITY) ? 0.0f : umma::ex2(mo - mt);
                            m_run[h] = mt;
                        }
                        fac[h] = f;
                        ofac[h] = force ? f * ap_pow2(ew) : f;
                    }
                    const float of = force ? f * ap_pow2(ew) : f;
                    const unsigned any = __ballot_sync(0xffffffffu, of != 1.0f);
                    if (lane == 0) flag[qd] = any != 0;
                }
                if (t >= 1) ok &= umma::mbar_wait_fast(sa(&b_odone[(t - 1) & 1]), ((t - 1) >> 1) & 1);   // O settled
                umma::bar_named(1, AP_SMT);
                umma::fence_after();
                if (t >= 1 && (flag[0] | flag[1] | flag[2] | flag[3])) {
                    // rescale O^T: this warp's lane quarter of dim tiles 2*half and 2*half+1, all 64 heads
#pragma unroll 1
                    for (int mt = 2 * half; mt < 2 * half + 2; ++mt) {
#pragma unroll 1
                        for (int c = 0; c < AP_H; c += 16) {
                            float v[16];
                            umma::tmem_ld16(lane_base + APT_O + 64 * mt + c, v);
                            umma::tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] *= ofac[c + i];
                            umma::tmem_st16(lane_base + APT_O + 64 * mt + c, v);
                        }
                    }
                    umma::tmem_wait_st();
                }
                lsum *= fac[h];
            }
            // the P buffer of this tile was last read by GEMM2 of tile t-2
            if (t >= 2) ok &= umma::mbar_wait_fast(sa(&b_odone[buf]), ((t >> 1) - 1) & 1);
            const float m = m_run[h];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                x[i] = (x[i] == -INFINITY || m == -INFINITY) ? 0.0f : umma::ex2_ftz(x[i] - m);
                lsum += x[i];
            }
            // P^T row h, keys 32*half + 16*par .. +15 from this thread: trade half of the values with
            // the lane of the other parity so that each holds 16 consecutive keys
            float rv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) rv[i] = __shfl_xor_sync(0xffffffffu, par ? x[i] : x[8 + i], 2);
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __half2 hp = par ? __floats2half2_rn(rv[j], x[8 + j]) : __floats2half2_rn(x[j], rv[j]);
                w[j] = *reinterpret_cast<const uint32_t*>(&hp);
            }
            uint8_t* P = sm + AP_SP + buf * AP_PBUF;
            *reinterpret_cast<uint4*>(P + apswz(h, 4 * half + 2 * par)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(P + apswz(h, 4 * half + 2 * par + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
            umma::fence_proxy_async();
            umma::fence_before();
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(sa(&b_pfull[buf]));
        }
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
        // ---- per-head max and row sum of this CTA, to the peer
        if (par == 0) red[half * AP_H + h] = lsum;
        umma::bar_named(1, AP_SMT);
    }
    umma::cluster_wait();              // both CTAs have started: the peer's shared memory exists
    if (warp < AP_SMW) {
        if (tid < AP_H) {
            const float l = red[tid] + red[AP_H + tid];
            own_ml[tid] = m_run[tid];
            own_ml[AP_H + tid] = l;
            const uint32_t mb = umma::mapa(sa(&b_ml), peer);
            umma::st_async_b32(umma::mapa(sa(peer_ml + tid), peer), __float_as_uint(m_run[tid]), mb);
            umma::st_async_b32(umma::mapa(sa(peer_ml + AP_H + tid), peer), __float_as_uint(l), mb);
        }
    }
    // ================= combine the pair: the peer's max / row sums arrive on b_ml (point to point; every
    // remote store of either CTA is counted on a barrier its owner waits for before it exits)
    if (warp < AP_SMW) {
        ok &= umma::mbar_wait_cluster(sa(&b_ml), 0);
        umma::bar_named(1, AP_SMT);    // own_ml of every head written
        if (tid < AP_H) {
            const float m0 = own_ml[tid], l0 = own_ml[AP_H + tid], m1 = peer_ml[tid], l1 = peer_ml[AP_H + tid];
            const float mm = fmaxf(m0, m1);
            const float s0 = (m0 == -INFINITY) ? 0.0f : umma::ex2(m0 - mm);
            const float s1 = (m1 == -INFINITY) ? 0.0f : umma::ex2(m1 - mm);
            const float Lt = l0 * s0 + l1 * s1;
            // O still carries the window rows' exponent when no FP4 tile followed them
            fown[tid] = Lt > 0.0f ? s0 / Lt * (T == 1 ? ap_pow2(wexp[0]) : 1.0f) : 0.0f;
            if (lse != nullptr && rank == 0)
                lse[gq * AP_H + tid] = Lt > 0.0f ? (mm + log2f(Lt)) * 0.69314718055994531f : -INFINITY;
        }
        umma::bar_named(1, AP_SMT);
        ok &= umma::mbar_wait_fast(sa(&b_odone[(T - 1) & 1]), ((T - 1) >> 1) & 1);   // every GEMM2 is done
        umma::fence_after();
        // this CTA's share of the peer's half of the dims (dim tile 2*peer + half, this warp's lane
        // quarter), scaled, goes into the peer's Q area (free: the peer's score MMAs are done) as
        // [head][256 dims], counted on the peer's exchange barrier
        const int qd = warp & 3, half = warp >> 2;
        {
            const int mt = 2 * (int)peer + half;
            const int dl = half * 128 + qd * 32 + lane;                 // dim within the peer's half
            const uint32_t dst = umma::mapa(sa(sm + AP_SQ), peer) + (uint32_t)dl * 4u;
            const uint32_t mb = umma::mapa(sa(&b_xch), peer);
#pragma unroll 1
            for (int c = 0; c < AP_H; c += 16) {
                float v[16];
                umma::tmem_ld16(tmem + ((uint32_t)(qd * 32) << 16) + APT_O + 64 * mt + c, v);
                umma::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    umma::st_async_b32(dst + (uint32_t)(c + i) * 1024u,
                                       __float_as_uint(ok ? __fmul_rn(v[i], fown[c + i]) : __int_as_float(0x7fc00000)), mb);
            }
        }
        // this CTA's half: its own share plus the peer's, one store
        {
            const bool got = umma::mbar_wait_cluster(sa(&b_xch), 0);
            ok &= got;
            const int mt = 2 * (int)rank + half;
            const int dl = half * 128 + qd * 32 + lane;
            const float* px = reinterpret_cast<const float*>(sm + AP_SQ) + dl;
            float* op = out + (gq * AP_H) * D_LAT + (int)rank * 256 + dl;
#pragma unroll 1
            for (int c = 0; c < AP_H; c += 16) {
                float v[16];
                umma::tmem_ld16(tmem + ((uint32_t)(qd * 32) << 16) + APT_O + 64 * mt + c, v);
                umma::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    op[(int64_t)(c + i) * D_LAT] =
                        ok ? __fadd_rn(__fmul_rn(v[i], fown[c + i]), px[(c + i) * 256]) : __int_as_float(0x7fc00000);
            }
        }
    }
    if (!ok) atomicExch(err, 1);
    umma::fence_before();
    __syncthreads();
    if (warp == 0) {
        umma::fence_after();
        umma::tmem_dealloc(tmem, APT_COLS);
    }
}

bool attn_pair_supported(int H) { return H == AP_H; }

size_t attn_pair_ws(int, int) { return 256; }

cudaError_t launch_sparse_attn_pair(const csa2_cache& c, const uint16_t* q, int n_q, const int64_t* q_pos,
                                    const int32_t* idx, int k, const uint16_t* swa, int64_t swa_pos0, int swa_len,
                                    float scale, float* out, float* lse, void* ws, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(k_sparse_attn_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)AP_DYN);
    if (e != cudaSuccess) return e;
    int* err = reinterpret_cast<int*>(ws);
    const float scale_log2e = scale * 1.4426950408889634f;
    for (int q0 = 0; q0 < n_q; q0 += 65535) {
        const int nqc = (n_q - q0) < 65535 ? (n_q - q0) : 65535;
        dim3 grid(2, nqc, c.batch);
        launch_k(k_sparse_attn_pair, grid, AP_THREADS, AP_DYN, st, c.lat_codes, c.lat_scales, c.capacity, q, n_q, q0, q_pos,
                                                             idx, k, swa, swa_pos0, swa_len, scale_log2e, out, lse, err);
        note_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace csa2

// Full indexer scan on the tensor cores ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の
// 限界を押し広げる", §2.3.1 lightweight indexer over FP4 keys).
//
// For one query and a chunk of 4096 entries, 128 entries at a time:
//   A = key codes  [128 entries x d_I] FP4 E2M1 (kind::f8f6f4: each 16-value
//       group is 8 packed bytes followed by 8 pad bytes in shared memory)
//   B = block-diagonal query [H*G rows x d_I]: row (h, g) holds head h's codes
//       of group g and zeros elsewhere
//   D = A . B^T   M = 128, N = H*G, K = d_I   (fp32 in TMEM)
// D[e][(h,g)] is the exact group sum sum_{i in g} k_i q_hi (multiples of 1/4,
// |.| <= 16 * 6 * 6 = 576).  The epilogue forms the exact terms t = D * s_q * s_k
// and adds them per head (even and odd groups in two chains, two groups' values
// per packed f32x2 instruction) into the fp32 score S~.  Its rounding error is
// at most fac * sum_h |w_h| sum_g |t_hg| (fac keeps a factor of two in hand),
// and with |D| <= 576 that sum is at most sum_g C_g s_kg, C_g = 576 sum_h |w_h|
// s_qhg being one number per group for the whole query: the bound costs one
// fma per group and entry.  It is looser than one built from the entry's own
// group sums, which only widens the band the selection rescores exactly.
//
// The epilogue writes, for every eligible entry, its upper bound S~+E to the
// query's dense list, and for each aligned group of 8 entries the largest
// lower bound S~-E (as an order key); with an HSI pool also each block's bounds
// (the largest member bounds, over the block's lanes).  The selection kernel
// takes its thresholds from those group maxima: each is the lower bound of a
// different entry, so the k-th largest of them never exceeds the k-th largest
// lower bound.
//
// Warp roles (384 threads): warps 0-7 epilogue in two groups of four that take
// alternate tiles, each with its own TMEM accumulator (in a group one TMEM lane
// = one entry); warp 8 lane 0 issues the MMAs, warp 9 lane 0 issues 1-D bulk
// copies of each tile's contiguous key rows (8 KB codes + 1 KB scales, four
// tiles in flight), warps 10-11 expand the packed codes into the padded MMA
// layout.  Two A slots and two TMEM accumulators keep copies, MMAs and
// epilogues overlapped.
#include "indexer_common.cuh"
#include "umma.cuh"

namespace csa2 {

constexpr int ITC_E = 4096;                 // entries per block
constexpr int ITC_TILE = 128;
constexpr int ITC_NR = 4;                   // raw staging slots (bulk-copy depth)
constexpr int ITC_NA = 2;                   // MMA-layout A slots
constexpr int ITC_DI = 128;
constexpr int ITC_G = ITC_DI / 16;
constexpr int ITC_THREADS = 384;
constexpr int ITC_MMAW = 8, ITC_COPYW = 9, ITC_XW0 = 10;   // warps 0-7 epilogue (two groups of four)
constexpr int ITC_XFORM = 64;               // warps 10-11 expand raw codes into the MMA layout
// shared memory (from the 1024-aligned base)
constexpr int ITC_H = 8;                    // indexer heads taken by this kernel
constexpr int ITC_N = ITC_H * ITC_G;        // MMA N: one column per (head, group)
constexpr uint32_t IS_B = 0;                                  // query operand, 64 rows x 128 B
constexpr uint32_t IS_A = ITC_N * 128;                        // 2 slots x 128 rows x 128 B
constexpr uint32_t RAW_SLOT = ITC_TILE * (ITC_DI / 2) + ITC_TILE * 8;   // codes 8 KB + scales 1 KB
constexpr uint32_t IS_RAW = IS_A + ITC_NA * ITC_TILE * 128;   // 4 slots of raw rows
constexpr uint32_t IS_Q = IS_RAW + ITC_NR * RAW_SLOT;         // sq [H][G] floats + w [H]
constexpr uint32_t IS_END = IS_Q + 2048;
constexpr uint32_t IS_DYN = IS_END + 1024;

__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t unit) { return row * 128 + ((unit ^ (row & 7)) << 4); }

// The outputs for query slab `slab` (row stride list_len): dense_ub(lu, slab, list_len)[e] = the
// upper bound of entry e (entries 0 .. n_elig-1), wmk[e / 8] = the largest lower-bound key of
// entries e .. e+7 (f32_key order; the key of -inf when none is eligible), blu[e / bs] = the bounds
// of HSI block e / bs (bs a power of two up to 32; bs == 0: no blocks).
__global__ void __launch_bounds__(384, 2) k_scan_full_tc(
    const uint8_t* __restrict__ kc_all, const uint8_t* __restrict__ ks_all, int capacity,
    const uint8_t* __restrict__ iq_codes, const uint8_t* __restrict__ iq_scales, const float* __restrict__ w_head,
    const int64_t* __restrict__ q_pos, int n_q, int q0, int n_qc, int H, int bs, unsigned int* __restrict__ wmk,
    float2* __restrict__ lu, float2* __restrict__ blu, int list_len, int* __restrict__ err, int ratio) {
    pdl_wait();             // the selection that follows is let in only as the scan's blocks exit
    extern __shared__ uint8_t dyn[];
    __shared__ __align__(8) unsigned long long bar_rfull[ITC_NR], bar_rfree[ITC_NR], bar_afull[ITC_NA], bar_afree[ITC_NA],
        bar_dfull[2], bar_dfree[2];
    __shared__ uint32_t tmem_base;
    __shared__ int s_nel;

    const uint32_t raw = umma::smem_u32(dyn);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = dyn + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, ql = blockIdx.y;
    const int64_t gq = (int64_t)b * n_q + q0 + ql;
    const int64_t slab = (int64_t)b * n_qc + ql;
    const int c0 = blockIdx.x * ITC_E;
    constexpr int N = ITC_N;

    if (tid == 0) {
        s_nel = n_elig_of(q_pos[gq], capacity, ratio);
        for (int i = 0; i < ITC_NR; ++i) {
            umma::mbar_init(umma::smem_u32(&bar_rfull[i]), 1);
            umma::mbar_init(umma::smem_u32(&bar_rfree[i]), 128);
        }
        for (int i = 0; i < ITC_NA; ++i) {
            umma::mbar_init(umma::smem_u32(&bar_afull[i]), ITC_XFORM);
            umma::mbar_init(umma::smem_u32(&bar_afree[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            umma::mbar_init(umma::smem_u32(&bar_dfull[i]), 1);
            umma::mbar_init(umma::smem_u32(&bar_dfree[i]), 128);
        }
        umma::fence_mbar_init();
    }
    // query operand: row n = (h, g) -> unit g holds head h's 8 code bytes of
    // group g; every other byte of the row is zero
    const uint8_t* qc = iq_codes + gq * H * (ITC_DI / 2);
    for (int i = tid; i < N * 8; i += blockDim.x) {
        const int n = i >> 3, u = i & 7, h = n / ITC_G, g = n % ITC_G;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (u == g) {
            const uint2 c = *reinterpret_cast<const uint2*>(qc + h * (ITC_DI / 2) + g * 8);
            v.x = c.x;
            v.y = c.y;
        }
        *reinterpret_cast<uint4*>(sm + IS_B + swz128(n, u)) = v;
    }
    float* sq = reinterpret_cast<float*>(sm + IS_Q);          // [H][G]
    float* ww = sq + H * ITC_G;                                // [H]
    for (int i = tid; i < H * ITC_G; i += blockDim.x) sq[i] = e4m3_to_f32(iq_scales[gq * H * ITC_G + i]);
    for (int i = tid; i < H; i += blockDim.x) ww[i] = w_head[gq * H + i];
    // zero the A slots once: the pad half of every 16-byte unit stays zero
    for (int i = tid; i < ITC_NA * ITC_TILE * 8; i += blockDim.x)
        reinterpret_cast<uint4*>(sm + IS_A)[i] = make_uint4(0, 0, 0, 0);
    if (warp == 0) umma::tmem_alloc(umma::smem_u32(&tmem_base), 128);
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = tmem_base;
    const int n_elig = s_nel;
    const int n_loc = min(max(n_elig - c0, 0), ITC_E);
    const int n_tiles = (n_loc + ITC_TILE - 1) / ITC_TILE;
    bool ok = true;

    // scale rows are 8 bytes; a bulk copy needs a 16-byte aligned source
    const uint8_t* ks_seq = ks_all + ((int64_t)b * capacity + c0) * ITC_G;
    const bool bulk_scales = ((reinterpret_cast<uintptr_t>(ks_seq) & 15u) == 0);
    if (warp == ITC_COPYW) {
        // ---- bulk-copy issuer
        if (lane == 0) {
            for (int t = 0; t < n_tiles; ++t) {
                const int r = t % ITC_NR;
                if (t >= ITC_NR) ok &= umma::mbar_wait(umma::smem_u32(&bar_rfree[r]), ((t / ITC_NR) - 1) & 1);
                const int e0 = c0 + t * ITC_TILE;
                const int rows = min(ITC_TILE, n_elig - e0);
                const uint32_t cb = (uint32_t)rows * (ITC_DI / 2);
                const uint32_t sbytes = bulk_scales ? (uint32_t)(rows & ~1) * ITC_G : 0u;
                const uint32_t mb = umma::smem_u32(&bar_rfull[r]);
                const uint32_t dst = base + IS_RAW + r * RAW_SLOT;
                umma::mbar_arrive_expect_tx(mb, cb + sbytes);
                umma::bulk_g2s(dst, kc_all + ((int64_t)b * capacity + e0) * (ITC_DI / 2), cb, mb);
                if (sbytes) umma::bulk_g2s(dst + ITC_TILE * (ITC_DI / 2), ks_all + ((int64_t)b * capacity + e0) * ITC_G, sbytes, mb);
            }
        }
    } else if (warp >= ITC_XW0) {
        // ---- expand packed codes (8 bytes per 16-value group) into the data half of each 16-byte unit
        const int xt = tid - ITC_XW0 * 32;
        for (int t = 0; t < n_tiles; ++t) {
            const int r = t % ITC_NR, a = t % ITC_NA;
            ok &= umma::mbar_wait(umma::smem_u32(&bar_rfull[r]), (t / ITC_NR) & 1);
            if (t >= ITC_NA) ok &= umma::mbar_wait(umma::smem_u32(&bar_afree[a]), ((t / ITC_NA) - 1) & 1);
            const uint4* raw = reinterpret_cast<const uint4*>(sm + IS_RAW + r * RAW_SLOT);
            uint8_t* as = sm + IS_A + a * (ITC_TILE * 128);
#pragma unroll 4
            for (int c = xt; c < ITC_TILE * 4; c += ITC_XFORM) {
                const int row = c >> 2, q4 = c & 3;
                const uint4 v = raw[c];
                *reinterpret_cast<uint2*>(as + swz128(row, 2 * q4)) = make_uint2(v.x, v.y);
                *reinterpret_cast<uint2*>(as + swz128(row, 2 * q4 + 1)) = make_uint2(v.z, v.w);
            }
            umma::fence_proxy_async();
            umma::mbar_arrive(umma::smem_u32(&bar_afull[a]));
        }
    } else if (warp == ITC_MMAW) {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (5u << 7) | (5u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            for (int t = 0; t < n_tiles; ++t) {
                const int s = t % ITC_NA, d = t & 1;
                ok &= umma::mbar_wait(umma::smem_u32(&bar_afull[s]), (t / ITC_NA) & 1);
                if (t >= 2) ok &= umma::mbar_wait(umma::smem_u32(&bar_dfree[d]), ((t >> 1) - 1) & 1);
                umma::fence_after();
#pragma unroll
                for (int ks = 0; ks < ITC_DI / 32; ++ks) {
                    const uint64_t ad = umma::desc(base + IS_A + s * (ITC_TILE * 128) + ks * 32, 16, 1024,
                                                   umma::LAYOUT_SW128);
                    const uint64_t bd = umma::desc(base + IS_B + ks * 32, 16, 1024, umma::LAYOUT_SW128);
                    asm volatile(
                        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(tmem + 64 * d),
                        "l"(ad), "l"(bd), "r"(idesc), "r"(ks));
                }
                umma::commit(umma::smem_u32(&bar_dfull[d]));
                umma::commit(umma::smem_u32(&bar_afree[s]));
            }
        }
    } else {
        // ---- epilogue: one entry per thread
        // fac * ||w||, with room for the rounding of the norms and of the sum of squares
        // C_g times fac, rounded up, with a factor 1 + 2^-10 for the rounding of the 8-term sum below
        float cb[ITC_G];
#pragma unroll
        for (int g = 0; g < ITC_G; ++g) {
            float a = 0.0f;
            for (int h = 0; h < ITC_H; ++h) a = __fmaf_ru(fabsf(ww[h]), sq[h * ITC_G + g], a);
            cb[g] = __fmul_ru(__fmul_ru(a, 576.0f * bound_factor(H, ITC_DI)), 1.0f + 0x1p-10f);
        }
        float* ub_q = dense_ub(lu, slab, list_len);
        unsigned int* wm_q = wmk + slab * list_len;
        float2* blu_q = blu + slab * list_len;
        const int bsh = (bs >= 2 && bs <= 32 && (bs & (bs - 1)) == 0) ? bs : 0;
        // warp w takes the tiles t with t % 2 == w / 4 (TMEM accumulator t % 2), lane quarter w % 4
        const int eg = warp >> 2, wq = warp & 3;
        for (int t = eg; t < n_tiles; t += 2) {
            const int s = t % ITC_NR, d = t & 1;
            const int r = wq * 32 + lane;               // row of the tile = TMEM lane
            const int e0 = c0 + t * ITC_TILE;
            const int rows = min(ITC_TILE, n_elig - e0);
            uint2 skw = make_uint2(0, 0);
            // the scales landed with this slot's bulk copy: observe that barrier phase too
            if (bulk_scales) ok &= umma::mbar_wait(umma::smem_u32(&bar_rfull[s]), (t / ITC_NR) & 1);
            if (bulk_scales && r < (rows & ~1))
                skw = *reinterpret_cast<const uint2*>(sm + IS_RAW + s * RAW_SLOT + ITC_TILE * (ITC_DI / 2) + r * 8);
            else if (r < rows)
                skw = __ldg(reinterpret_cast<const uint2*>(ks_all + ((int64_t)b * capacity + e0 + r) * ITC_G));
            float skf[ITC_G], E = 0.0f;
#pragma unroll
            for (int g = 0; g < ITC_G; ++g) {
                skf[g] = e4m3_to_f32(((g < 4 ? skw.x : skw.y) >> (8 * (g & 3))) & 255u);
                E = __fmaf_rn(cb[g], skf[g], E);
            }
            // the group sums in two halves of four heads (32 columns), to keep registers low
            ok &= umma::mbar_wait(umma::smem_u32(&bar_dfull[d]), (t >> 1) & 1);
            umma::fence_after();
            // the raw slot may be refilled only now: the tile's MMAs were issued, so the expanding warps
            // are done reading its codes (and this thread has its scales)
            umma::mbar_arrive(umma::smem_u32(&bar_rfree[s]));
            const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16) + 64 * d;
            float S = 0.0f;
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
                float dv[32];
                umma::tmem_ld16(lane_base + 32 * hp, dv);
                umma::tmem_ld16(lane_base + 32 * hp + 16, dv + 16);
                umma::tmem_wait_ld();
                if (hp == 1) {
                    umma::fence_before();
                    umma::mbar_arrive(umma::smem_u32(&bar_dfree[d]));
                }
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    const int h = 4 * hp + hh;
                    float de = 0.0f, dod = 0.0f;
#pragma unroll
                    for (int g = 0; g < ITC_G; g += 2) {
                        // x = D s_q is exact (a multiple of 1/4 below 2^10 times an E4M3 value), and so is
                        // its product with the key scale inside the fma
                        float x0 = 0.0f, x1 = 0.0f;
                        fma2_rn(x0, x1, dv[hh * ITC_G + g], dv[hh * ITC_G + g + 1], sq[h * ITC_G + g], sq[h * ITC_G + g + 1]);
                        fma2_rn(de, dod, skf[g], skf[g + 1], x0, x1);
                    }
                    S = __fmaf_rn(ww[h], fmaxf(de + dod, 0.0f), S);
                }
            }
            const int i = t * ITC_TILE + r, e = c0 + i;
            const bool valid = i < n_loc;
            const float lb = valid ? S - E : -INFINITY, ub = valid ? S + E : -INFINITY;
            if (valid) ub_q[e] = ub;
            // the largest lower-bound key of each aligned group of 8 entries
            unsigned int km = f32_key(lb);
#pragma unroll
            for (int o2 = 1; o2 < 8; o2 <<= 1) km = max(km, __shfl_xor_sync(0xffffffffu, km, o2));
            if ((lane & 7) == 0) wm_q[e >> 3] = km;
            if (bsh) {
                float lbb = lb, ubb = ub;
                for (int o2 = 1; o2 < bsh; o2 <<= 1) {
                    lbb = fmaxf(lbb, __shfl_xor_sync(0xffffffffu, lbb, o2));
                    ubb = fmaxf(ubb, __shfl_xor_sync(0xffffffffu, ubb, o2));
                }
                if ((lane & (bsh - 1)) == 0 && e < n_elig) blu_q[e / bsh] = make_float2(lbb, ubb);
            }
        }
    }
    if (!ok) atomicExch(err, 1);
    umma::fence_before();
    __syncthreads();
    if (warp == 0) {
        umma::fence_after();
        umma::tmem_dealloc(tmem, 128);
    }
}

// decode (one query per block), d_I = 128, 8 heads; an HSI pool of blocks of a power of two up to 32
bool scan_tc_supported(int d_idx, int H, int QB, int pool_blocks, int bs) {
    return d_idx == ITC_DI && QB == 1 && H == ITC_H && (pool_blocks == 0 || (bs >= 2 && bs <= 32 && (bs & (bs - 1)) == 0));
}

cudaError_t launch_scan_full_tc(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                                const float* w_head, int n_q, const int64_t* q_pos, int q0, int n_qc, int H,
                                int pool_blocks, int bs, unsigned int* wmk, float2* lu, float2* blu, int list_len,
                                int* err, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(k_scan_full_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)IS_DYN);
    if (e != cudaSuccess) return e;
    dim3 grid((c.capacity + ITC_E - 1) / ITC_E, n_qc, c.batch);
    launch_k(k_scan_full_tc, grid, ITC_THREADS, IS_DYN, st, c.ikey_codes, c.ikey_scales, c.capacity, iq_codes, iq_scales, w_head,
                                              q_pos, n_q, q0, n_qc, H, pool_blocks > 0 ? bs : 0, wmk, lu, blu,
                                              list_len, err, (int)c.ratio);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa2

// Full indexer scan on the tensor cores ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の
// 限界を押し広げる", §2.3.1 lightweight indexer over FP4 keys).
//
// For one query and a chunk of its entries (a multiple of 128, sized so that
// the blocks fill two waves of the GPU), 128 entries at a time:
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
// Warp roles (320 threads): warps 0-7 epilogue in two groups of four that take
// alternate tiles (in a group one TMEM lane = one entry), warp 8 lane 0 issues
// the MMAs, warp 9 lane 0 the copies.  A tile's key codes come in one tensor
// copy (TMA) whose 4-bit data type spreads every 8 packed bytes into the low
// half of a 16-byte unit, which is the MMA's operand layout (the high halves
// were zeroed once and the copy leaves them alone); its scales come in a 1-D
// bulk copy.  Five operand slots, eight scale slots and four TMEM accumulators
// let the copies, MMAs and epilogues overlap, and an operand slot is refilled
// as soon as its MMAs are done.
#include <cuda.h>
#include "indexer_common.cuh"
#include "umma.cuh"

namespace csa2 {

constexpr int ITC_TILE = 128;
constexpr int ITC_NA = 5;                   // MMA operand slots (filled by the tensor copy)
constexpr int ITC_NS = 8;                   // key-scale slots
constexpr int ITC_ND = 4;                   // TMEM accumulators
constexpr int ITC_DI = 128;
constexpr int ITC_G = ITC_DI / 16;
constexpr int ITC_THREADS = 320;
constexpr int ITC_MMAW = 8, ITC_COPYW = 9;  // warps 0-7 epilogue (two groups of four)
constexpr int ITC_H = 8;                    // indexer heads taken by this kernel
constexpr int ITC_N = ITC_H * ITC_G;        // MMA N: one column per (head, group)
// shared memory (from the 1024-aligned base)
constexpr uint32_t IS_B = 0;                                  // query operand, 64 rows x 128 B
constexpr uint32_t IS_A = ITC_N * 128;                        // operand slots, 128 rows x 128 B each
constexpr uint32_t A_SLOT = ITC_TILE * 128;
constexpr uint32_t IS_S = IS_A + ITC_NA * A_SLOT;             // scale slots, 8 B per row
constexpr uint32_t S_SLOT = ITC_TILE * ITC_G;
constexpr uint32_t IS_Q = IS_S + ITC_NS * S_SLOT;             // sq [H][G] floats + w [H]
constexpr uint32_t IS_END = IS_Q + 512;
// two blocks per SM: both blocks' shared memory (with the 1 KB the system keeps per block) fits the SM's 228 KB
static_assert(2 * (IS_END + 1024 + 512 + 1024) <= 228 * 1024, "two blocks per SM");
constexpr uint32_t IS_DYN = IS_END + 1024;
constexpr uint32_t TMA_TX = ITC_TILE * (ITC_DI / 2);          // bytes one tensor copy delivers (the packed codes)

__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t unit) { return row * 128 + ((unit ^ (row & 7)) << 4); }

// one 128-row box of the key-code tensor (rows y .. y+127) into an operand slot; rows past the
// end of the tensor are filled with zeros
__device__ __forceinline__ void tma_codes(uint32_t dst, const CUtensorMap* tm, int y, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(y), "r"(mbar)
        : "memory");
}

// The outputs for query slab `slab` (row stride list_len): dense_ub(lu, slab, list_len)[e] = the
// upper bound of entry e (entries 0 .. n_elig-1), wmk[e / 8] = the largest lower-bound key of
// entries e .. e+7 (f32_key order; the key of -inf when none is eligible), blu[e / bs] = the bounds
// of HSI block e / bs (bs a power of two up to 32; bs == 0: no blocks).  `tmap` describes the key
// codes of all sequences as one tensor of batch * capacity rows of d_I 4-bit values.
__global__ void __launch_bounds__(ITC_THREADS, 2) k_scan_full_tc(
    const __grid_constant__ CUtensorMap tmap, const uint8_t* __restrict__ ks_all, int capacity,
    const uint8_t* __restrict__ iq_codes, const uint8_t* __restrict__ iq_scales, const float* __restrict__ w_head,
    const int64_t* __restrict__ q_pos, int n_q, int q0, int n_qc, int H, int bs, unsigned int* __restrict__ wmk,
    float2* __restrict__ lu, float2* __restrict__ blu, int list_len, int* __restrict__ err, int ratio, int chunk) {
    pdl_wait();             // the selection that follows is let in only as the scan's blocks exit
    extern __shared__ uint8_t dyn[];
    __shared__ __align__(8) unsigned long long bar_full[ITC_NA], bar_afree[ITC_NA], bar_sfull[ITC_NS],
        bar_sfree[ITC_NS], bar_dfull[ITC_ND], bar_dfree[ITC_ND];
    __shared__ uint32_t tmem_base;
    __shared__ int s_nel;

    const uint32_t raw = umma::smem_u32(dyn);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = dyn + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, ql = blockIdx.y;
    const int64_t gq = (int64_t)b * n_q + q0 + ql;
    const int64_t slab = (int64_t)b * n_qc + ql;
    const int c0 = blockIdx.x * chunk;               // this block's entries: [c0, c0 + chunk)
    constexpr int N = ITC_N;
    auto sa = [](const void* p) { return umma::smem_u32(p); };

    if (tid == 0) {
        s_nel = n_elig_of(q_pos[gq], capacity, ratio);
        for (int i = 0; i < ITC_NA; ++i) {
            umma::mbar_init(sa(&bar_full[i]), 1);
            umma::mbar_init(sa(&bar_afree[i]), 1);
        }
        for (int i = 0; i < ITC_NS; ++i) {
            umma::mbar_init(sa(&bar_sfull[i]), 1);
            umma::mbar_init(sa(&bar_sfree[i]), 4);         // one arrival per epilogue warp of the group
        }
        for (int i = 0; i < ITC_ND; ++i) {
            umma::mbar_init(sa(&bar_dfull[i]), 1);
            umma::mbar_init(sa(&bar_dfree[i]), 4);
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
    // zero the operand slots once: the tensor copies write only the low half of every 16-byte unit
    for (int i = tid; i < ITC_NA * ITC_TILE * 8; i += blockDim.x)
        reinterpret_cast<uint4*>(sm + IS_A)[i] = make_uint4(0, 0, 0, 0);
    if (warp == 0) umma::tmem_alloc(sa(&tmem_base), 64 * ITC_ND);
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = tmem_base;
    const int n_elig = s_nel;
    const int n_loc = min(max(n_elig - c0, 0), chunk);
    const int n_tiles = (n_loc + ITC_TILE - 1) / ITC_TILE;
    bool ok = true;
    int n_issued = 0;                                       // tiles the copy issuer started

    // scale rows are 8 bytes; a bulk copy needs a 16-byte aligned source
    const uint8_t* ks_seq = ks_all + ((int64_t)b * capacity + c0) * ITC_G;
    const bool bulk_scales = ((reinterpret_cast<uintptr_t>(ks_seq) & 15u) == 0);
    if (warp == ITC_COPYW) {
        // ---- copy issuer: tile t into operand slot t % NA and scale slot t % NS once both are free
        if (lane == 0) {
            for (int t = 0; t < n_tiles && ok; ++t) {
                const int a = t % ITC_NA, s = t % ITC_NS;
                if (t >= ITC_NA) ok &= umma::mbar_wait(sa(&bar_afree[a]), ((t / ITC_NA) - 1) & 1);
                if (t >= ITC_NS && ok) ok &= umma::mbar_wait(sa(&bar_sfree[s]), ((t / ITC_NS) - 1) & 1);
                if (!ok) break;
                const int e0 = c0 + t * ITC_TILE;
                const int rows = min(ITC_TILE, n_elig - e0);
                const uint32_t sbytes = bulk_scales ? (uint32_t)(rows & ~1) * ITC_G : 0u;
                umma::mbar_arrive_expect_tx(sa(&bar_full[a]), TMA_TX);
                tma_codes(base + IS_A + a * A_SLOT, &tmap, b * capacity + e0, sa(&bar_full[a]));
                umma::mbar_arrive_expect_tx(sa(&bar_sfull[s]), sbytes);
                if (sbytes)
                    umma::bulk_g2s(base + IS_S + s * S_SLOT, ks_all + ((int64_t)b * capacity + e0) * ITC_G, sbytes,
                                   sa(&bar_sfull[s]));
                n_issued = t + 1;
            }
        }
    } else if (warp == ITC_MMAW) {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (5u << 7) | (5u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            for (int t = 0; t < n_tiles && ok; ++t) {
                const int a = t % ITC_NA, d = t % ITC_ND;
                ok &= umma::mbar_wait(sa(&bar_full[a]), (t / ITC_NA) & 1);
                if (t >= ITC_ND && ok) ok &= umma::mbar_wait(sa(&bar_dfree[d]), ((t / ITC_ND) - 1) & 1);
                if (!ok) break;
                umma::fence_after();
#pragma unroll
                for (int ks = 0; ks < ITC_DI / 32; ++ks) {
                    const uint64_t ad = umma::desc(base + IS_A + a * A_SLOT + ks * 32, 16, 1024, umma::LAYOUT_SW128);
                    const uint64_t bd = umma::desc(base + IS_B + ks * 32, 16, 1024, umma::LAYOUT_SW128);
                    asm volatile(
                        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(tmem + 64 * d),
                        "l"(ad), "l"(bd), "r"(idesc), "r"(ks));
                }
                umma::commit(sa(&bar_dfull[d]));
                umma::commit(sa(&bar_afree[a]));     // the operand slot is free once these MMAs are done
            }
        }
    } else if (warp < ITC_MMAW) {
        // ---- epilogue: one entry per thread
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
        // warp w takes the tiles t with t % 2 == w / 4, lane quarter w % 4
        const int eg = warp >> 2, wq = warp & 3;
        for (int t = eg; t < n_tiles; t += 2) {
            const int s = t % ITC_NS, d = t % ITC_ND;
            const int r = wq * 32 + lane;               // row of the tile = TMEM lane
            const int e0 = c0 + t * ITC_TILE;
            const int rows = min(ITC_TILE, n_elig - e0);
            uint2 skw = make_uint2(0, 0);
            if (ok) ok &= umma::mbar_wait_fast(sa(&bar_sfull[s]), (t / ITC_NS) & 1);
            if (bulk_scales && r < (rows & ~1))
                skw = *reinterpret_cast<const uint2*>(sm + IS_S + s * S_SLOT + r * 8);
            else if (r < rows)
                skw = __ldg(reinterpret_cast<const uint2*>(ks_all + ((int64_t)b * capacity + e0 + r) * ITC_G));
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(sa(&bar_sfree[s]));
            float skf[ITC_G];
#pragma unroll
            for (int p = 0; p < ITC_G / 2; ++p) {
                const float2 f = e4m3_pair_f32(((p < 2 ? skw.x : skw.y) >> (16 * (p & 1))) & 0xffffu);
                skf[2 * p] = f.x;
                skf[2 * p + 1] = f.y;
            }
            float E = 0.0f;
#pragma unroll
            for (int g = 0; g < ITC_G; ++g) E = __fmaf_rn(cb[g], skf[g], E);
            // the group sums in two halves of four heads (32 columns), to keep registers low
            if (ok) ok &= umma::mbar_wait_fast(sa(&bar_dfull[d]), (t / ITC_ND) & 1);
            umma::fence_after();
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
                    __syncwarp();
                    if (lane == 0) umma::mbar_arrive(sa(&bar_dfree[d]));
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
    // a copy issuer that gave up may have copies in flight into this block's shared memory: let
    // the last one issued into each slot land (bounded) before the block exits
    if (warp == ITC_COPYW && lane == 0 && !ok) {
        for (int t = max(0, n_issued - ITC_NS); t < n_issued; ++t) {
            if (t >= n_issued - ITC_NA) umma::mbar_wait(sa(&bar_full[t % ITC_NA]), (t / ITC_NA) & 1, 1u << 16);
            umma::mbar_wait(sa(&bar_sfull[t % ITC_NS]), (t / ITC_NS) & 1, 1u << 16);
        }
    }
    if (!ok) atomicExch(err, 1);
    umma::fence_before();
    __syncthreads();
    if (warp == 0) {
        umma::fence_after();
        umma::tmem_dealloc(tmem, 64 * ITC_ND);
    }
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime (no link to libcuda)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// decode (one query per block), d_I = 128, 8 heads; an HSI pool of blocks of a power of two up to
// 32; the key codes 32-byte aligned (the tensor copy of packed 4-bit data wants it)
bool scan_tc_supported(int d_idx, int H, int QB, int pool_blocks, int bs, const csa2_cache& c) {
    return d_idx == ITC_DI && QB == 1 && H == ITC_H && (pool_blocks == 0 || (bs >= 2 && bs <= 32 && (bs & (bs - 1)) == 0)) &&
           (reinterpret_cast<uintptr_t>(c.ikey_codes) & 31u) == 0 && (int64_t)c.batch * c.capacity < (1ll << 31) &&
           encode_tiled() != nullptr;
}

cudaError_t launch_scan_full_tc(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                                const float* w_head, int n_q, const int64_t* q_pos, int q0, int n_qc, int H,
                                int pool_blocks, int bs, unsigned int* wmk, float2* lu, float2* blu, int list_len,
                                int* err, cudaStream_t st) {
    const EncodeTiledFn enc = encode_tiled();
    if (enc == nullptr) return cudaErrorNotSupported;
    // the key codes of every sequence as one 2-D tensor: batch * capacity rows of d_I 4-bit values
    // (d_I / 2 bytes); a box is one tile of 128 rows, spread in shared memory to the MMA layout
    CUtensorMap tm;
    const cuuint64_t dims[2] = {(cuuint64_t)ITC_DI, (cuuint64_t)c.batch * (cuuint64_t)c.capacity};
    const cuuint64_t strides[1] = {(cuuint64_t)(ITC_DI / 2)};
    const cuuint32_t box[2] = {(cuuint32_t)ITC_DI, (cuuint32_t)ITC_TILE};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, static_cast<void*>(c.ikey_codes), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_scan_full_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)IS_DYN);
    if (e != cudaSuccess) return e;
    // chunk size: the queries' tiles split into as many chunks as fill two waves of resident blocks
    // (fewer, longer blocks pay the pipeline fill less often; whole waves leave no thin tail)
    int dev = 0, n_sm = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_scan_full_tc, ITC_THREADS, IS_DYN)) != cudaSuccess)
        return e;
    const int64_t tiles_q = (c.capacity + ITC_TILE - 1) / ITC_TILE;
    const int64_t slabs = (int64_t)n_qc * c.batch;
    int64_t chunks_q = (2 * (int64_t)(per_sm > 0 ? per_sm : 1) * n_sm) / (slabs > 0 ? slabs : 1);
    chunks_q = chunks_q < 1 ? 1 : (chunks_q > tiles_q ? tiles_q : chunks_q);
    const int chunk = (int)((tiles_q + chunks_q - 1) / chunks_q) * ITC_TILE;
    dim3 grid((unsigned)((c.capacity + chunk - 1) / chunk), n_qc, c.batch);
    launch_k(k_scan_full_tc, grid, ITC_THREADS, IS_DYN, st, tm, (const uint8_t*)c.ikey_scales, c.capacity, iq_codes,
             iq_scales, w_head, q_pos, n_q, q0, n_qc, H, pool_blocks > 0 ? bs : 0, wmk, lu, blu, list_len, err,
             (int)c.ratio, chunk);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa2

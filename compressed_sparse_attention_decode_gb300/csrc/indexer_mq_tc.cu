// Multi-query Full indexer scan on the tensor cores, for a chunked prefill
// ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる", §2.3.1 lightweight
// indexer over FP4 keys; §2.3.4 a Full layer scores every causally visible entry).
//
// One block takes MQ_QB = 4 consecutive queries of the chunk and every entry
// any of them may read, 128 entries a tile.  Per 16-dim group g, one MMA
// (kind::f16, M = 128 entries, N = 32 (query, head) rows, K = 16):
//   A = the E2M1 key codes of the tile as fp16 (exact)
//   B = the query values q = code x scale as fp16 (exact: an E2M1 value times
//       an E4M3 scale has at most 6 significant bits and lies in [2^-10, 2688])
//   D_g[e][(q,h)] = sum over the group's 16 dims of k_code q   (fp32 in TMEM)
// Every product is a multiple of a quarter of the query scale and the sum
// stays below 2^12 such quarters, so D_g is exact; it is the group sum times
// the query's group scale.  The epilogue forms every (entry, query) score S~
// exactly as the single-query scans do (per head, the key-scaled terms t_g
// added in group order, then the head weights), and a bound E on its rounding
// error: the scans bound it by fac * sum_h |w_h| sum_g |t_gh|, where fac
// holds a factor of two to spare; with every |x| = |group sum| * s_q at most
// 576 s_q (x the MMA outputs), that sum is at most sum_g C_g s_kg, with
// C_g = fac * 576 * sum_h |w_h| s_qhg fixed per query (the decode scan's
// bound): eight multiply-adds per pair instead of 64 absolute values.  Two
// accumulators of 8 x 32 columns.
//
// Which entries go on to the exact selection: those whose upper bound S~+E
// reaches a threshold tau_q that lies below the query's k-th largest lower
// bound.  tau_q comes from a sample: the block first scores up to 32 tiles
// spread evenly over the range, and takes the value that the lower bounds of
// about 2k of all entries should reach, judging by the sample; then it scores
// every tile, forwards by tau_q and counts the lower bounds that reach tau_q.
// If fewer than k do, tau_q was too high for that query: its list is cleared
// and every tile is scored once more with no threshold.  Whatever the data,
// the forwarded set holds every entry the exact top-k can contain.
//
// Warps (704 threads): 0-15 epilogue (warp w: TMEM lane quarter w%4, query
// w/4; four warps per scheduler hide the TMEM and arithmetic latencies), 16-19
// convert the packed codes to the fp16 MMA layout and decode each entry's key
// scales once (to fp32 in shared memory), 20 lane 0 issues
// the MMAs, 21 lane 0 the 1-D bulk copies of each tile's contiguous key rows
// (four tiles in flight).
#include "indexer_common.cuh"
#include "umma.cuh"

namespace csa2 {

constexpr int MQ_QB = 4;
constexpr int MQ_TILE = 128;
constexpr int MQ_DI = 128;
constexpr int MQ_G = MQ_DI / 16;
constexpr int MQ_H = 8;
constexpr int MQ_NQH = MQ_QB * MQ_H;                      // 32: MMA N, one column per (query, head)
constexpr int MQ_NR = 4;                                  // raw staging slots
constexpr int MQ_NA = 2;                                  // MMA-layout A slots
constexpr int MQ_SAMPLE_TILES = 32;
constexpr int MQ_THREADS = 704;
constexpr int MQ_EPI = 512;                               // warps 0-15
constexpr int MQ_W_XF = 16, MQ_W_MMA = 20, MQ_W_COPY = 21;
constexpr int MQ_XF = 128;                                // warps 16-19
constexpr uint32_t MQ_RAW_SLOT = MQ_TILE * (MQ_DI / 2) + MQ_TILE * 8;          // codes 8 KB + scales 1 KB
// fp16 operands, K-major, 128-byte swizzle: slabs of 64 dims (128 B per row)
constexpr uint32_t MQ_ASLAB = MQ_TILE * 128;                                    // 16 KB
constexpr uint32_t MQ_BSLAB = MQ_NQH * 128;                                     // 4 KB
constexpr uint32_t MQS_A = 0;                                                   // 2 slots x 2 slabs
constexpr uint32_t MQS_B = MQS_A + MQ_NA * 2 * MQ_ASLAB;                        // 2 slabs
constexpr uint32_t MQS_RAW = MQS_B + 2 * MQ_BSLAB;                              // 4 x 9 KB
constexpr uint32_t MQS_SAMP = MQS_RAW + MQ_NR * MQ_RAW_SLOT;                    // [QB][32 x 128] lower bounds
constexpr uint32_t MQS_SK = MQS_SAMP + MQ_QB * MQ_SAMPLE_TILES * MQ_TILE * 4;   // per raw slot: [128][8] scales
constexpr uint32_t MQ_SK_SLOT = MQ_TILE * MQ_G * 4;
constexpr uint32_t MQS_Q = MQS_SK + MQ_NR * MQ_SK_SLOT;                         // w [QB][8], C_g [QB][8]
constexpr uint32_t MQS_END = MQS_Q + MQ_QB * (MQ_H + MQ_G) * 4;
constexpr uint32_t MQS_DYN = MQS_END + 1024;

__device__ __forceinline__ uint32_t mq_swz(uint32_t row, uint32_t unit) { return row * 128 + ((unit ^ (row & 7)) << 4); }
// eight E2M1 codes (one 32-bit word, low nibble first) to four fp16 pairs, exactly
__device__ __forceinline__ void mq_e2m1x8(uint32_t w, uint32_t* o) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}
// two E4M3 bytes (low byte -> low half) to an fp16 pair, exactly
__device__ __forceinline__ __half2 mq_e4m3x2_h2(uint32_t two) {
    uint32_t r;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(r) : "r"(two));
    return *reinterpret_cast<__half2*>(&r);
}
// an E4M3 byte to an fp16 pair holding it twice, exactly
__device__ __forceinline__ __half2 mq_e4m3_h2(uint32_t byte) {
    uint32_t r;
    const uint32_t two = byte | (byte << 8);
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(r) : "r"(two));
    return *reinterpret_cast<__half2*>(&r);
}

__global__ void __launch_bounds__(MQ_THREADS, 1) k_scan_mq_tc(
    const uint8_t* __restrict__ kc_all, const uint8_t* __restrict__ ks_all, int capacity,
    const uint8_t* __restrict__ iq_codes, const uint8_t* __restrict__ iq_scales, const float* __restrict__ w_head,
    const int64_t* __restrict__ q_pos, int n_q, int q0, int n_qc, int k, int* __restrict__ counts,
    int* __restrict__ cid, float2* __restrict__ clu, int list_len, int* __restrict__ err, int ratio) {
    pdl_wait();
    extern __shared__ uint8_t dyn[];
    __shared__ __align__(8) unsigned long long bar_rfull[MQ_NR], bar_rfree[MQ_NR], bar_sfull[MQ_NR], bar_afull[MQ_NA],
        bar_afree[MQ_NA], bar_dfull[2], bar_dfree[2];
    __shared__ uint32_t tmem_base;
    __shared__ int s_nel[MQ_QB], s_cnt[MQ_QB], s_retry[MQ_QB + 1];
    __shared__ uint32_t s_tau[MQ_QB];
    __shared__ int s_hist[256], s_pick[2];

    const uint32_t raw = umma::smem_u32(dyn);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = dyn + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y, qa = blockIdx.x * MQ_QB;
    const int nqb = min(MQ_QB, n_qc - qa);

    if (tid < MQ_QB) {
        s_nel[tid] = tid < nqb ? n_elig_of(q_pos[(int64_t)b * n_q + q0 + qa + tid], capacity, ratio) : 0;
        s_cnt[tid] = 0;
        s_tau[tid] = 0u;                 // key 0: every eligible entry passes
        s_retry[tid] = 0;
    }
    if (tid == 0) {
        s_retry[MQ_QB] = 0;
        for (int i = 0; i < MQ_NR; ++i) {
            umma::mbar_init(umma::smem_u32(&bar_rfull[i]), 1);
            umma::mbar_init(umma::smem_u32(&bar_rfree[i]), MQ_EPI);
            umma::mbar_init(umma::smem_u32(&bar_sfull[i]), MQ_XF);
        }
        for (int i = 0; i < MQ_NA; ++i) {
            umma::mbar_init(umma::smem_u32(&bar_afull[i]), MQ_XF);
            umma::mbar_init(umma::smem_u32(&bar_afree[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            umma::mbar_init(umma::smem_u32(&bar_dfull[i]), 1);
            umma::mbar_init(umma::smem_u32(&bar_dfree[i]), MQ_EPI);
        }
        umma::fence_mbar_init();
    }
    // query operand: row n = (q, h), the 128 values code x scale of query q's head h in fp16;
    // unit u (8 dims) of a row comes from one code word and its group's scale
    for (int i = tid; i < MQ_NQH * 16; i += MQ_THREADS) {
        const int n = i >> 4, u = i & 15;
        const int q = n >> 3, h = n & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (q < nqb) {
            const int64_t gq = (int64_t)b * n_q + q0 + qa + q;
            const uint32_t w = *reinterpret_cast<const uint32_t*>(iq_codes + (gq * MQ_H + h) * (MQ_DI / 2) + u * 4);
            const __half2 s2 = mq_e4m3_h2(iq_scales[(gq * MQ_H + h) * MQ_G + (u >> 1)]);
            uint32_t f[4];
            mq_e2m1x8(w, f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __half2 x = __hmul2(*reinterpret_cast<__half2*>(&f[j]), s2);
                f[j] = *reinterpret_cast<uint32_t*>(&x);
            }
            v = make_uint4(f[0], f[1], f[2], f[3]);
        }
        *reinterpret_cast<uint4*>(sm + MQS_B + (u >> 3) * MQ_BSLAB + mq_swz(n, u & 7)) = v;
    }
    float* ww = reinterpret_cast<float*>(sm + MQS_Q);                // [QB][8]
    for (int i = tid; i < MQ_QB * MQ_H; i += MQ_THREADS) {
        const int q = i >> 3;
        ww[i] = q < nqb ? w_head[((int64_t)b * n_q + q0 + qa + q) * MQ_H + (i & 7)] : 0.0f;
    }
    // per query and group: C_g = fac * 576 * sum_h |w_h| s_qhg (rounded up, times 1 + 2^-10 for the
    // rounding of the 8-term sum below): every |x| = |group sum| * s_q <= 576 s_q, so
    // sum_g C_g s_kg bounds fac * sum_h |w_h| sum_g |x s_k|, the error of S~
    float* cq = ww + MQ_QB * MQ_H;                                   // [QB][8]
    if (tid < MQ_QB * MQ_G) {
        const int q = tid >> 3, g = tid & 7;
        float a = 0.0f;
        if (q < nqb) {
            const int64_t gq = (int64_t)b * n_q + q0 + qa + q;
            for (int h = 0; h < MQ_H; ++h)
                a = __fmaf_ru(fabsf(w_head[gq * MQ_H + h]), e4m3_to_f32(iq_scales[(gq * MQ_H + h) * MQ_G + g]), a);
        }
        cq[tid] = __fmul_ru(__fmul_ru(a, 576.0f * bound_factor(MQ_H, MQ_DI)), 1.0f + 0x1p-10f);
    }
    if (warp == 0) umma::tmem_alloc(umma::smem_u32(&tmem_base), 512);
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = tmem_base;

    int nmax = 0;
    bool need_tau = false;
    for (int q = 0; q < nqb; ++q) {
        nmax = max(nmax, s_nel[q]);
        need_tau |= s_nel[q] > 4 * k;
    }
    const int n_tiles = (nmax + MQ_TILE - 1) / MQ_TILE;
    const int stride = max(1, (n_tiles + MQ_SAMPLE_TILES - 1) / MQ_SAMPLE_TILES);
    const int n_s0 = need_tau ? (n_tiles + stride - 1) / stride : 0;    // sample tiles 0, stride, 2 stride, ..
    // scale rows are 8 bytes; a bulk copy needs a 16-byte aligned source
    const bool bulk_scales = ((reinterpret_cast<uintptr_t>(ks_all + (int64_t)b * capacity * MQ_G) & 15u) == 0);
    float* samp = reinterpret_cast<float*>(sm + MQS_SAMP);
    bool ok = true;
    int v_end = 0;                       // virtual tiles issued so far (all roles agree)

    // phase 0: the sample tiles; 1: every tile, forwarded by tau; 2: every tile again, for the
    // queries whose tau proved too high, forwarded with no threshold
    for (int phase = 0; phase < 3; ++phase) {
        const int v0 = v_end;
        const int nv = phase == 0 ? n_s0 : n_tiles;
        v_end = v0 + nv;
        auto tile_of = [&](int v) { return phase == 0 ? (v - v0) * stride : v - v0; };
        if (warp == MQ_W_COPY) {
            // ---- bulk-copy issuer
            if (lane == 0) {
                for (int v = v0; v < v_end && ok; ++v) {
                    const int r = v % MQ_NR;
                    if (v >= MQ_NR) ok &= umma::mbar_wait(umma::smem_u32(&bar_rfree[r]), ((v / MQ_NR) - 1) & 1);
                    if (!ok) break;
                    const int e0 = tile_of(v) * MQ_TILE;
                    const int rows = min(MQ_TILE, nmax - e0);
                    const uint32_t cb = (uint32_t)rows * (MQ_DI / 2);
                    const uint32_t sbytes = bulk_scales ? (uint32_t)(rows & ~1) * MQ_G : 0u;
                    const uint32_t mb = umma::smem_u32(&bar_rfull[r]);
                    const uint32_t dst = base + MQS_RAW + r * MQ_RAW_SLOT;
                    umma::mbar_arrive_expect_tx(mb, cb + sbytes);
                    umma::bulk_g2s(dst, kc_all + ((int64_t)b * capacity + e0) * (MQ_DI / 2), cb, mb);
                    if (sbytes)
                        umma::bulk_g2s(dst + MQ_TILE * (MQ_DI / 2), ks_all + ((int64_t)b * capacity + e0) * MQ_G, sbytes,
                                       mb);
                }
            }
        } else if (warp >= MQ_W_XF && warp < MQ_W_XF + MQ_XF / 32) {
            // ---- codes to fp16: raw chunk c (16 bytes) = row c/4, dims 32(c%4) .. +31
            const int xt = tid - 32 * MQ_W_XF;
            for (int v = v0; v < v_end && ok; ++v) {
                const int r = v % MQ_NR, a = v % MQ_NA;
                ok &= umma::mbar_wait(umma::smem_u32(&bar_rfull[r]), (v / MQ_NR) & 1);
                if (v >= MQ_NA) ok &= umma::mbar_wait(umma::smem_u32(&bar_afree[a]), ((v / MQ_NA) - 1) & 1);
                if (!ok) break;
                const uint4* rw = reinterpret_cast<const uint4*>(sm + MQS_RAW + r * MQ_RAW_SLOT);
                uint8_t* as = sm + MQS_A + a * (2 * MQ_ASLAB);
#pragma unroll 2
                for (int c = xt; c < MQ_TILE * 4; c += MQ_XF) {
                    const int row = c >> 2, j = c & 3;
                    const uint4 x = rw[c];
                    const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
                    uint8_t* slab = as + (j >> 1) * MQ_ASLAB;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t f[4];
                        mq_e2m1x8(wd[i], f);
                        *reinterpret_cast<uint4*>(slab + mq_swz(row, (j & 1) * 4 + i)) = make_uint4(f[0], f[1], f[2], f[3]);
                    }
                }
                umma::fence_proxy_async();
                umma::mbar_arrive(umma::smem_u32(&bar_afull[a]));
                // entry xt's eight key scales as fp32, for the epilogue
                {
                    const int e0 = tile_of(v) * MQ_TILE;
                    const int rows = min(MQ_TILE, nmax - e0);
                    uint2 skw = make_uint2(0, 0);
                    if (bulk_scales && xt < (rows & ~1))
                        skw = *reinterpret_cast<const uint2*>(sm + MQS_RAW + r * MQ_RAW_SLOT + MQ_TILE * (MQ_DI / 2) + xt * 8);
                    else if (xt < rows)
                        skw = __ldg(reinterpret_cast<const uint2*>(ks_all + ((int64_t)b * capacity + e0 + xt) * MQ_G));
                    float sk[MQ_G];
#pragma unroll
                    for (int g = 0; g < MQ_G; g += 2) {
                        const __half2 h2 = mq_e4m3x2_h2(((g < 4 ? skw.x : skw.y) >> (8 * (g & 3))) & 0xffffu);
                        sk[g] = __low2float(h2);
                        sk[g + 1] = __high2float(h2);
                    }
                    float* dst = reinterpret_cast<float*>(sm + MQS_SK + r * MQ_SK_SLOT);
                    reinterpret_cast<float4*>(dst)[2 * xt] = make_float4(sk[0], sk[1], sk[2], sk[3]);
                    reinterpret_cast<float4*>(dst)[2 * xt + 1] = make_float4(sk[4], sk[5], sk[6], sk[7]);
                    umma::mbar_arrive(umma::smem_u32(&bar_sfull[r]));
                }
            }
        } else if (warp == MQ_W_MMA) {
            // ---- MMA issuer
            if (lane == 0) {
                const uint32_t idesc = umma::idesc_f16(MQ_TILE, MQ_NQH, 0, 0);
                for (int v = v0; v < v_end && ok; ++v) {
                    const int s = v % MQ_NA, d = v & 1;
                    ok &= umma::mbar_wait(umma::smem_u32(&bar_afull[s]), (v / MQ_NA) & 1);
                    if (v >= 2) ok &= umma::mbar_wait(umma::smem_u32(&bar_dfree[d]), ((v >> 1) - 1) & 1);
                    if (!ok) break;
                    umma::fence_after();
                    // group g: dims 16g .. 16g+15 = slab g/4, bytes 32(g%4) of every row; its own
                    // 32 accumulator columns, never accumulated into
#pragma unroll
                    for (int g = 0; g < MQ_G; ++g) {
                        const uint64_t ad = umma::desc(base + MQS_A + s * (2 * MQ_ASLAB) + (g >> 2) * MQ_ASLAB + (g & 3) * 32,
                                                       16, 1024, umma::LAYOUT_SW128);
                        const uint64_t bd = umma::desc(base + MQS_B + (g >> 2) * MQ_BSLAB + (g & 3) * 32, 16, 1024,
                                                       umma::LAYOUT_SW128);
                        umma::mma_f16(tmem + 256 * d + MQ_NQH * g, ad, bd, idesc, 0u);
                    }
                    umma::commit(umma::smem_u32(&bar_dfull[d]));
                    umma::commit(umma::smem_u32(&bar_afree[s]));
                }
            }
        } else {
            // ---- epilogue: one entry (TMEM lane) and one query per thread
            const int qd = warp & 3, qi = warp >> 2;
            const int r = qd * 32 + lane;
            const bool live = qi < nqb;                       // warp-uniform
            const int nel = s_nel[qi];
            const float* wq = ww + qi * MQ_H;
            const float* cg = cq + qi * MQ_G;
            const int64_t slab = (int64_t)b * n_qc + qa + qi;
            // tau as a float: key 0 (no threshold) is -inf; every other key comes from a finite value
            const uint32_t tau_key = s_tau[qi];
            float tau = key_value(tau_key);
            if (tau_key == 0u || !(tau == tau)) tau = -INFINITY;
            const bool retry = s_retry[qi] != 0;
            int cge = 0;
            for (int v = v0; v < v_end && ok; ++v) {
                const int rs = v % MQ_NR, d = v & 1;
                const int e0 = tile_of(v) * MQ_TILE;
                const int rows = min(MQ_TILE, nmax - e0);
                const int e = e0 + r;
                ok &= umma::mbar_wait(umma::smem_u32(&bar_dfull[d]), (v >> 1) & 1);
                ok &= umma::mbar_wait(umma::smem_u32(&bar_sfull[rs]), (v / MQ_NR) & 1);
                if (!ok) break;
                umma::fence_after();
                const float* skp = reinterpret_cast<const float*>(sm + MQS_SK + rs * MQ_SK_SLOT);
                const float4 s0 = reinterpret_cast<const float4*>(skp)[2 * r];
                const float4 s1 = reinterpret_cast<const float4*>(skp)[2 * r + 1];
                const float skf[MQ_G] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                umma::mbar_arrive(umma::smem_u32(&bar_rfree[rs]));
                // columns of group g, query qi: 32 g + 8 qi + h; two groups at a time, in order (each
                // head's sums still take the groups in order)
                const uint32_t tb = tmem + ((uint32_t)(qd * 32) << 16) + 256 * d + MQ_H * qi;
                float dd[MQ_H];
#pragma unroll
                for (int h = 0; h < MQ_H; ++h) dd[h] = 0.0f;
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    float dv[16];                              // [g][h]: the group sum times the query scale
#pragma unroll
                    for (int g = 0; g < 2; ++g) umma::tmem_ld8(tb + MQ_NQH * (2 * part + g), dv + MQ_H * g);
                    umma::tmem_wait_ld();
                    if (part == 3) {
                        umma::fence_before();
                        umma::mbar_arrive(umma::smem_u32(&bar_dfree[d]));
                    }
                    if (!live) continue;
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        const float sk = skf[2 * part + g];
#pragma unroll
                        for (int h = 0; h < MQ_H; h += 2) {
                            // x times the key scale is exact inside the fma: the same sums as adding
                            // t = (group sum) * (sq * sk) one by one; two heads per instruction
                            const float x0 = dv[g * MQ_H + h], x1 = dv[g * MQ_H + h + 1];
                            fma2_rn(dd[h], dd[h + 1], sk, sk, x0, x1);
                        }
                    }
                }
                if (!live) continue;
                float S = 0.0f, E = 0.0f;
#pragma unroll
                for (int h = 0; h < MQ_H; ++h) S = __fmaf_rn(wq[h], fmaxf(dd[h], 0.0f), S);
#pragma unroll
                for (int g = 0; g < MQ_G; ++g) E = __fmaf_rn(cg[g], skf[g], E);
                const float L = S - E, U = S + E;
                const bool elig = e < nel;
                if (phase == 0) {
                    samp[qi * (MQ_SAMPLE_TILES * MQ_TILE) + (v - v0) * MQ_TILE + r] = elig ? L : -INFINITY;
                } else {
                    const bool fwd = elig && (phase == 1 ? U >= tau : retry);
                    if (phase == 1) cge += (elig && L >= tau) ? 1 : 0;
                    const int pos = append_slot(fwd, counts + 2 * slab);
                    if (fwd) {
                        cid[slab * list_len + pos] = e;
                        clu[slab * list_len + pos] = make_float2(L, U);
                    }
                }
            }
            if (phase == 1 && live) {
                const int c = __reduce_add_sync(0xffffffffu, cge);
                if (lane == 0 && c) atomicAdd(&s_cnt[qi], c);
            }
        }
        __syncthreads();
        if (phase == 0 && need_tau) {
            // tau_q: a value at most the m-th largest sampled lower bound, m about 2k times the sampled
            // share of the query's entries (two 8-bit digits of the order-preserving key)
            for (int q = 0; q < nqb; ++q) {
                const int ne = s_nel[q];
                if (ne <= 4 * k) continue;                    // uniform: no threshold
                int ns = 0;
                for (int i = 0; i < n_s0; ++i) ns += max(0, min(MQ_TILE, ne - i * stride * MQ_TILE));
                const long long m_ll = ((long long)2 * k * ns + ne - 1) / ne;
                const int m = (int)max(1LL, min((long long)ns, m_ll));
                const float* sv = samp + q * (MQ_SAMPLE_TILES * MQ_TILE);
                const int n_all = n_s0 * MQ_TILE;
                uint32_t prefix = 0u;
                int mrem = m;
                for (int pass = 0; pass < 2; ++pass) {
                    for (int i = tid; i < 256; i += MQ_THREADS) s_hist[i] = 0;
                    __syncthreads();
                    for (int i = tid; i < n_all; i += MQ_THREADS) {
                        const uint32_t key = f32_key(sv[i]);
                        if (pass == 0) atomicAdd(&s_hist[key >> 24], 1);
                        else if ((key >> 24) == (prefix >> 24)) atomicAdd(&s_hist[(key >> 16) & 255u], 1);
                    }
                    __syncthreads();
                    if (tid == 0) {
                        int above = 0, bin = 255;
                        for (; bin > 0; --bin) {
                            if (above + s_hist[bin] >= mrem) break;
                            above += s_hist[bin];
                        }
                        s_pick[0] = bin;
                        s_pick[1] = mrem - above;
                    }
                    __syncthreads();
                    prefix |= (uint32_t)s_pick[0] << (pass == 0 ? 24 : 16);
                    mrem = s_pick[1];
                    __syncthreads();
                }
                if (tid == 0) s_tau[q] = prefix;
            }
            __syncthreads();
        }
        if (phase == 1) {
            if (tid < nqb) {
                const bool again = s_tau[tid] != 0u && s_cnt[tid] < k;
                s_retry[tid] = again ? 1 : 0;
                if (again) {
                    counts[2 * ((int64_t)b * n_qc + qa + tid)] = 0;
                    atomicOr(&s_retry[MQ_QB], 1);
                }
            }
            __syncthreads();
            if (!s_retry[MQ_QB]) break;
        }
    }
    // the copies issued are all consumed on the normal path; after a timeout, wait (bounded)
    // for the last ones before the block's shared memory is given up
    if (warp == MQ_W_COPY && lane == 0 && !ok) {
        for (int v = max(0, v_end - MQ_NR); v < v_end; ++v)
            umma::mbar_wait(umma::smem_u32(&bar_rfull[v % MQ_NR]), (v / MQ_NR) & 1, 1u << 16);
    }
    if (!ok) atomicExch(err, 1);
    umma::fence_before();
    __syncthreads();
    if (warp == 0) {
        umma::fence_after();
        umma::tmem_dealloc(tmem, 512);
    }
}

bool scan_mq_tc_supported(int d_idx, int H, int n_q, int pool_blocks) {
    return d_idx == MQ_DI && H == MQ_H && n_q >= MQ_QB && pool_blocks == 0;
}

cudaError_t launch_scan_mq_tc(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                              const float* w_head, int n_q, const int64_t* q_pos, int q0, int n_qc, int k, int* counts,
                              int* cid, float2* clu, int list_len, int* err, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(k_scan_mq_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MQS_DYN);
    if (e != cudaSuccess) return e;
    dim3 grid((n_qc + MQ_QB - 1) / MQ_QB, c.batch);
    launch_k(k_scan_mq_tc, grid, MQ_THREADS, MQS_DYN, st, c.ikey_codes, c.ikey_scales, c.capacity, iq_codes, iq_scales,
             w_head, q_pos, n_q, q0, n_qc, k, counts, cid, clu, list_len, err, (int)c.ratio);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa2

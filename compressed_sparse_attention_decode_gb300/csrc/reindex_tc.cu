// Reindex on the tensor cores: the indexer re-run on the Full layer's
// candidate pool, top k kept ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し
// 広げる", §2.3.2 Reindex mode, §2.3.4 HSI pool).  One launch per layer.
//
// A cluster of RT_CTAS blocks per query; block r takes pool slots
// [512 r, 512 r + 512) as four tiles of 128 (one slot per thread):
//   - each thread loads the key row of its slot (four 16-byte loads of codes,
//     one of scales) while the query is staged, then writes the row in the
//     kind::f8f6f4 operand layout (each 16-value group: 8 code bytes, 8 zero
//     bytes); the query's codes form a block-diagonal operand (row (head,
//     group) holds that head's codes of that group, zeros elsewhere);
//   - D = keys . query^T (M = 128 slots, N = 8 heads x 8 groups, K = 128) holds
//     the exact group sums in TMEM, from which every slot gets the same fp32
//     score as the scans, and the bound E = sum_g C_g s_kg with the query's
//     per-group constants C_g (the full scan's bound): the exact score lies in
//     [lo, hi];
//   - each block sends its slots' bounds and entries, and the count, smallest
//     lower and largest upper bound of its slots, into the shared memory of
//     block 0 with asynchronous remote stores counted on an mbarrier of block
//     0, and is done; block 0 waits on that barrier alone (no cluster-wide
//     barrier).
// Block 0 then selects with a few block-wide phases:
//   - one pass builds two histograms of 1024 equal-width value buckets, of the
//     lower and of the upper bounds; bucket b_lam holds the k-th largest lower
//     bound, bucket b_mu the (k+1)-th largest upper bound;
//   - a slot whose lower bound lies in a bucket above b_mu is in (at most k
//     slots have an upper bound in those buckets, itself included); a slot
//     whose upper bound lies in a bucket below b_lam is out (at least k slots
//     have a lower bound in bucket b_lam or above, all larger than it);
//   - the undecided rest is scored exactly (one warp per slot: int64 group
//     terms, then the fp64 head chain in ascending head order) and ranked by
//     (exact score desc, entry asc) for the places left;
//   - the chosen entries are written in ascending entry order, -1 padded.
#include "indexer_common.cuh"
#include "umma.cuh"

namespace csa2 {

constexpr int RT_CTAS = 4;
constexpr int RT_THREADS = 512;
constexpr int RT_TILE = 128;
constexpr int RT_TILES = 4;
constexpr int RT_SLOTS = RT_TILE * RT_TILES;       // 512 slots per block
constexpr int RT_POOL = RT_CTAS * RT_SLOTS;        // 2048 slots per query
constexpr int RT_DI = 128, RT_G = 8, RT_H = 8, RT_N = RT_H * RT_G;
constexpr int RT_NB = 1024;                        // histogram buckets

// shared memory, from a 1024-byte aligned base
constexpr uint32_t RT_A = 0;                                     // 4 tiles x 128 rows x 128 B
constexpr uint32_t RT_B = RT_A + RT_TILES * RT_TILE * 128;       // 64 rows x 128 B
constexpr uint32_t RT_SC = RT_B + RT_N * 128;                    // key scales, 8 B per slot
constexpr uint32_t RT_ENT = RT_SC + RT_SLOTS * 8;                // entry of each slot of the block
constexpr uint32_t RT_Q = RT_ENT + RT_SLOTS * 4;                 // QView<128>, packed codes, sq, C_g
constexpr uint32_t RT_LU = RT_Q + 4096;                          // block 0: bounds of every pool slot
constexpr uint32_t RT_PENT = RT_LU + RT_POOL * 8;                // block 0: entry of every pool slot
constexpr uint32_t RT_END = RT_PENT + RT_POOL * 4;
constexpr uint32_t RT_DYN = RT_END + 1024;

// Block 0's selection state, laid over its A tiles once its MMAs are done.
struct RtSel {
    int und[RT_POOL];
    unsigned long long ukey[RT_POOL];
    int hist[2 * RT_NB];           // lower-bound and upper-bound buckets; then the output list
    unsigned char chosen[RT_POOL];
    int wtot[RT_POOL / RT_THREADS][RT_THREADS / 32];   // chosen slots per (chunk, warp)
    int ctl[8];                    // [0] undecided count [1] sure-in count [2] valid count [3] b_lam [4] b_mu
    unsigned int kmin, kmax;
};
static_assert(sizeof(RtSel) <= RT_TILES * RT_TILE * 128, "selection state must fit the A tiles");

__device__ __forceinline__ uint32_t rt_swz(uint32_t row, uint32_t unit) { return row * 128 + ((unit ^ (row & 7)) << 4); }


__device__ __forceinline__ int rt_bucket(float x, float vmin, float scale) {
    return min((int)((x - vmin) * scale), RT_NB - 1);
}

// warp-wide search of the bucket of hist[RT_NB] in which the count from the top
// first reaches `need`: lane l sums its 32 buckets (starting at a lane-dependent
// one, so that the 32 lanes read 32 different banks), a warp scan finds the
// lane, then the warp scans that lane's 32 buckets one per lane
__device__ int rt_find_bucket(const int* hist, int need) {
    const int lane = threadIdx.x & 31;
    constexpr int PER = RT_NB / 32;
    const int top = RT_NB - PER * lane;            // lane 0 holds the top buckets
    int c = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) c += hist[top - 1 - ((i + lane) & (PER - 1))];
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
    const int L = hit ? __ffs(hit) - 1 : 31;
    const int before = __shfl_sync(0xffffffffu, incl - c, L);
    // lane i takes bucket (top of lane L) - 1 - i
    const int bk = RT_NB - PER * L - 1 - lane;
    int cum = hist[bk];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, cum, o);
        if (lane >= o) cum += y;
    }
    hit = __ballot_sync(0xffffffffu, before + cum >= need);
    const int i = hit ? __ffs(hit) - 1 : 31;
    return RT_NB - PER * L - 1 - i;
}

// The query's FP4 codes and its view for the exact scores, from its fp32
// values: four threads per 16-value group (each takes four values), with the
// arithmetic of the query quantisation kernel (the group's scale from its
// largest magnitude; nearest E2M1 code by exact threshold comparisons).
__device__ void rt_quantize_query(QView<RT_DI> v, uint2* packed, const float* __restrict__ raw, int tid) {
    const int g = tid >> 2, q4 = tid & 3;                  // group g, values 4 q4 .. 4 q4 + 3
    const float4 x4 = __ldg(reinterpret_cast<const float4*>(raw + (int64_t)g * 16) + q4);
    const float x[4] = {x4.x, x4.y, x4.z, x4.w};
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const uint32_t sb = f32_to_e4m3_satfinite(__fdiv_rn(amax, 6.0f));
    const float sc = e4m3_to_f32(sb);
    uint32_t nib = 0u;
    if (sc > 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; ++i) nib |= e2m1_code(x[i], sc) << (4 * i);
    }
    v.qp[4 * g + q4] = (int)unpack4_int8(nib);
    const uint32_t n1 = __shfl_xor_sync(0xffffffffu, nib, 1);
    const uint32_t n2 = __shfl_xor_sync(0xffffffffu, nib, 2);
    const uint32_t n3 = __shfl_xor_sync(0xffffffffu, nib, 3);
    if (q4 == 0) {
        packed[g] = make_uint2(nib | (n1 << 16), n2 | (n3 << 16));
        v.qsc[g] = sc;
        v.qsi[g] = e4m3_times_512(sb);
    }
}

__global__ void __launch_bounds__(RT_THREADS, 2) k_reindex_tc(const int32_t* __restrict__ pool, int pool_len,
                                                               const uint8_t* __restrict__ kc_all,
                                                               const uint8_t* __restrict__ ks_all, int capacity,
                                                               const uint8_t* __restrict__ iq_codes,
                                                               const uint8_t* __restrict__ iq_scales,
                                                               const float* __restrict__ iq_raw,
                                                               const float* __restrict__ w_head, int n_q, int k,
                                                               int32_t* __restrict__ idx_out, int* __restrict__ err) {
    pdl_wait();
    pdl_launch_next();
    extern __shared__ uint8_t dyn[];
    __shared__ __align__(8) unsigned long long bar_mma, bar_x;
    __shared__ uint32_t tmem_base;
    __shared__ __align__(16) unsigned int p_stat[RT_CTAS][4];   // block 0: per block valid slots, smallest lower / largest upper bound key
    __shared__ unsigned int l_stat[3];        // this block's own
    const uint32_t raw_base = umma::smem_u32(dyn);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* sm = dyn + (base - raw_base);
    const uint32_t rank = umma::cluster_rank();
    const int ql = blockIdx.y, b = blockIdx.z;
    const int64_t gq = (int64_t)b * n_q + ql;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s0 = (int)rank * RT_SLOTS;                    // first pool slot of this block
    int* ent = reinterpret_cast<int*>(sm + RT_ENT);
    uint8_t* scl = sm + RT_SC;
    QView<RT_DI> v;
    v.bind(reinterpret_cast<int*>(sm + RT_Q), RT_H);
    uint2* packed = reinterpret_cast<uint2*>(sm + RT_Q + QView<RT_DI>::words(RT_H) * 4);
    float* sq = reinterpret_cast<float*>(packed + RT_N);
    float* cbs = sq + RT_N;                                 // C_g, g = 0..7
    // the query area holds the view (QView<128>::words(8) = 408 words), the packed codes, sq and C_g
    static_assert(408 * 4 + RT_N * 8 + RT_N * 4 + RT_G * 4 <= RT_LU - RT_Q, "query area");
    bool ok = true;

    if (tid == 0) {
        umma::mbar_init(umma::smem_u32(&bar_mma), RT_TILES);   // one commit per tile issuer
        umma::mbar_init(umma::smem_u32(&bar_x), 1);
        umma::fence_mbar_init();
        // block 0 expects every other block's bounds, entries and statistics
        if (rank == 0)
            umma::mbar_arrive_expect_tx(umma::smem_u32(&bar_x), (RT_CTAS - 1) * (RT_SLOTS * 12 + 16));
        l_stat[0] = 0u;
        l_stat[1] = ~0u;
        l_stat[2] = 0u;
    }
    // block 0's barrier is set up before any block stores into it
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    if (warp == 0) umma::tmem_alloc(umma::smem_u32(&tmem_base), RT_TILES * 64);
    const int sl = tid;                                     // this thread's slot of the block
    int j = -1;
    if (s0 + sl < pool_len) {
        j = pool[gq * pool_len + s0 + sl];
        if (j < 0 || j >= capacity) j = -1;
    }
    ent[sl] = j;
    // the key rows of the warp's 32 slots into registers (64 code bytes and 8 scale bytes each; an
    // empty slot's row is zero): load i of lane l takes the 16 code bytes (unit l%4) of slot
    // 8i + l/4, so that the eight consecutive rows of a pool block are one 512-byte piece per
    // instruction (the gather is paced by the lines looked up, not the bytes)
    uint4 kw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int jr = __shfl_sync(0xffffffffu, j, 8 * i + (lane >> 2));
        kw[i] = make_uint4(0, 0, 0, 0);
        if (jr >= 0)
            kw[i] = __ldg(reinterpret_cast<const uint4*>(kc_all + ((int64_t)b * capacity + jr) * (RT_DI / 2)) + (lane & 3));
    }
    uint2 kscw = make_uint2(0, 0);
    if (j >= 0) kscw = __ldg(reinterpret_cast<const uint2*>(ks_all + ((int64_t)b * capacity + j) * RT_G));
    // meanwhile: the query, and its block-diagonal operand
    if (iq_raw) {
        if (tid < RT_N * 4) rt_quantize_query(v, packed, iq_raw + gq * RT_H * RT_DI, tid);
        if (tid < RT_H) {
            v.w[tid] = w_head[gq * RT_H + tid];
            v.wd[tid] = (double)v.w[tid] * 0x1p-20;
        }
    } else {
        stage_query<RT_DI>(v, iq_codes + gq * RT_H * (RT_DI / 2), iq_scales + gq * RT_H * RT_G, nullptr,
                           w_head + gq * RT_H, RT_H, tid, RT_THREADS, packed);
    }
    __syncthreads();
    {
        const int n = tid >> 3, u = tid & 7, g = n % RT_G;    // 64 rows x 8 units: one unit per thread
        uint4 val = make_uint4(0, 0, 0, 0);
        if (u == g) {
            const uint2 c = packed[n];
            val.x = c.x;
            val.y = c.y;
        }
        *reinterpret_cast<uint4*>(sm + RT_B + rt_swz(n, u)) = val;
        if (tid < RT_N) sq[tid] = v.qsc[tid];
        if (tid < RT_G) {
            // C_g = fac * 576 * sum_h |w_h| s_qhg, rounded up, times 1 + 2^-10 for the rounding of the
            // 8-term sum of the bound: |D_hg| <= 576, so sum_g C_g s_kg bounds the scan's error term
            float a = 0.0f;
            for (int h = 0; h < RT_H; ++h) a = __fmaf_ru(fabsf(v.w[h]), v.qsc[h * RT_G + tid], a);
            cbs[tid] = __fmul_ru(__fmul_ru(a, 576.0f * bound_factor(RT_H, RT_DI)), 1.0f + 0x1p-10f);
        }
    }
    // the slot's row in the operand layout: unit g = the 8 code bytes of group g, then 8 zero bytes
    {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = (sl & ~31) + 8 * i + (lane >> 2), g = 2 * (lane & 3);
            uint8_t* row = sm + RT_A + (s / RT_TILE) * (RT_TILE * 128);
            *reinterpret_cast<uint4*>(row + rt_swz(s % RT_TILE, g)) = make_uint4(kw[i].x, kw[i].y, 0u, 0u);
            *reinterpret_cast<uint4*>(row + rt_swz(s % RT_TILE, g + 1)) = make_uint4(kw[i].z, kw[i].w, 0u, 0u);
        }
        *reinterpret_cast<uint2*>(sm + RT_SC + sl * 8) = kscw;
    }
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = tmem_base;
    if (lane == 0 && warp < RT_TILES) {
        // warp t issues tile t's MMAs (four issuers keep the tensor pipe busier than one)
        const uint32_t idesc = (1u << 4) | (5u << 7) | (5u << 10) | ((uint32_t)(RT_N >> 3) << 17) |
                               ((uint32_t)(RT_TILE >> 4) << 24);
        const int t = warp;
        if (s0 + t * RT_TILE < pool_len) {
#pragma unroll
            for (int ks = 0; ks < RT_DI / 32; ++ks) {
                const uint64_t ad = umma::desc(base + RT_A + t * (RT_TILE * 128) + ks * 32, 16, 1024, umma::LAYOUT_SW128);
                const uint64_t bd = umma::desc(base + RT_B + ks * 32, 16, 1024, umma::LAYOUT_SW128);
                asm volatile(
                    "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                    " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(tmem + 64 * t),
                    "l"(ad), "l"(bd), "r"(idesc), "r"(ks));
            }
        }
        umma::commit(umma::smem_u32(&bar_mma));
    }
    ok &= umma::mbar_wait(umma::smem_u32(&bar_mma), 0);
    umma::fence_after();
    RtSel& sel = *reinterpret_cast<RtSel*>(sm + RT_A);     // the A tiles are free once the MMAs are done
    if (rank == 0) {
        // block 0's selection state starts at zero; its barriers below order these stores
        constexpr int NCH0 = RT_POOL / RT_THREADS;
        reinterpret_cast<unsigned int*>(sel.chosen)[tid] = 0u;
        static_assert(RT_POOL == 4 * RT_THREADS && NCH0 == 4, "one word of chosen flags per thread");
        for (int i = tid; i < 2 * RT_NB; i += RT_THREADS) sel.hist[i] = 0;
        if (tid < 8) sel.ctl[tid] = 0;
    }
    // bounds: warp w reads TMEM lane quarter w % 4 of tile w / 4; thread = tile row
    const int t_ep = warp >> 2;
    const int sl_ep = t_ep * RT_TILE + (warp & 3) * 32 + lane;
    float2 mine = make_float2(-INFINITY, -INFINITY);
    if (s0 + t_ep * RT_TILE < pool_len) {                    // warp-uniform
        const uint32_t lb = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 64 * t_ep;
        const bool valid = ent[sl_ep] >= 0;
        const uint2 skw = *reinterpret_cast<const uint2*>(scl + sl_ep * 8);
        float skf[RT_G];
#pragma unroll
        for (int p = 0; p < RT_G / 2; ++p) {
            const float2 f = e4m3_pair_f32(((p < 2 ? skw.x : skw.y) >> (16 * (p & 1))) & 0xffffu);
            skf[2 * p] = f.x;
            skf[2 * p + 1] = f.y;
        }
        float E = 0.0f;
#pragma unroll
        for (int g = 0; g < RT_G; ++g) E = __fmaf_rn(cbs[g], skf[g], E);
        float S = 0.0f;
#pragma unroll
        for (int hh = 0; hh < RT_H; hh += 4) {
            float dv[4 * RT_G];
#pragma unroll
            for (int c = 0; c < 4 * RT_G; c += 16) umma::tmem_ld16(lb + hh * RT_G + c, dv + c);
            umma::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float dd = 0.0f;
#pragma unroll
                for (int g = 0; g < RT_G; ++g) dd += dv[h * RT_G + g] * (sq[(hh + h) * RT_G + g] * skf[g]);   // terms exact
                S = __fmaf_rn(v.w[hh + h], fmaxf(dd, 0.0f), S);
            }
        }
        if (valid) mine = make_float2(S - E, S + E);
    }
    // this block's count and range of its slots' bounds
    {
        const bool valid = ent[sl_ep] >= 0 && s0 + sl_ep < pool_len;
        const unsigned c = __popc(__ballot_sync(0xffffffffu, valid));
        const unsigned mn = __reduce_min_sync(0xffffffffu, valid ? f32_key(mine.x) : ~0u);
        const unsigned mx = __reduce_max_sync(0xffffffffu, valid ? f32_key(mine.y) : 0u);
        if (lane == 0 && c) {
            atomicAdd(&l_stat[0], c);
            atomicMin(&l_stat[1], mn);
            atomicMax(&l_stat[2], mx);
        }
    }
    umma::fence_before();
    __syncthreads();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // block 0 exists and is set up
    float2* glu = reinterpret_cast<float2*>(sm + RT_LU);    // meaningful in block 0
    int* gent = reinterpret_cast<int*>(sm + RT_PENT);
    if (warp == 0) {
        umma::fence_after();
        umma::tmem_dealloc(tmem, RT_TILES * 64);
    }
    if (!ok) atomicExch(err, 1);
    if (rank != 0) {
        // 12 bytes per slot and 16 bytes of statistics per block, counted on block 0's barrier
        const uint32_t mb = umma::mapa(umma::smem_u32(&bar_x), 0);
        umma::st_async_v2_b32(umma::mapa(umma::smem_u32(&glu[s0 + sl_ep]), 0), __float_as_uint(mine.x),
                              __float_as_uint(mine.y), mb);
        umma::st_async_b32(umma::mapa(umma::smem_u32(&gent[s0 + sl_ep]), 0), (uint32_t)ent[sl_ep], mb);
        if (tid == 0)
            umma::st_async_v4_b32(umma::mapa(umma::smem_u32(&p_stat[rank][0]), 0), l_stat[0], l_stat[1], l_stat[2], 0u,
                                  mb);
        return;
    }
    glu[sl_ep] = mine;
    gent[sl_ep] = ent[sl_ep];
    if (tid < 3) p_stat[0][tid] = l_stat[tid];
    if (!umma::mbar_wait_cluster(umma::smem_u32(&bar_x), 0)) atomicExch(err, 1);   // the other blocks' stores have landed
    __syncthreads();
    unsigned int s_stat[3] = {0u, ~0u, 0u};  // valid slots, smallest lower / largest upper bound key of the pool
#pragma unroll
    for (int r = 0; r < RT_CTAS; ++r) {
        s_stat[0] += p_stat[r][0];
        s_stat[1] = min(s_stat[1], p_stat[r][1]);
        s_stat[2] = max(s_stat[2], p_stat[r][2]);
    }

    // ================= block 0: selection over the n slots of the pool (slot u = c * 512 + tid)
    const int n = pool_len < RT_POOL ? pool_len : RT_POOL;
    constexpr int NCH = RT_POOL / RT_THREADS;
    const int n_valid = (int)s_stat[0];
    if (n_valid <= k) {
        for (int u = tid; u < n; u += RT_THREADS) sel.chosen[u] = gent[u] >= 0;
    } else {
        const float vmin = key_value(s_stat[1]), vmax = key_value(s_stat[2]);
        float scale = (float)RT_NB / (vmax - vmin);
        if (!(scale > 0.0f && scale < INFINITY)) scale = 0.0f;      // one bucket
        int blo[NCH], bhi[NCH];
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            const int u = ch * RT_THREADS + tid;
            blo[ch] = -1;
            bhi[ch] = -1;
            if (u < n && gent[u] >= 0) {
                const float2 b2 = glu[u];
                blo[ch] = rt_bucket(b2.x, vmin, scale);
                bhi[ch] = rt_bucket(b2.y, vmin, scale);
                atomicAdd(&sel.hist[blo[ch]], 1);
                atomicAdd(&sel.hist[RT_NB + bhi[ch]], 1);
            }
        }
        __syncthreads();
        if (warp == 0) {
            const int bl = rt_find_bucket(sel.hist, k);
            if (lane == 0) sel.ctl[3] = bl;
        } else if (warp == 1) {
            const int bm = rt_find_bucket(sel.hist + RT_NB, k + 1);
            if (lane == 0) sel.ctl[4] = bm;
        }
        __syncthreads();
        const int b_lam = sel.ctl[3], b_mu = sel.ctl[4];
        int ns = 0;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            const int u = ch * RT_THREADS + tid;
            bool und = false;
            if (blo[ch] >= 0) {
                if (blo[ch] > b_mu) {
                    sel.chosen[u] = 1;
                    ++ns;
                } else if (bhi[ch] >= b_lam) {
                    und = true;
                }
            }
            const int pos = append_slot(und, &sel.ctl[0]);
            if (und) sel.und[pos] = u;
        }
        ns = __reduce_add_sync(0xffffffffu, ns);
        if (lane == 0) atomicAdd(&sel.ctl[1], ns);
        __syncthreads();
        const int nu = sel.ctl[0], r = k - sel.ctl[1];
        if (r > 0) {
            // exact score of each undecided slot, one warp per slot: lane l takes the group
            // terms of (head l/8, group l%8) and (head l/8 + 4, group l%8)
            const uint8_t* kc = kc_all + (int64_t)b * capacity * (RT_DI / 2);
            const uint8_t* ks = ks_all + (int64_t)b * capacity * RT_G;
            const int g = lane & 7, h1 = lane >> 3, h2 = h1 + 4;
            for (int i = warp; i < nu; i += RT_THREADS / 32) {
                const int jj = gent[sel.und[i]];
                const uint2 cw = __ldg(reinterpret_cast<const uint2*>(kc + (int64_t)jj * (RT_DI / 2)) + g);
                const int ski = e4m3_times_512(__ldg(ks + (int64_t)jj * RT_G + g));
                const uint32_t kv[4] = {unpack4_int8(cw.x & 0xffffu), unpack4_int8(cw.x >> 16),
                                        unpack4_int8(cw.y & 0xffffu), unpack4_int8(cw.y >> 16)};
                long long d1 = (long long)(group_dot4(v.qp + h1 * (RT_DI / 4) + 4 * g, kv) * v.qsi[h1 * RT_G + g]) * ski;
                long long d2 = (long long)(group_dot4(v.qp + h2 * (RT_DI / 4) + 4 * g, kv) * v.qsi[h2 * RT_G + g]) * ski;
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    d1 += __shfl_xor_sync(0xffffffffu, d1, o);
                    d2 += __shfl_xor_sync(0xffffffffu, d2, o);
                }
                // D_h sits in lanes 8(h%4) (d1 for h < 4, d2 otherwise): the head chain in
                // ascending order
                double S = 0.0;
#pragma unroll
                for (int h = 0; h < RT_H; ++h) {
                    const long long D = __shfl_sync(0xffffffffu, h < 4 ? d1 : d2, 8 * (h & 3));
                    S = fma(v.wd[h], u53_to_f64(D), S);
                }
                if (lane == 0) sel.ukey[i] = f64_key(S);
            }
            __syncthreads();
            // the r best undecided slots by (exact score desc, entry asc)
            for (int i = tid; i < nu; i += RT_THREADS) {
                const unsigned long long key = sel.ukey[i];
                const int id = gent[sel.und[i]];
                int rk = 0;
                for (int m = 0; m < nu; ++m) {
                    const unsigned long long km = sel.ukey[m];
                    rk += (km > key) || (km == key && gent[sel.und[m]] < id);
                }
                if (rk < r) sel.chosen[sel.und[i]] = 1;
            }
        }
    }
    __syncthreads();
    // the chosen entries in slot order (ballots per chunk and warp), then in ascending
    // entry order: an HSI pool is ascending already, any other pool is ordered by counting
    unsigned int mask[NCH];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
        const int u = ch * RT_THREADS + tid;
        mask[ch] = __ballot_sync(0xffffffffu, u < n && sel.chosen[u]);
        if (lane == 0) sel.wtot[ch][warp] = __popc(mask[ch]);
    }
    __syncthreads();
    // exclusive prefix of the (chunk, warp) counts in slot order: every warp scans the 64 counts
    // (two per lane) and takes the four of its own
    constexpr int NW = RT_THREADS / 32;
    static_assert(NCH * NW == 64, "two (chunk, warp) counts per lane");
    int kept, wbase[NCH];
    {
        const int* wt = &sel.wtot[0][0];
        const int a = wt[2 * lane], b2 = wt[2 * lane + 1];
        int incl = a + b2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        kept = __shfl_sync(0xffffffffu, incl, 31);
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            const int idx = ch * NW + warp;                  // count idx sits in lane idx / 2
            const int ex = __shfl_sync(0xffffffffu, incl - a - b2, idx >> 1);
            const int aa = __shfl_sync(0xffffffffu, a, idx >> 1);
            wbase[ch] = (idx & 1) ? ex + aa : ex;
        }
    }
    int* list = reinterpret_cast<int*>(sel.hist);
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
        if ((mask[ch] >> lane) & 1u)
            list[wbase[ch] + __popc(mask[ch] & ((1u << lane) - 1u))] = gent[ch * RT_THREADS + tid];
    __syncthreads();
    // the list is written out as it stands while its order is checked (an HSI pool is ascending);
    // any other pool is put in ascending order by counting
    bool unordered = false;
    int32_t* out = idx_out + gq * k;
    for (int i = tid; i < k; i += RT_THREADS) {
        const int id = i < kept ? list[i] : -1;
        out[i] = id;
        if (i + 1 < kept) unordered |= id >= list[i + 1];
    }
    if (__syncthreads_or(unordered)) {
        for (int i = tid; i < kept; i += RT_THREADS) {
            const int id = list[i];
            int p = 0;
            for (int m = 0; m < kept; ++m) p += list[m] < id;
            out[p] = id;
        }
    }
}

bool reindex_tc_supported(int d_idx, int H, int pool_len) {
    return d_idx == RT_DI && H == RT_H && pool_len <= RT_POOL;
}

cudaError_t launch_reindex_tc(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                              const float* iq_raw, const float* w_head, int n_q, const int32_t* pool, int pool_len,
                              int k, int32_t* idx_out, int* err, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(k_reindex_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RT_DYN);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(RT_CTAS, n_q, c.batch);
    cfg.blockDim = dim3(RT_THREADS);
    cfg.dynamicSmemBytes = RT_DYN;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = RT_CTAS;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, k_reindex_tc, pool, pool_len, (const uint8_t*)c.ikey_codes,
                           (const uint8_t*)c.ikey_scales, c.capacity, iq_codes, iq_scales, iq_raw, w_head, n_q, k,
                           idx_out, err);
    note_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csa2

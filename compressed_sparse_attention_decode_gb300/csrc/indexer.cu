// Lightweight indexer, exact top-k, HSI candidate pool, Reindex and Reuse
// ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる", §2.3.1 indexer and
// top-k, §2.3.2 Full / Reindex / Reuse, §2.3.4 HSI).
//
// Score of entry j for one query: S_j = sum_h w_h * ReLU(q_h . k_j) with q, k
// the dequantised FP4 vectors; the ranking (S desc, j asc) must match an fp64
// evaluation exactly.  The per-group sums G = sum_i 2q_i * 2k_i over 16-value
// groups are exact integers (dp4a on doubled E2M1 values); each group term
// t = G * s_q * s_k / 4 is exact in fp32.  The scan computes
//     S~ = fp32 chain sum_h w_h max(sum_g t_hg, 0)
//     E  = fac * sum_h |w_h| sum_g |t_hg|,  fac = 2 (2H + G + 8) 2^-24
// so that the fp64-exact score lies in [S~ - E, S~ + E] (recursive-summation
// error bounds).  Selection then needs exact scores only for entries whose
// interval reaches the k-th largest lower bound: usually k plus a handful.
#include "indexer_common.cuh"
#include "umma.cuh"

namespace csa2 {

// ---------------------------------------------------------------- scans

// Full scan with local selection.  One block per (sequence, QB queries,
// chunk of E entries): the (S~-E, S~+E) bounds of the chunk stay in shared
// memory; for each query the block finds the chunk's k-th largest lower bound
// and forwards every entry whose upper bound reaches it (the global k-th
// lower bound is never smaller, so nothing the exact top-k needs is dropped),
// and likewise for HSI blocks (bounds = max of member bounds; the newest
// block, always kept, is not forwarded).
template <int DI>
__global__ void __launch_bounds__(256) k_scan_full(const uint8_t* __restrict__ kc_all, const uint8_t* __restrict__ ks_all,
                                                   int capacity, const uint8_t* __restrict__ iq_codes,
                                                   const uint8_t* __restrict__ iq_scales, const float* __restrict__ w_head,
                                                   const int64_t* __restrict__ q_pos, int n_q, int q0, int n_qc, int H,
                                                   int QB, int E, int k, int pool_blocks, int bs,
                                                   int* __restrict__ counts, int* __restrict__ cid,
                                                   float2* __restrict__ clu, int* __restrict__ bid,
                                                   float2* __restrict__ blu, int list_len, int ratio) {
    pdl_wait();
    pdl_launch_next();
    extern __shared__ int smem[];
    __shared__ RadixSmem rs;
    const int b = blockIdx.z;
    const int qa = blockIdx.y * QB;
    const int nqb = min(QB, n_qc - qa);
    const int words = QView<DI>::words(H);
    int* nel = smem;
    float2* slu = reinterpret_cast<float2*>(smem + 32 + QB * words);
    rs.whist = reinterpret_cast<int*>(slu + QB * E);         // 8 warps x 256
    for (int t = 0; t < nqb; ++t) {
        QView<DI> v;
        v.bind(smem + 32 + t * words, H);
        const int64_t gq = (int64_t)b * n_q + q0 + qa + t;
        stage_query<DI>(v, iq_codes + gq * H * (DI / 2), iq_scales + gq * H * (DI / 16), nullptr, w_head + gq * H, H,
                        threadIdx.x, blockDim.x);
        if (threadIdx.x == 0) nel[t] = n_elig_of(q_pos[gq], capacity, ratio);
    }
    __syncthreads();
    const int c0 = blockIdx.x * E;
    int maxn = 0;
    for (int t = 0; t < nqb; ++t) maxn = max(maxn, nel[t]);
    if (c0 >= maxn) return;                       // uniform over the block
    const float fac = bound_factor(H, DI);
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        const int j = c0 + i;
        if (j < maxn) {
            KeyRow<DI> kr;
            const int64_t row = (int64_t)b * capacity + j;
            kr.load(kc_all + row * (DI / 2), ks_all + row * (DI / 16));
            for (int t = 0; t < nqb; ++t) {
                float L = -INFINITY, U = -INFINITY;
                if (j < nel[t]) {
                    QView<DI> v;
                    v.bind(smem + 32 + t * words, H);
                    approx_score<DI>(kr, v, H, fac, L, U);
                }
                slu[t * E + i] = make_float2(L, U);
            }
        } else {
            for (int t = 0; t < nqb; ++t) slu[t * E + i] = make_float2(-INFINITY, -INFINITY);
        }
    }
    __syncthreads();
    for (int t = 0; t < nqb; ++t) {
        forward_candidates(slu + t * E, c0, E, nel[t], k, pool_blocks, bs, (int64_t)b * n_qc + qa + t, list_len,
                           counts, cid, clu, bid, blu, rs);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- exact selection

struct SelectSmem {
    RadixSmem rs;
    __align__(16) int whist[16 * 256];   // per-warp radix histograms (up to 512 threads)
    unsigned long long key[MAX_K];
    int id[MAX_K];
    unsigned long long* key2;     // merge buffers, MAX_K each (dynamic shared memory)
    int* id2;
    int* din;                     // MAX_K ints of scratch (dynamic shared memory)
    unsigned int* bitmap;         // SEL_BITMAP_BITS bits (dynamic shared memory, k_select only)
};
// dynamic shared memory of k_select after the staged query: key2 | id2 | din | bitmap
constexpr size_t SEL_DYN_EXTRA = (size_t)MAX_K * (8 + 4 + 4);
constexpr int SEL_BITMAP_BITS = 1 << 19;
constexpr size_t SEL_BITMAP_BYTES = SEL_BITMAP_BITS / 8;

// the double whose order-preserving key (f64_key) is u
__device__ __forceinline__ double f64_of_key(unsigned long long u) {
    return __longlong_as_double((long long)((u & 0x8000000000000000ull) ? (u & 0x7fffffffffffffffull) : ~u));
}

// An order-preserving 32-bit image of the double whose key (f64_key) is u:
// the double truncated to float precision by integer operations.  Truncation
// of the magnitude is monotone in the value, so a larger double never gets a
// smaller image; magnitudes below the smallest normal float map to the image
// of zero, above the largest finite float to that float.
__device__ __forceinline__ uint32_t f32_image_of_key(unsigned long long u) {
    const unsigned long long b = (u & 0x8000000000000000ull) ? (u & 0x7fffffffffffffffull) : ~u;
    const uint32_t sgn = (uint32_t)(b >> 63);
    const int e = (int)((b >> 52) & 0x7ffu) - (1023 - 127);
    if (e <= 0) return 0x80000000u;
    const uint32_t mag = e > 254 ? 0x7f7fffffu : ((uint32_t)e << 23) | (uint32_t)((b >> 29) & 0x7fffffu);
    return sgn ? ~mag : (mag | 0x80000000u);
}

// exclusive prefix sum of v over the block; *total gets the sum.  ws: 65 ints
// of shared memory; every thread calls it.
__device__ int block_exclusive_scan(int v, int* total, int* ws) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int s0 = lane < nw ? ws[lane] : 0;
        int inc2 = s0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc2, o);
            if (lane >= o) inc2 += y;
        }
        if (lane < nw) ws[32 + lane] = inc2 - s0;
        if (lane == nw - 1) ws[64] = inc2;
    }
    __syncthreads();
    const int r = ws[32 + warp] + incl - v;
    *total = ws[64];
    __syncthreads();
    return r;
}

// Flags (sm.id2[t] = 1) the k best of the n <= MAX_K items sm.key/sm.id[t] by
// (key desc, id asc); key 0 marks a slot that holds no entry.  A band of float
// images of the scores around the k-th (block_kth_band) splits the items into
// sure (above the band), out (below) and the band, whose members are ranked
// exactly by counting.  The float images are computed once into key2 (viewed
// as 32-bit words; 0 for an empty slot, which the band skips as non-finite).
// Returns the number flagged, min(k, entries).
__device__ __noinline__ int select_best_set(int n, int k, SelectSmem& sm) {
    int* flag = sm.id2;
    unsigned int* fkey = reinterpret_cast<unsigned int*>(sm.key2);
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        sm.rs.ctl[3] = 0;
        sm.rs.kmin32 = ~0u;
        sm.rs.kmax32 = 0u;
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sm.rs.hist[i] = 0;
    __syncthreads();
    // one pass: images, the number of entries and the range of their images
    int c = 0;
    unsigned int mn = ~0u, mx = 0u;
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
        const unsigned long long u = sm.key[t];
        flag[t] = 0;
        const unsigned int f = u != 0ull ? f32_image_of_key(u) : 0u;
        fkey[t] = f;
        if (u != 0ull) {
            ++c;
            mn = min(mn, f);
            mx = max(mx, f);
        }
    }
    c = __reduce_add_sync(0xffffffffu, c);
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
        atomicAdd(&sm.rs.ctl[3], c);
        atomicMin(&sm.rs.kmin32, mn);
        atomicMax(&sm.rs.kmax32, mx);
    }
    __syncthreads();
    const int n_ent = sm.rs.ctl[3];
    if (n_ent <= k) {
        for (int t = threadIdx.x; t < n; t += blockDim.x) flag[t] = sm.key[t] != 0ull;
        __syncthreads();
        return n_ent;
    }
    auto fk = [&](int t, unsigned int& key) {
        key = fkey[t];
        return key != 0u;
    };
    const uint2 band = block_kth_band_from(fk, n, k, sm.rs.kmin32, sm.rs.kmax32, sm.rs);
    if (threadIdx.x == 0) {
        sm.rs.ctl[0] = 0;
        sm.rs.ctl[3] = 0;
    }
    __syncthreads();
    // above the band: in; in the band: listed with (key, id, slot), contiguously in the
    // per-warp histogram space (idle here) when they fit, else by slot only
    uint4* bl = reinterpret_cast<uint4*>(sm.whist);
    constexpr int BL_CAP = (int)(sizeof(sm.whist) / sizeof(uint4));
    int above = 0;
    for (int t0 = 0; t0 < n; t0 += blockDim.x) {
        const int t = t0 + threadIdx.x;
        bool inband = false;
        unsigned int f;
        if (t < n && fk(t, f)) {
            if (f > band.y) {
                flag[t] = 1;
                ++above;
            } else if (f >= band.x) {
                inband = true;
            }
        }
        const int pos = append_slot(inband, &sm.rs.ctl[0]);
        if (inband) {
            sm.din[pos] = t;
            if (pos < BL_CAP) {
                const unsigned long long key = sm.key[t];
                bl[pos] = make_uint4((unsigned int)key, (unsigned int)(key >> 32), (unsigned int)sm.id[t], (unsigned int)t);
            }
        }
    }
    above = __reduce_add_sync(0xffffffffu, above);
    if (lane == 0) atomicAdd(&sm.rs.ctl[3], above);
    __syncthreads();
    // exact rank of each band member among the band by (key desc, id asc); the r best are in
    const int nb = sm.rs.ctl[0], r = k - sm.rs.ctl[3];
    if (nb <= BL_CAP) {
        for (int i = threadIdx.x; i < nb; i += blockDim.x) {
            const uint4 me = bl[i];
            const unsigned long long key = ((unsigned long long)me.y << 32) | me.x;
            const int id = (int)me.z;
            int rank = 0;
#pragma unroll 4
            for (int j = 0; j < nb; ++j) {
                const uint4 o = bl[j];
                const unsigned long long kj = ((unsigned long long)o.y << 32) | o.x;
                rank += (kj > key) || (kj == key && (int)o.z < id);
            }
            flag[me.w] = rank < r;
        }
    } else {
        for (int i = threadIdx.x; i < nb; i += blockDim.x) {
            const int t = sm.din[i];
            const unsigned long long key = sm.key[t];
            const int id = sm.id[t];
            int rank = 0;
            for (int j = 0; j < nb; ++j) {
                const int tj = sm.din[j];
                const unsigned long long kj = sm.key[tj];
                rank += (kj > key) || (kj == key && sm.id[tj] < id);
            }
            flag[t] = rank < r;
        }
    }
    __syncthreads();
    return k;
}


// Among m candidates (cid[t], ckey[t]) keep the k best by (key desc, id asc):
// the kept ones end up in sm.key/sm.id[0..kept), unordered.  Returns kept.
__device__ int keep_best(const int* cid, const unsigned long long* ckey, int m, int k, SelectSmem& sm) {
    if (m <= k) {
        for (int t = threadIdx.x; t < m; t += blockDim.x) {
            sm.key[t] = ckey[t];
            sm.id[t] = cid[t];
        }
        __syncthreads();
        return m;
    }
    int krem;
    const unsigned long long kth = block_kth_largest<unsigned long long>(
        [&](int t, unsigned long long& key) {
            key = ckey[t];
            return true;
        },
        m, k, sm.rs, &krem);
    // among the ties with key == kth keep the krem lowest ids
    int krem2;
    const unsigned int idcut = block_kth_largest<unsigned int>(
        [&](int t, unsigned int& key) {
            key = ~(unsigned int)cid[t];
            return ckey[t] == kth;
        },
        m, krem, sm.rs, &krem2);
    if (threadIdx.x == 0) sm.rs.ctl[0] = 0;
    __syncthreads();
    for (int base = 0; base < m; base += blockDim.x) {
        const int t = base + threadIdx.x;
        bool take = false;
        if (t < m) take = ckey[t] > kth || (ckey[t] == kth && ~(unsigned int)cid[t] >= idcut);
        const int slot = append_slot(take, &sm.rs.ctl[0]);
        if (take) {
            sm.key[slot] = ckey[t];
            sm.id[slot] = cid[t];
        }
    }
    __syncthreads();
    return k;
}

__device__ __forceinline__ bool sel_before(unsigned long long ka, int ia, unsigned long long kb, int ib, bool by_key) {
    return by_key ? (ka > kb || (ka == kb && ia < ib)) : (ia < ib);
}

// Sort sm.key/sm.id[0..n) (n <= MAX_K), padded with sentinels (key 0, id max)
// to N = a power of two >= 32.  by_key: order (key desc, id asc); otherwise
// (id asc).  Each warp sorts runs of 32 in registers (bitonic network over
// shuffles); then runs are merged pairwise, every element going to its index
// in its run plus the number of sibling-run elements ahead of it (binary
// search; ties between runs go to the left run), alternating with key2/id2.
__device__ void sort_kept(int n, bool by_key, SelectSmem& sm) {
    int N = 32;
    while (N < n) N <<= 1;
    for (int t = n + threadIdx.x; t < N; t += blockDim.x) {
        sm.key[t] = 0ull;
        sm.id[t] = 0x7fffffff;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int r = threadIdx.x >> 5; r < N / 32; r += nw) {
        unsigned long long k = sm.key[r * 32 + lane];
        int id = sm.id[r * 32 + lane];
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
            for (int j = size >> 1; j > 0; j >>= 1) {
                const unsigned long long ko = __shfl_xor_sync(0xffffffffu, k, j);
                const int io = __shfl_xor_sync(0xffffffffu, id, j);
                const bool lower = (lane & j) == 0, up = (lane & size) == 0;
                const bool mine_first = sel_before(k, id, ko, io, by_key);
                if (mine_first != (lower == up)) {
                    k = ko;
                    id = io;
                }
            }
        }
        sm.key[r * 32 + lane] = k;
        sm.id[r * 32 + lane] = id;
    }
    __syncthreads();
    unsigned long long *ka = sm.key, *kb = sm.key2;
    int *ia = sm.id, *ib = sm.id2;
    for (int L = 32; L < N; L <<= 1) {
        for (int e = threadIdx.x; e < N; e += blockDim.x) {
            const int r = e / L, i = e - r * L;
            const unsigned long long x = ka[e];
            const int xi = ia[e];
            const unsigned long long* ks = ka + (r ^ 1) * L;
            const int* is = ia + (r ^ 1) * L;
            const bool left = (r & 1) == 0;
            int lo = 0, hi = L;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                const bool ahead = left ? sel_before(ks[mid], is[mid], x, xi, by_key)
                                        : !sel_before(x, xi, ks[mid], is[mid], by_key);
                if (ahead) lo = mid + 1;
                else hi = mid;
            }
            const int o = (r & ~1) * L + i + lo;
            kb[o] = x;
            ib[o] = xi;
        }
        __syncthreads();
        unsigned long long* tk = ka;
        ka = kb;
        kb = tk;
        int* ti = ia;
        ia = ib;
        ib = ti;
    }
    if (ka != sm.key) {
        for (int t = threadIdx.x; t < n; t += blockDim.x) {
            sm.key[t] = ka[t];
            sm.id[t] = ia[t];
        }
        __syncthreads();
    }
}

// The distinct ids ids[t] (t < n) with flags[t] != 0 (flags == nullptr: all),
// all in [0, id_bound), written to dst[0..cnt) in ascending order; returns cnt.
// bitmap_clear: the caller has zeroed the bitmap's first ceil(id_bound / 32)
// words, with a block barrier since.
// Through a bitmap of id_bound bits and a block prefix sum over its words when
// that fits SEL_BITMAP_BITS, else by sort_kept.  dst must not alias ids.
__device__ __noinline__ int ascending_ids(const int* ids, const int* flags, int n, int id_bound, int* dst, SelectSmem& sm,
                             bool bitmap_clear = false) {
    int total;
    if (id_bound <= SEL_BITMAP_BITS) {
        const int W = (id_bound + 31) >> 5;
        if (!bitmap_clear) {
            for (int w = threadIdx.x; w < W; w += blockDim.x) sm.bitmap[w] = 0u;
            __syncthreads();
        }
        for (int t = threadIdx.x; t < n; t += blockDim.x)
            if (!flags || flags[t]) {
                const int id = ids[t];
                atomicOr(&sm.bitmap[id >> 5], 1u << (id & 31));
            }
        __syncthreads();
        const int per = (W + blockDim.x - 1) / blockDim.x;
        const int w0 = threadIdx.x * per, w1 = min(W, w0 + per);
        int c = 0;
        for (int w = w0; w < w1; ++w) c += __popc(sm.bitmap[w]);
        int pos = block_exclusive_scan(c, &total, sm.rs.hist);
        for (int w = w0; w < w1; ++w) {
            unsigned int bits = sm.bitmap[w];
            while (bits) {
                dst[pos++] = (w << 5) + __ffs(bits) - 1;
                bits &= bits - 1u;
            }
        }
        __syncthreads();
        return total;
    }
    if (threadIdx.x == 0) sm.rs.ctl[0] = 0;
    __syncthreads();
    for (int t0 = 0; t0 < n; t0 += blockDim.x) {
        const int t = t0 + threadIdx.x;
        const bool f = t < n && (!flags || flags[t]);
        const int pos = append_slot(f, &sm.rs.ctl[0]);
        if (f) dst[pos] = ids[t];
    }
    __syncthreads();
    total = sm.rs.ctl[0];
    for (int t = threadIdx.x; t < total; t += blockDim.x) {
        sm.id[t] = dst[t];
        sm.key[t] = 0ull;
    }
    __syncthreads();
    sort_kept(total, false, sm);
    for (int t = threadIdx.x; t < total; t += blockDim.x) dst[t] = sm.id[t];
    __syncthreads();
    return total;
}

// The k best of m candidates (cid[t], ckey[t]) by (key desc, id asc), sorted,
// in sm.key/sm.id[0..kept).  When every candidate fits in shared memory (the
// usual case: k plus the few entries whose bounds straddle the threshold) one
// bitonic sort does it; otherwise a radix selection cuts them to k first.
__device__ __noinline__ int best_sorted(const int* cid, const unsigned long long* ckey, int m, int k, SelectSmem& sm) {
    if (m <= MAX_K) {
        for (int t = threadIdx.x; t < m; t += blockDim.x) {
            sm.key[t] = ckey[t];
            sm.id[t] = cid[t];
        }
        __syncthreads();
        sort_kept(m, true, sm);
        return m < k ? m : k;
    }
    const int kept = keep_best(cid, ckey, m, k, sm);
    sort_kept(kept, true, sm);
    return kept;
}

// Reindex, first pass: the (S~-E, S~+E) bounds of every pool slot (-inf for
// an empty slot), one thread per slot, blockIdx.z taking 512 slots of the
// query's pool ("DeepSeek-v4.1 Flash" §2.3.2, the indexer re-run on the pool).
template <int DI>
__global__ void __launch_bounds__(512) k_pool_bounds(const int32_t* __restrict__ pool, int pool_len,
                                                     const uint8_t* __restrict__ kc_all,
                                                     const uint8_t* __restrict__ ks_all, int capacity,
                                                     const uint8_t* __restrict__ iq_codes,
                                                     const uint8_t* __restrict__ iq_scales, const float* __restrict__ iq_raw,
                                                     const float* __restrict__ w_head, int n_q, int H,
                                                     float2* __restrict__ lu) {
    pdl_wait();
    pdl_launch_next();
    extern __shared__ int qsm[];
    const int ql = blockIdx.x, b = blockIdx.y;
    const int64_t gq = (int64_t)b * n_q + ql;
    QView<DI> v;
    v.bind(qsm, H);
    stage_query<DI>(v, iq_codes + gq * H * (DI / 2), iq_scales + gq * H * (DI / 16),
                    iq_raw ? iq_raw + gq * H * DI : nullptr, w_head + gq * H, H, threadIdx.x,
                    blockDim.x);
    __syncthreads();
    const int t = blockIdx.z * blockDim.x + threadIdx.x;
    if (t >= pool_len) return;
    const int j = pool[gq * pool_len + t];
    float lo = -INFINITY, hi = -INFINITY;
    if (j >= 0 && j < capacity) {
        KeyRow<DI> kr;
        const int64_t row = (int64_t)b * capacity + j;
        kr.load(kc_all + row * (DI / 2), ks_all + row * (DI / 16));
        approx_score<DI>(kr, v, H, bound_factor(H, DI), lo, hi);
    }
    lu[gq * pool_len + t] = make_float2(lo, hi);
}

// Reindex over a pool of at most RX_POOL slots in one launch ("DeepSeek-v4.1
// Flash" §2.3.2 and §2.3.4: the indexer re-run on the Full layer's candidate
// pool).  A cluster of RX_CTAS blocks per query: block r bounds the exact
// score of slots [512 r, 512 r + 512) (the same (S~-E, S~+E) interval as the
// scans) and stores the bounds into the shared memory of block 0 (distributed
// shared memory).  Block 0 then
//   - finds lam <= the k-th largest lower bound and mu >= the (k+1)-th
//     largest upper bound (value-bucket bands);
//   - keeps every slot whose lower bound is above mu (at most k slots have an
//     upper bound above mu, so it is among the k best), drops every slot whose
//     upper bound is below lam (k slots have a lower bound at or above lam);
//   - scores the undecided rest exactly and keeps the best of them by (exact
//     score desc, entry asc) for the remaining places;
//   - writes the chosen entries in ascending order, -1 padded.
constexpr int RX_CTAS = 4;
constexpr int RX_THREADS = 512;
constexpr int RX_POOL = RX_CTAS * RX_THREADS;

struct ReindexSmem {
    float2 lu[RX_POOL];       // bounds of every slot (-inf, -inf for an empty slot)
    int ent[RX_POOL];         // entry of every slot, -1 = empty
    int und[RX_POOL];         // undecided slots
    unsigned char chosen[RX_POOL];
};

template <int DI>
__global__ void __launch_bounds__(RX_THREADS) k_reindex_fused(const int32_t* __restrict__ pool, int pool_len,
                                                               const uint8_t* __restrict__ kc_all,
                                                               const uint8_t* __restrict__ ks_all, int capacity,
                                                               const uint8_t* __restrict__ iq_codes,
                                                               const uint8_t* __restrict__ iq_scales,
                                                               const float* __restrict__ iq_raw,
                                                               const float* __restrict__ w_head, int n_q, int H, int k,
                                                               int32_t* __restrict__ idx_out) {
    pdl_wait();
    pdl_launch_next();
    // dynamic shared memory: the staged query | key2 | id2 | din | ReindexSmem
    extern __shared__ int qsm[];
    __shared__ SelectSmem sm;
    uint8_t* extra = reinterpret_cast<uint8_t*>(qsm + QView<DI>::words(H));
    sm.key2 = reinterpret_cast<unsigned long long*>(extra);
    sm.id2 = reinterpret_cast<int*>(extra + (size_t)MAX_K * 8);
    sm.din = sm.id2 + MAX_K;
    ReindexSmem& rx = *reinterpret_cast<ReindexSmem*>(extra + SEL_DYN_EXTRA);
    const uint32_t rank = umma::cluster_rank();
    const int ql = blockIdx.y, b = blockIdx.z;
    const int64_t gq = (int64_t)b * n_q + ql;
    const int tid = threadIdx.x;
    umma::cluster_arrive_relaxed();          // waited for before the first store into block 0
    QView<DI> v;
    v.bind(qsm, H);
    stage_query<DI>(v, iq_codes + gq * H * (DI / 2), iq_scales + gq * H * (DI / 16),
                    iq_raw ? iq_raw + gq * H * DI : nullptr, w_head + gq * H, H, tid, RX_THREADS);
    __syncthreads();
    const int t = (int)rank * RX_THREADS + tid;
    int j = -1;
    float lo = -INFINITY, hi = -INFINITY;
    if (t < pool_len) {
        j = pool[gq * pool_len + t];
        if (j >= 0 && j < capacity) {
            KeyRow<DI> kr;
            const int64_t row = (int64_t)b * capacity + j;
            kr.load(kc_all + row * (DI / 2), ks_all + row * (DI / 16));
            approx_score<DI>(kr, v, H, bound_factor(H, DI), lo, hi);
        } else {
            j = -1;
        }
    }
    umma::cluster_wait();
    {
        const uint32_t a_lu = umma::mapa(umma::smem_u32(&rx.lu[t]), 0);
        const uint32_t a_id = umma::mapa(umma::smem_u32(&rx.ent[t]), 0);
        asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a_lu), "f"(lo), "f"(hi) : "memory");
        asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(a_id), "r"(j) : "memory");
    }
    umma::cluster_sync();                    // every slot's bounds are in block 0
    if (rank != 0) return;

    const int n = pool_len < RX_POOL ? pool_len : RX_POOL;
    sm.rs.whist = sm.whist;
    if (tid == 0) {
        sm.rs.ctl[0] = 0;
        sm.rs.ctl[3] = 0;
    }
    __syncthreads();
    int c = 0;
    for (int u = tid; u < n; u += RX_THREADS) {
        rx.chosen[u] = 0;
        c += rx.ent[u] >= 0;
    }
    c = __reduce_add_sync(0xffffffffu, c);
    if ((tid & 31) == 0) atomicAdd(&sm.rs.ctl[3], c);
    __syncthreads();
    const int n_valid = sm.rs.ctl[3];
    __syncthreads();
    if (n_valid <= k) {
        for (int u = tid; u < n; u += RX_THREADS) rx.chosen[u] = rx.ent[u] >= 0;
    } else {
        const unsigned int lam = block_kth_bound(
            [&](int u, unsigned int& key) {
                key = f32_key(rx.lu[u].x);
                return true;
            },
            n, k, false, sm.rs);
        const unsigned int mu = block_kth_bound(
            [&](int u, unsigned int& key) {
                key = f32_key(rx.lu[u].y);
                return true;
            },
            n, k + 1, true, sm.rs);
        // sure-in and undecided slots (empty slots have -inf bounds: never in, never undecided)
        if (tid == 0) {
            sm.rs.ctl[0] = 0;
            sm.rs.ctl[3] = 0;
        }
        __syncthreads();
        int ns = 0;
        for (int u0 = 0; u0 < n; u0 += RX_THREADS) {
            const int u = u0 + tid;
            bool und = false;
            if (u < n && rx.ent[u] >= 0) {
                const float2 b2 = rx.lu[u];
                if (f32_key(b2.x) > mu) {
                    rx.chosen[u] = 1;
                    ++ns;
                } else if (f32_key(b2.y) >= lam) {
                    und = true;
                }
            }
            const int pos = append_slot(und, &sm.rs.ctl[0]);
            if (und) rx.und[pos] = u;
        }
        ns = __reduce_add_sync(0xffffffffu, ns);
        if ((tid & 31) == 0) atomicAdd(&sm.rs.ctl[3], ns);
        __syncthreads();
        const int nu = sm.rs.ctl[0], r = k - sm.rs.ctl[3];
        __syncthreads();
        if (r > 0) {
            // exact scores of the undecided slots, then the r best of them
            const uint8_t* kc = kc_all + (int64_t)b * capacity * (DI / 2);
            const uint8_t* ks = ks_all + (int64_t)b * capacity * (DI / 16);
            for (int i = tid; i < nu; i += RX_THREADS) {
                const int jj = rx.ent[rx.und[i]];
                sm.key[i] = f64_key(exact_score<DI>(kc + (int64_t)jj * (DI / 2), ks + (int64_t)jj * (DI / 16), v, H));
                sm.id[i] = jj;
            }
            __syncthreads();
            select_best_set(nu, r, sm);
            for (int i = tid; i < nu; i += RX_THREADS)
                if (sm.id2[i]) rx.chosen[rx.und[i]] = 1;
        }
    }
    __syncthreads();
    // the chosen entries in slot order (each thread takes consecutive slots), then in ascending
    // entry order: an HSI pool is already ascending, any other pool is sorted here
    constexpr int PER = RX_POOL / RX_THREADS;
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int u = tid * PER + i;
        cnt += (u < n && rx.chosen[u]) ? 1 : 0;
    }
    int kept;
    int pos = block_exclusive_scan(cnt, &kept, sm.rs.hist);
    int* list = sm.din;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int u = tid * PER + i;
        if (u < n && rx.chosen[u]) list[pos++] = rx.ent[u];
    }
    __syncthreads();
    bool unordered = false;
    for (int i = tid; i + 1 < kept; i += RX_THREADS) unordered |= list[i] >= list[i + 1];
    if (__syncthreads_or(unordered)) {
        for (int i = tid; i < kept; i += RX_THREADS) {
            sm.id[i] = list[i];
            sm.key[i] = 0ull;
        }
        __syncthreads();
        sort_kept(kept, false, sm);
        for (int i = tid; i < kept; i += RX_THREADS) list[i] = sm.id[i];
        __syncthreads();
    }
    int32_t* out = idx_out + gq * k;
    for (int i = tid; i < k; i += RX_THREADS) out[i] = i < kept ? list[i] : -1;
}

// One block per (sequence, query).  Items t in [0, n): entry ids[t] (-1 =
// empty) with bounds lu[t]; n is *count (Full: the forwarded candidates) or
// n_fixed (Reindex: the pool slots, bounds from k_pool_bounds).  Keeps the
// exact top k; with HSI (Full only) also builds the pool from the forwarded
// block candidates.  dense (the tensor-core decode scan): lu holds the upper
// bound of every eligible entry (item t = entry t), blu the bounds of every HSI
// block, and ids the largest lower-bound key of each aligned group of 8 entries,
// which the thresholds come from.
template <int DI, bool DENSE>
__global__ void __launch_bounds__(512) k_select(const int32_t* __restrict__ ids, const float2* __restrict__ lu,
                                                const int* __restrict__ counts, int n_fixed, int list_len,
                                                const uint8_t* __restrict__ kc_all, const uint8_t* __restrict__ ks_all,
                                                int capacity, const uint8_t* __restrict__ iq_codes,
                                                const uint8_t* __restrict__ iq_scales, const float* __restrict__ iq_raw,
                                                const float* __restrict__ w_head,
                                                const int64_t* __restrict__ q_pos, int n_q, int q0, int n_qc, int H,
                                                int k, int32_t* __restrict__ idx_out, int pool_blocks, int bs,
                                                int32_t* __restrict__ pool_out, const int32_t* __restrict__ bid,
                                                const float2* __restrict__ blu, int* __restrict__ c2id,
                                                unsigned long long* __restrict__ c2key, int* __restrict__ h2id,
                                                unsigned long long* __restrict__ h2key, int ratio) {
    // one instantiation per input form: each holds only the code its form runs (the selection code
    // is large, and what a launch runs should stay in the instruction cache)
    constexpr bool dense = DENSE;
    pdl_wait();
    pdl_launch_next();
    extern __shared__ int qsm[];
    __shared__ SelectSmem sm;
    // gridDim.z == 2 (Full layer with a candidate pool): block z = 0 keeps the top k, z = 1 builds
    // the pool, side by side; the pool block's scratch (h2id, h2key) is its own.  bs == 0 asks for
    // the pure pool: the pool_blocks best entries, chosen by the same code as the top k.
    const bool split = gridDim.z == 2;
    const bool pure = pool_blocks > 0 && bs == 0;
    const bool pure_pool = pure && split && blockIdx.z == 1;
    const int kk = pure_pool ? pool_blocks : k;
    const int b = blockIdx.y, ql = blockIdx.x;
    const int64_t gq = (int64_t)b * n_q + q0 + ql;     // global query row
    const int64_t slab = (int64_t)b * n_qc + ql;        // workspace row
    QView<DI> v;
    v.bind(qsm, H);
    stage_query<DI>(v, iq_codes + gq * H * (DI / 2), iq_scales + gq * H * (DI / 16),
                    iq_raw ? iq_raw + gq * H * DI : nullptr, w_head + gq * H, H, threadIdx.x,
                    blockDim.x);
    const int32_t* id = ids + slab * list_len;
    uint8_t* extra = reinterpret_cast<uint8_t*>(qsm + QView<DI>::words(H));
    sm.key2 = reinterpret_cast<unsigned long long*>(extra);
    sm.id2 = reinterpret_cast<int*>(extra + (size_t)MAX_K * 8);
    sm.din = sm.id2 + MAX_K;
    sm.bitmap = reinterpret_cast<unsigned int*>(extra + SEL_DYN_EXTRA);
    const float2* L = lu + slab * list_len;
    const int n = dense ? n_elig_of(q_pos[gq], capacity, ratio) : (counts ? counts[2 * slab] : n_fixed);
    // dense: the group maxima of the lower bounds (8 entries a group); the kk-th largest of them is
    // a lower bound of the kk-th largest lower bound (each is a different entry's), when there are at
    // least kk groups
    const unsigned int* wmk = reinterpret_cast<const unsigned int*>(ids) + slab * list_len;
    // (taken over groups of 32 or 16 entries, maxima of 4 or 2 group maxima, while those are enough:
    // fewer keys for the band search)
    // The keys are staged in shared memory (the bitmap region is idle here) once, so the passes of the
    // band search do not go back to L2.
    auto wm_floor = [&](int kk2) -> unsigned int {
        constexpr int STAGE_CAP = SEL_BITMAP_BITS / 32 - 64;   // the last 64 words: per-warp key ranges
        const int n8 = n / 8;                     // whole groups of 8 (their maxima are all written)
        int st = 4;
        while (st > 1 && n8 / st < kk2) st >>= 1;
        while (n8 / st > STAGE_CAP) st <<= 1;
        int nk = n8 / st;
        if (nk < kk2) {                           // with the last, partial group too
            st = 1;
            nk = (n + 7) / 8;
            if (nk < kk2 || nk > STAGE_CAP) return 0u;
        }
        // the keys are staged with their range taken on the way (each warp's into its own pair of
        // words), so that the band search needs no range pass of its own
        unsigned int* stage = sm.bitmap;
        unsigned int* wrange = sm.bitmap + (SEL_BITMAP_BITS / 32 - 64);
        unsigned int mn = ~0u, mx = 0u;
        for (int t = threadIdx.x; t < nk; t += blockDim.x) {
            unsigned int key = wmk[st * t];
            for (int i = 1; i < st; ++i) key = max(key, wmk[st * t + i]);
            stage[t] = key;
            if (isfinite(key_value(key))) {
                mn = min(mn, key);
                mx = max(mx, key);
            }
        }
        mn = __reduce_min_sync(0xffffffffu, mn);
        mx = __reduce_max_sync(0xffffffffu, mx);
        const int nw = blockDim.x >> 5;
        if ((threadIdx.x & 31) == 0) {
            wrange[2 * (threadIdx.x >> 5)] = mn;
            wrange[2 * (threadIdx.x >> 5) + 1] = mx;
        }
        for (int i = threadIdx.x; i < 256; i += blockDim.x) sm.rs.hist[i] = 0;
        __syncthreads();
        unsigned int lo = ~0u, hi = 0u;
        for (int w = 0; w < nw; ++w) {
            lo = min(lo, wrange[2 * w]);
            hi = max(hi, wrange[2 * w + 1]);
        }
        return block_kth_bound_arr(stage, nullptr, nk, kk2, false, sm.rs, 1, true, lo, hi);
    };
    // the pure pool's block has the whole block-candidate lists (the scan forwards no blocks then)
    const int64_t hoff = pure ? 0 : list_len / 2;
    int* cid = split && blockIdx.z == 1 ? h2id + slab * list_len + hoff : c2id + slab * list_len;
    unsigned long long* ckey = split && blockIdx.z == 1 ? h2key + slab * list_len + hoff : c2key + slab * list_len;
    const uint8_t* kc = kc_all + (int64_t)b * capacity * (DI / 2);
    const uint8_t* ks = ks_all + (int64_t)b * capacity * (DI / 16);
    auto entry_of = [&](int t) -> int {
        if (dense) return t;
        const int j = id[t];
        return (j >= 0 && j < capacity) ? j : -1;
    };
    if (threadIdx.x == 0) {
        sm.rs.ctl[0] = 0;
        sm.rs.ctl[3] = 0;
    }
    sm.rs.whist = sm.whist;
    __syncthreads();
    if (!split || blockIdx.z == 0 || pure_pool) {
    const int k = kk;                        // the number kept by this block
    // ---- 1. k-th largest lower bound, candidates whose upper bound reaches it.
    // Every forwarded item (Full) is a real entry; an empty pool slot (Reindex)
    // has bounds (-inf, -inf), below every real entry, so the selection may
    // count it as long as more than k real entries exist.
    int c = 0;
    if (counts || dense) {
        c = threadIdx.x == 0 ? n : 0;
    } else {
        for (int t = threadIdx.x; t < n; t += blockDim.x) c += L[t].y != -INFINITY;
    }
    c = __reduce_add_sync(0xffffffffu, c);
    if ((threadIdx.x & 31) == 0) atomicAdd(&sm.rs.ctl[3], c);
    __syncthreads();
    const int n_valid = sm.rs.ctl[3];
    __syncthreads();
    unsigned int lam = 0u;                       // <= the k-th largest lower bound
    if (n_valid > k && dense) {
        lam = wm_floor(k);
    } else if (n_valid > k) {
        // the lower-bound keys, staged once in shared memory (the bitmap region is idle
        // here) when they fit, so the passes of the selection do not go back to L2
        unsigned int* stage = sm.bitmap;
        const bool staged = n <= SEL_BITMAP_BITS / 32;
        if (staged) {
            for (int t = threadIdx.x; t < n; t += blockDim.x) stage[t] = f32_key(L[t].x);
            __syncthreads();
        }
        if (staged)
            lam = block_kth_bound_arr(stage, nullptr, n, k, false, sm.rs);
        else
            lam = block_kth_bound(
                [&](int t, unsigned int& key) {
                    key = f32_key(L[t].x);
                    return true;
                },
                n, k, false, sm.rs);
    }
    if (threadIdx.x == 0) sm.rs.ctl[0] = 0;
    __syncthreads();
    if (dense) {
        // the upper bounds of every eligible entry, four per load and 16 loads in flight per thread;
        // each thread marks its candidates in a 64-bit mask, and a warp reserves their places with
        // one atomic and writes them in a short loop over the mask
        const float* U = dense_ub(lu, slab, list_len);
        const int n4 = n >> 2;
        const int lane = threadIdx.x & 31;
        auto place = [&](unsigned long long mask, int base) {   // every lane of the warp calls it
            const int cnt = __popcll(mask);
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int wb = 0;
            if (lane == 31 && incl) wb = atomicAdd(&sm.rs.ctl[0], incl);
            int pos = __shfl_sync(0xffffffffu, wb, 31) + incl - cnt;
#pragma unroll 1
            while (mask) {
                const int bi = __ffsll((long long)mask) - 1;
                mask &= mask - 1ull;
                const int t = 4 * (base + (bi >> 2) * (int)blockDim.x + (int)threadIdx.x) + (bi & 3);
                cid[pos] = t;
                if (pos < MAX_K) sm.id[pos] = t;
                ++pos;
            }
        };
        for (int base = 0; base < n4; base += 16 * blockDim.x) {
            float4 v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int i4 = base + u * blockDim.x + threadIdx.x;
                v[u] = i4 < n4 ? __ldg(reinterpret_cast<const float4*>(U) + i4)
                               : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            unsigned long long mask = 0ull;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                if (base + u * (int)blockDim.x + (int)threadIdx.x < n4) {
                    mask |= (unsigned long long)(f32_key(v[u].x) >= lam) << (4 * u);
                    mask |= (unsigned long long)(f32_key(v[u].y) >= lam) << (4 * u + 1);
                    mask |= (unsigned long long)(f32_key(v[u].z) >= lam) << (4 * u + 2);
                    mask |= (unsigned long long)(f32_key(v[u].w) >= lam) << (4 * u + 3);
                }
            }
            place(mask, base);
        }
        for (int base = 4 * n4; base < n; base += blockDim.x) {
            const int t = base + threadIdx.x;
            const bool f = t < n && f32_key(U[t]) >= lam;
            const int pos = append_slot(f, &sm.rs.ctl[0]);
            if (f) {
                cid[pos] = t;
                if (pos < MAX_K) sm.id[pos] = t;
            }
        }
    } else {
    for (int base = 0; base < n; base += blockDim.x) {
        const int t = base + threadIdx.x;
        const bool f = t < n && f32_key(L[t].y) >= lam && L[t].y != -INFINITY && entry_of(t) >= 0;
        const int pos = append_slot(f, &sm.rs.ctl[0]);
        if (f) {
            const int j = entry_of(t);
            cid[pos] = j;
            if (pos < MAX_K) sm.id[pos] = j;
        }
    }
    }
    __syncthreads();
    const int m = sm.rs.ctl[0];
    __syncthreads();
    // ---- 2. exact scores of the candidates, 3. the k best, written in
    // ascending entry order (in shared memory when they fit, the usual case:
    // k plus the few entries whose bounds straddle the threshold)
    const int id_bound = (counts || dense) ? n_elig_of(q_pos[gq], capacity, ratio) : capacity;
    int kept;
    if (m <= MAX_K) {
        for (int t = threadIdx.x; t < m; t += blockDim.x) {
            const int j = sm.id[t];
            sm.key[t] = f64_key(exact_score<DI>(kc + (int64_t)j * (DI / 2), ks + (int64_t)j * (DI / 16), v, H));
        }
        __syncthreads();
        select_best_set(m, k, sm);
        kept = ascending_ids(sm.id, sm.id2, m, id_bound, sm.din, sm);
    } else {
        for (int t = threadIdx.x; t < m; t += blockDim.x) {
            const int j = cid[t];
            ckey[t] = f64_key(exact_score<DI>(kc + (int64_t)j * (DI / 2), ks + (int64_t)j * (DI / 16), v, H));
        }
        __syncthreads();
        kept = best_sorted(cid, ckey, m, k, sm);
        kept = ascending_ids(sm.id, nullptr, kept, id_bound, sm.din, sm);
    }
    int32_t* out = pure_pool ? pool_out + gq * k : idx_out + gq * k;
    for (int t = threadIdx.x; t < k; t += blockDim.x) out[t] = t < kept ? sm.din[t] : -1;
    __syncthreads();
    }

    // ---- 4. HSI candidate pool (Full only)
    if (pool_blocks <= 0 || pure || !counts || (split && blockIdx.z == 0)) return;
    const int n_elig = n_elig_of(q_pos[gq], capacity, ratio);
    const int P = pool_blocks * bs;
    int32_t* pout = pool_out + gq * P;
    const int nb = (n_elig + bs - 1) / bs;
    int nsel;
    if (nb <= pool_blocks) {                 // every block fits
        for (int t = threadIdx.x; t < nb; t += blockDim.x) sm.id[t] = t;
        nsel = nb;
        __syncthreads();
    } else if (pool_blocks == 1) {           // one slot: the forced newest block
        if (threadIdx.x == 0) sm.id[0] = nb - 1;
        nsel = 1;
        __syncthreads();
    } else {
        const int Kp = pool_blocks - 1;      // blocks chosen by score besides the forced newest one
        // dense: every block but the forced newest one, by id; its threshold from the group maxima:
        // Kp + 1 distinct blocks (one may be the forced block) need Kp + 1 groups when a block holds
        // at most one group (bs <= 8), bs / 8 times as many otherwise
        const int mb = dense ? nb - 1 : counts[2 * slab + 1];
        const int32_t* bi = bid + slab * list_len;
        const float2* bl = blu + slab * list_len;
        unsigned int lamb = 0u;
        if (dense) {
            if (mb > Kp) lamb = wm_floor((Kp + 1) * (bs > 8 ? bs / 8 : 1));
        } else if (mb > Kp) {                 // <= the Kp-th largest lower bound
            unsigned int* stage = sm.bitmap;
            const bool staged = mb <= SEL_BITMAP_BITS / 32;
            if (staged) {
                for (int t = threadIdx.x; t < mb; t += blockDim.x) stage[t] = f32_key(bl[t].x);
                __syncthreads();
            }
            if (staged)
                lamb = block_kth_bound_arr(stage, nullptr, mb, Kp, false, sm.rs);
            else
                lamb = block_kth_bound(
                    [&](int t, unsigned int& key) {
                        key = f32_key(bl[t].x);
                        return true;
                    },
                    mb, Kp, false, sm.rs);
        }
        // candidates: blocks whose upper bound reaches the Kp-th largest lower
        // bound, with their (upper, lower) bound keys packed in ckey
        if (threadIdx.x == 0) sm.rs.ctl[0] = 0;
        __syncthreads();
        for (int base0 = 0; base0 < mb; base0 += 8 * blockDim.x) {
            float2 b8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = base0 + u * blockDim.x + threadIdx.x;
                b8[u] = t < mb ? bl[t] : make_float2(0.0f, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = base0 + u * blockDim.x + threadIdx.x;
                const float2 b2 = b8[u];
                const bool f = t < mb && f32_key(b2.y) >= lamb;
                const int pos = append_slot(f, &sm.rs.ctl[0]);
                if (f) {
                    cid[pos] = dense ? t : bi[t];
                    ckey[pos] = ((unsigned long long)f32_key(b2.y) << 32) | f32_key(b2.x);
                }
            }
        }
        __syncthreads();
        const int mc = sm.rs.ctl[0];
        __syncthreads();
        if (mc <= Kp) {
            // all of them (there are never fewer than Kp)
            for (int t = threadIdx.x; t < mc; t += blockDim.x) sm.id[t] = cid[t];
        } else {
            // mu >= the (Kp+1)-th largest upper bound.  A block whose lower bound
            // is above mu can be outranked only by blocks whose upper bound is
            // above mu too, at most Kp-1 others: it is in.  Only the rest get
            // exact block maxima, and fill the remaining slots by (max desc, id asc).
            // >= the (Kp+1)-th largest upper bound
            const unsigned int mu = block_kth_bound_arr(nullptr, ckey, mc, Kp + 1, true, sm.rs);
            if (threadIdx.x == 0) {
                sm.rs.ctl[0] = 0;
                sm.rs.ctl[3] = 0;
            }
            __syncthreads();
            // in-place compaction of the undecided ones: a window is read in full
            // before any of it is written, and no slot beyond the window is written
            for (int base = 0; base < mc; base += blockDim.x) {
                const int t = base + threadIdx.x;
                int j = 0;
                bool in = false, und = false;
                if (t < mc) {
                    j = cid[t];
                    in = (unsigned int)ckey[t] > mu;
                    und = !in;
                }
                __syncthreads();
                const int pd = append_slot(in, &sm.rs.ctl[3]);
                if (in) sm.din[pd] = j;
                const int pu = append_slot(und, &sm.rs.ctl[0]);
                if (und) {
                    cid[pu] = j;
                    ckey[pu] = 0ull;
                }
            }
            __syncthreads();
            const int nu = sm.rs.ctl[0], nd = sm.rs.ctl[3];
            __syncthreads();
            for (int u = threadIdx.x; u < nu * bs; u += blockDim.x) {
                const int t = u / bs, j = cid[t] * bs + u % bs;
                const double S = exact_score<DI>(kc + (int64_t)j * (DI / 2), ks + (int64_t)j * (DI / 16), v, H);
                atomicMax(&ckey[t], f64_key(S));
            }
            __syncthreads();
            const int r = Kp - nd;               // 0 <= r < nu
            if (r > 0 && nu <= 256) {
                // few undecided blocks (the usual case): each one's rank by (max desc, id asc) among
                // them, counted directly from a copy in shared memory; ids are distinct, so the r best
                // fill sm.id[0..r)
                for (int t = threadIdx.x; t < nu; t += blockDim.x) {
                    sm.key2[t] = ckey[t];
                    sm.id2[t] = cid[t];
                }
                __syncthreads();
                for (int t = threadIdx.x; t < nu; t += blockDim.x) {
                    const unsigned long long kt = sm.key2[t];
                    const int it = sm.id2[t];
                    int rk = 0;
                    for (int m2 = 0; m2 < nu; ++m2) {
                        const unsigned long long km = sm.key2[m2];
                        rk += (km > kt) || (km == kt && sm.id2[m2] < it);
                    }
                    if (rk < r) sm.id[rk] = it;
                }
            } else if (r > 0) {
                best_sorted(cid, ckey, nu, r, sm);
            }
            __syncthreads();
            for (int t = threadIdx.x; t < nd; t += blockDim.x) sm.id[r + t] = sm.din[t];
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            sm.id[Kp] = nb - 1;
            sm.key[Kp] = 0ull;
        }
        nsel = pool_blocks;
        __syncthreads();
    }
    ascending_ids(sm.id, nullptr, nsel, nb, sm.din, sm);
    for (int u = threadIdx.x; u < P; u += blockDim.x) {
        const int t = u / bs;
        const int j = t < nsel ? sm.din[t] * bs + u % bs : -1;
        // only the newest block can run past n_elig; it has the largest id and sorts last
        pout[u] = (j >= 0 && j < n_elig) ? j : -1;
    }
}

// Reuse: the latest indices, unchanged ("DeepSeek-v4.1 Flash" §2.3.2)
__global__ void k_copy_idx(const int32_t* __restrict__ src, int32_t* __restrict__ dst, int64_t n) {
    pdl_wait();
    pdl_launch_next();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = src[i];
}

// ---------------------------------------------------------------- launchers

constexpr int QUERY_CHUNK = 608;        // queries per scan + select pass (the multi-query tensor scan: one wave)

// workspace of one query slab with item lists of length n:
// counts (2 ints, padded to 16 B) | ids n | lu n | c2id n | c2key n | bid n | blu n
static size_t slab_bytes(int64_t n) { return (size_t)n * (4 + 8 + 4 + 8 + 4 + 8); }

struct SelectWs {
    int* err;
    int* counts;
    int32_t* ids;
    float2* lu;
    int* c2id;
    unsigned long long* c2key;
    int32_t* bid;
    float2* blu;
};

// The first 16 bytes hold the error word (set by a kernel that gave up on a
// bounded wait, read and cleared by csa2_poll_error); the counts follow.
static SelectWs carve(void* ws, int64_t slabs, int64_t n) {
    uint8_t* p = reinterpret_cast<uint8_t*>(ws);
    SelectWs w;
    w.err = reinterpret_cast<int*>(p);
    w.counts = reinterpret_cast<int*>(p + 16);
    p += ((16 + slabs * 2 * sizeof(int) + 255) / 256) * 256;
    w.c2key = reinterpret_cast<unsigned long long*>(p);
    p += slabs * n * 8;
    w.lu = reinterpret_cast<float2*>(p);
    p += slabs * n * 8;
    w.blu = reinterpret_cast<float2*>(p);
    p += slabs * n * 8;
    w.ids = reinterpret_cast<int32_t*>(p);
    p += slabs * n * 4;
    w.c2id = reinterpret_cast<int*>(p);
    p += slabs * n * 4;
    w.bid = reinterpret_cast<int32_t*>(p);
    return w;
}

static size_t ws_bytes(int64_t slabs, int64_t n) {
    return ((16 + slabs * 2 * sizeof(int) + 255) / 256) * 256 + slabs * slab_bytes(n);
}

bool scan_tc_supported(int d_idx, int H, int QB, int pool_blocks, int bs, const csa2_cache& c);
bool scan_mq_tc_supported(int d_idx, int H, int n_q, int pool_blocks);
cudaError_t launch_scan_mq_tc(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                              const float* w_head, int n_q, const int64_t* q_pos, int q0, int n_qc, int k, int* counts,
                              int* cid, float2* clu, int list_len, int* err, cudaStream_t st);
bool reindex_tc_supported(int d_idx, int H, int pool_len);
cudaError_t launch_reindex_tc(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                              const float* iq_raw, const float* w_head, int n_q, const int32_t* pool, int pool_len,
                              int k, int32_t* idx_out, int* err, cudaStream_t st);
cudaError_t launch_scan_full_tc(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                                const float* w_head, int n_q, const int64_t* q_pos, int q0, int n_qc, int H,
                                int pool_blocks, int bs, unsigned int* wmk, float2* lu, float2* blu, int list_len,
                                int* err, cudaStream_t st);

size_t indexer_full_ws(int batch, int n_q, int64_t capacity) {
    const int qc = n_q < QUERY_CHUNK ? n_q : QUERY_CHUNK;
    return ws_bytes((int64_t)batch * qc, capacity + 1);
}

size_t reindex_ws(int batch, int n_q, int64_t pool_len) { return ws_bytes((int64_t)batch * n_q, pool_len); }

template <int DI>
cudaError_t launch_indexer_full_t(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                                  const float* w_head, int n_q, const int64_t* q_pos, int H, int k, int32_t* idx_out,
                                  int pool_blocks, int bs, int32_t* pool_out, void* ws, cudaStream_t st) {
    const int qchunk = n_q < QUERY_CHUNK ? n_q : QUERY_CHUNK;
    const int64_t list_len = (int64_t)c.capacity + 1;
    const SelectWs w = carve(ws, (int64_t)c.batch * qchunk, list_len);
    const size_t qwords = (size_t)QView<DI>::words(H) * sizeof(int);
    // the pure pool (bs == 0): the pool_blocks best entries; the scans then forward every entry
    // that may be among the max(k, pool_blocks) best and no blocks
    const bool pure = pool_blocks > 0 && bs == 0;
    const int kf = pure ? (k > pool_blocks ? k : pool_blocks) : k;
    const int pb_scan = pure ? 0 : pool_blocks, bs_scan = pure ? 1 : bs;
    // queries per scan block and entries per chunk: one query and 4096 entries
    // for decode, 8 queries sharing each key load (1024 entries) otherwise
    const int QB = (n_q >= 8 && pb_scan == 0) ? 8 : 1;
    int E = QB == 1 ? 4096 : 1024;
    if (pb_scan > 0) E = bs_scan * (4096 / bs_scan > 0 ? 4096 / bs_scan : 1);
    const size_t smem1 = 32 * sizeof(int) + QB * qwords + (size_t)QB * E * sizeof(float2) + 8 * 256 * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(k_scan_full<DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    if (e != cudaSuccess) return e;
    for (int q0 = 0; q0 < n_q; q0 += qchunk) {
        const int n_qc = (n_q - q0) < qchunk ? (n_q - q0) : qchunk;
        e = cudaMemsetAsync(w.counts, 0, (size_t)c.batch * n_qc * 2 * sizeof(int), st);
        if (e != cudaSuccess) return e;
        int dense = 0;
        if (scan_mq_tc_supported(DI, H, n_q, pb_scan)) {
            e = launch_scan_mq_tc(c, iq_codes, iq_scales, w_head, n_q, q_pos, q0, n_qc, kf, w.counts, w.ids, w.lu,
                                  (int)list_len, w.err, st);
        } else if (scan_tc_supported(DI, H, QB, pb_scan, bs_scan, c)) {
            e = launch_scan_full_tc(c, iq_codes, iq_scales, w_head, n_q, q_pos, q0, n_qc, H, pb_scan, bs_scan,
                                    reinterpret_cast<unsigned int*>(w.ids), w.lu, w.blu, (int)list_len, w.err, st);
            dense = 1;
        } else {
            dim3 g1((c.capacity + E - 1) / E, (n_qc + QB - 1) / QB, c.batch);
            launch_k(k_scan_full<DI>, g1, 256, smem1, st, c.ikey_codes, c.ikey_scales, c.capacity, iq_codes, iq_scales,
                                                    w_head, q_pos, n_q, q0, n_qc, H, QB, E, kf, pb_scan, bs_scan,
                                                    w.counts, w.ids, w.lu, w.bid, w.blu, (int)list_len, (int)c.ratio);
            note_launch();
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
        // with an HSI pool the top k and the pool are built by two blocks per query at once; the
        // pool block's scratch is the upper half of the block-candidate lists (a query has at most
        // ceil(capacity / bs) <= list_len / 2 block candidates when bs >= 2)
        dim3 g2(n_qc, c.batch, ((pool_blocks > 1 && bs >= 2) || pure) ? 2 : 1);
        const size_t smem2 = qwords + SEL_DYN_EXTRA + SEL_BITMAP_BYTES;
        auto kern = dense ? k_select<DI, true> : k_select<DI, false>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
        if (e != cudaSuccess) return e;
        launch_k(kern, g2, 512, smem2, st, w.ids, w.lu, w.counts, 0, (int)list_len, c.ikey_codes, c.ikey_scales,
                                              c.capacity, iq_codes, iq_scales, (const float*)nullptr, w_head, q_pos, n_q, q0, n_qc, H, k,
                                              idx_out, pool_blocks, bs, pool_out, w.bid, w.blu, w.c2id, w.c2key,
                                              w.bid, reinterpret_cast<unsigned long long*>(w.blu), (int)c.ratio);
        note_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int DI>
cudaError_t launch_reindex_t(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                             const float* iq_raw, const float* w_head, int n_q, int H, const int32_t* pool, int pool_len,
                             int k, int32_t* idx_out, void* ws, cudaStream_t st) {
    const SelectWs w = carve(ws, (int64_t)c.batch * n_q, pool_len);
    const size_t qwords = (size_t)QView<DI>::words(H) * sizeof(int);
    if (reindex_tc_supported(DI, H, pool_len))
        return launch_reindex_tc(c, iq_codes, iq_scales, iq_raw, w_head, n_q, pool, pool_len, k, idx_out, w.err, st);
    if (pool_len <= RX_POOL) {
        // one launch: a cluster of RX_CTAS blocks per query
        const size_t smem = qwords + SEL_DYN_EXTRA + sizeof(ReindexSmem);
        cudaError_t e = cudaFuncSetAttribute(k_reindex_fused<DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(RX_CTAS, n_q, c.batch);
        cfg.blockDim = dim3(RX_THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = RX_CTAS;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, k_reindex_fused<DI>, pool, pool_len, (const uint8_t*)c.ikey_codes,
                               (const uint8_t*)c.ikey_scales, c.capacity, iq_codes, iq_scales, iq_raw, w_head, n_q, H, k,
                               idx_out);
        note_launch();
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    dim3 g0(n_q, c.batch, (pool_len + 511) / 512);
    launch_k(k_pool_bounds<DI>, g0, 512, qwords, st, pool, pool_len, c.ikey_codes, c.ikey_scales, c.capacity, iq_codes,
                                                iq_scales, iq_raw, w_head, n_q, H, w.lu);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = qwords + SEL_DYN_EXTRA + SEL_BITMAP_BYTES;
    e = cudaFuncSetAttribute(k_select<DI, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 g(n_q, c.batch);
    launch_k(k_select<DI, false>, g, 512, smem, st, pool, w.lu, nullptr, pool_len, pool_len, c.ikey_codes, c.ikey_scales,
                                       c.capacity, iq_codes, iq_scales, iq_raw, w_head, nullptr, n_q, 0, n_q, H, k, idx_out, 0,
                                       1, nullptr, nullptr, nullptr, w.c2id, w.c2key, (int*)nullptr,
                                       (unsigned long long*)nullptr, (int)c.ratio);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_indexer_full(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales,
                                const float* w_head, int n_q, const int64_t* q_pos, int H, int k, int32_t* idx_out,
                                int pool_blocks, int bs, int32_t* pool_out, void* ws, cudaStream_t st) {
    if (c.d_idx == 128)
        return launch_indexer_full_t<128>(c, iq_codes, iq_scales, w_head, n_q, q_pos, H, k, idx_out, pool_blocks, bs,
                                          pool_out, ws, st);
    return launch_indexer_full_t<64>(c, iq_codes, iq_scales, w_head, n_q, q_pos, H, k, idx_out, pool_blocks, bs,
                                     pool_out, ws, st);
}

// iq_raw != nullptr: fp32 queries [batch][n_q][H][d_idx], quantised inside the kernels (codes unused)
cudaError_t launch_reindex(const csa2_cache& c, const uint8_t* iq_codes, const uint8_t* iq_scales, const float* iq_raw,
                           const float* w_head, int n_q, int H, const int32_t* pool, int pool_len, int k,
                           int32_t* idx_out, void* ws, cudaStream_t st) {
    if (c.d_idx == 128)
        return launch_reindex_t<128>(c, iq_codes, iq_scales, iq_raw, w_head, n_q, H, pool, pool_len, k, idx_out, ws, st);
    return launch_reindex_t<64>(c, iq_codes, iq_scales, iq_raw, w_head, n_q, H, pool, pool_len, k, idx_out, ws, st);
}

cudaError_t launch_reuse(const int32_t* prev, int32_t* out, int64_t n, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    launch_k(k_copy_idx, (unsigned)((n + 255) / 256), 256, 0, st, prev, out, n);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa2

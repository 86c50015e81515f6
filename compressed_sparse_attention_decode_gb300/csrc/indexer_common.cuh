// Indexer pieces shared by the CUDA-core and the tensor-core scans: query
// staging, key rows, the approximate score with its rigorous error bound, the
// exact fp64 score, block-wide radix selection and candidate forwarding.
#pragma once
#include "common.cuh"

namespace csa2 {

// ---------------------------------------------------------------- query staging

// E4M3 value times 2^9: every E4M3 value is a multiple of 2^-9 (the smallest
// subnormal), so this is an integer; at most 448 * 512 = 229,376
__device__ __forceinline__ int e4m3_times_512(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    return e ? (int)((8u + m) << (e - 1u)) : (int)m;
}

template <int DI>
struct QView {
    int* qp;     // [H][DI/4] doubled E2M1 values, signed int8 x4
    float* qsc;  // [H][DI/16] E4M3 scales as float
    int* qsi;    // [H][DI/16] the same scales times 2^9 (integers < 2^18)
    float* w;    // [H]
    double* wd;  // [H] the weights times 2^-20 in fp64 (exact)
    // 32-bit words of one view; a multiple of 4, so consecutive views stay 16-byte aligned
    __host__ __device__ static int head_words(int H) { return (H * (DI / 4) + 2 * H * (DI / 16) + H + 1) & ~1; }
    __host__ __device__ static int words(int H) { return (head_words(H) + 2 * H + 3) & ~3; }
    __device__ void bind(int* base, int H) {
        qp = base;
        qsc = reinterpret_cast<float*>(qp + H * (DI / 4));
        qsi = reinterpret_cast<int*>(qsc + H * (DI / 16));
        w = reinterpret_cast<float*>(qsi + H * (DI / 16));
        wd = reinterpret_cast<double*>(base + head_words(H));
    }
};

// One query's view: from its FP4 codes and scales, or (raw != nullptr) from
// its unquantised fp32 values, which are quantised here exactly as the query
// quantisation kernel does it (quant_group16, one 16-value group per thread).
// packed != nullptr also receives each group's 8 code bytes (the FP4 codes as
// the tensor-core operands take them).
template <int DI>
__device__ void stage_query(QView<DI> v, const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                            const float* __restrict__ raw, const float* __restrict__ w, int H, int tid, int nthr,
                            uint2* packed = nullptr) {
    if (raw != nullptr) {
        for (int g = tid; g < H * (DI / 16); g += nthr) {
            float x[16];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float4 p = __ldg(reinterpret_cast<const float4*>(raw + (int64_t)g * 16) + t);
                x[4 * t] = p.x;
                x[4 * t + 1] = p.y;
                x[4 * t + 2] = p.z;
                x[4 * t + 3] = p.w;
            }
            uint32_t c0, c1, sb;
            quant_group16(x, c0, c1, sb);
            if (packed) packed[g] = make_uint2(c0, c1);
            v.qp[4 * g] = (int)unpack4_int8(c0 & 0xffffu);
            v.qp[4 * g + 1] = (int)unpack4_int8(c0 >> 16);
            v.qp[4 * g + 2] = (int)unpack4_int8(c1 & 0xffffu);
            v.qp[4 * g + 3] = (int)unpack4_int8(c1 >> 16);
            v.qsc[g] = e4m3_to_f32(sb);
            v.qsi[g] = e4m3_times_512(sb);
        }
    } else {
        for (int i = tid; i < H * (DI / 4); i += nthr)
            v.qp[i] = (int)unpack4_int8(reinterpret_cast<const uint16_t*>(codes)[i]);
        for (int i = tid; i < H * (DI / 16); i += nthr) {
            v.qsc[i] = e4m3_to_f32(scales[i]);
            v.qsi[i] = e4m3_times_512(scales[i]);
            if (packed) packed[i] = *reinterpret_cast<const uint2*>(codes + (size_t)i * 8);
        }
    }
    for (int i = tid; i < H; i += nthr) {
        v.w[i] = w[i];
        v.wd[i] = (double)w[i] * 0x1p-20;
    }
}

template <int DI>
struct KeyRow {
    uint32_t kv[DI / 4];         // doubled key values, signed int8 x4
    float sk[DI / 16];
    __device__ __forceinline__ void load(const uint8_t* __restrict__ kc, const uint8_t* __restrict__ ks) {
#pragma unroll
        for (int v = 0; v < DI / 32; ++v) {
            uint4 c = __ldg(reinterpret_cast<const uint4*>(kc) + v);
            const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                kv[8 * v + 2 * t] = unpack4_int8(cw[t] & 0xffffu);
                kv[8 * v + 2 * t + 1] = unpack4_int8(cw[t] >> 16);
            }
        }
        if (DI == 128) {
            uint2 s = __ldg(reinterpret_cast<const uint2*>(ks));
#pragma unroll
            for (int g = 0; g < 4; ++g) sk[g] = e4m3_to_f32((s.x >> (8 * g)) & 255u);
#pragma unroll
            for (int g = 0; g < DI / 16 - 4; ++g) sk[4 + g] = e4m3_to_f32((s.y >> (8 * g)) & 255u);
        } else {
            uint32_t s = __ldg(reinterpret_cast<const uint32_t*>(ks));
#pragma unroll
            for (int g = 0; g < DI / 16; ++g) sk[g] = e4m3_to_f32((s >> (8 * g)) & 255u);
        }
    }
};

// approximate score and its error bound (see the file header)
template <int DI>
__device__ __forceinline__ void approx_score(const KeyRow<DI>& k, QView<DI> q, int H, float fac, float& L,
                                             float& U) {
    float S = 0.0f, B = 0.0f;
    for (int h = 0; h < H; ++h) {
        float d = 0.0f, A = 0.0f;
#pragma unroll
        for (int g = 0; g < DI / 16; ++g) {
            int G = group_dot4(q.qp + h * (DI / 4) + 4 * g, k.kv + 4 * g);
            float c = q.qsc[h * (DI / 16) + g] * k.sk[g] * 0.25f;   // exact
            float t = (float)G * c;                                  // exact
            d += t;
            A += fabsf(t);
        }
        S = __fmaf_rn(q.w[h], fmaxf(d, 0.0f), S);
        B = __fmaf_rn(fabsf(q.w[h]), A, B);
    }
    float E = B * fac;
    L = S - E;
    U = S + E;
}

// 0 <= D < 2^53 to fp64 exactly, by integer operations (the conversion
// instruction runs on the scarce fp64 units)
__device__ __forceinline__ double u53_to_f64(long long D) {
    if (D <= 0) return 0.0;
    const unsigned long long u = (unsigned long long)D;
    const int e = 63 - __clzll((long long)u);                    // 0 .. 52
    const unsigned long long man = (u << (52 - e)) & 0x000FFFFFFFFFFFFFull;
    return __longlong_as_double((long long)(((unsigned long long)(1023 + e) << 52) | man));
}

// The exact score.  With 2^9-scaled integer scales Sq, Sk and the doubled-code
// group sum G4 = sum 2q*2k, a group term is G4 * Sq * Sk * 2^-20 exactly, so
// D_h = d_h * 2^20 is an integer (|.| < 2^51) summed in int64.  The ReLU is
// taken on D_h, D_h goes to fp64 without rounding, and the head chain
// S = fma(w_h, d_h, S) in ascending h is evaluated as fma(w_h 2^-20, D_h, S):
// the same exact product, so the same rounded result, with one fp64
// operation per head.
template <int DI>
__device__ __noinline__ double exact_score(const uint8_t* __restrict__ kc, const uint8_t* __restrict__ ks, QView<DI> q, int H) {
    KeyRow<DI> k;
    k.load(kc, ks);
    int ski[DI / 16];
    if (DI == 128) {
        const uint2 s = __ldg(reinterpret_cast<const uint2*>(ks));
#pragma unroll
        for (int g = 0; g < DI / 16; ++g) ski[g] = e4m3_times_512(((g < 4 ? s.x : s.y) >> (8 * (g & 3))) & 255u);
    } else {
        const uint32_t s = __ldg(reinterpret_cast<const uint32_t*>(ks));
#pragma unroll
        for (int g = 0; g < DI / 16; ++g) ski[g] = e4m3_times_512((s >> (8 * (g & 3))) & 255u);
    }
    double S = 0.0;
    for (int h = 0; h < H; ++h) {
        long long D = 0;
#pragma unroll
        for (int g = 0; g < DI / 16; ++g) {
            const int G4 = group_dot4(q.qp + h * (DI / 4) + 4 * g, k.kv + 4 * g);
            D += (long long)(G4 * q.qsi[h * (DI / 16) + g]) * ski[g];     // |G4*Sq| < 2^30
        }
        S = fma(q.wd[h], u53_to_f64(D), S);
    }
    return S;
}

// entries wholly before the window [p-127, p] of a query at raw position p, for
// a cache of `ratio` raw positions per entry; clamped to the capacity
__device__ __forceinline__ int n_elig_of(int64_t p, int capacity, int ratio) {
    int64_t n = ratio == 1 ? p - (WINDOW - 1) : (p - (WINDOW - 1)) >> 1;
    if (p < WINDOW - 1) n = 0;
    return (int)(n < capacity ? n : capacity);
}

// The dense upper-bound list of query slab `slab` inside its bound list (list_len float2 slots),
// started on a 16-byte boundary so that it can be read four at a time
__host__ __device__ inline float* dense_ub(float2* lu, int64_t slab, int list_len) {
    return reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(lu + slab * list_len) + 15) & ~(uintptr_t)15);
}
__host__ __device__ inline const float* dense_ub(const float2* lu, int64_t slab, int list_len) {
    return dense_ub(const_cast<float2*>(lu), slab, list_len);
}

__host__ __device__ inline float bound_factor(int H, int DI) { return 2.0f * (float)(2 * H + DI / 16 + 8) * 0x1p-24f; }

// two E4M3 bytes (low byte first) to floats, exactly (through an fp16 pair: every E4M3 value is
// an fp16 value)
__device__ __forceinline__ float2 e4m3_pair_f32(uint32_t two) {
    uint32_t r;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(r) : "r"(two));
    return __half22float2(*reinterpret_cast<__half2*>(&r));
}

// ---------------------------------------------------------------- block-wide radix selection

struct RadixSmem {
    int hist[256];
    int ctl[8];   // [0] append counter, [1] digit, [2] krem, [3] scratch, [4] [5] global append
    unsigned long long kmin, kmax;
    unsigned int kmin32, kmax32;  // the same for 32-bit keys (native shared-memory atomics)
    int* whist;   // per-warp histograms, (blockDim.x / 32) x 256 ints, set by the caller
};

template <typename KeyT>
__device__ __forceinline__ KeyT warp_min_key(KeyT v) {
    if constexpr (sizeof(KeyT) == 4) {
        return (KeyT)__reduce_min_sync(0xffffffffu, (unsigned int)v);
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const KeyT w = __shfl_xor_sync(0xffffffffu, v, o);
            v = w < v ? w : v;
        }
        return v;
    }
}
template <typename KeyT>
__device__ __forceinline__ KeyT warp_max_key(KeyT v) {
    if constexpr (sizeof(KeyT) == 4) {
        return (KeyT)__reduce_max_sync(0xffffffffu, (unsigned int)v);
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const KeyT w = __shfl_xor_sync(0xffffffffu, v, o);
            v = w > v ? w : v;
        }
        return v;
    }
}

// k-th largest key (1 <= k <= number of taking items) over items t in [0, n):
// getkey(t, key) returns false for items that do not take part.  Returns the
// key and sets *krem to how many items equal to it are needed.  A first pass
// finds the keys' range; the bits above the highest bit in which the smallest
// and largest keys differ are common to every key, so the digit passes (8 bits
// each) start right below them, where the keys spread.  Each warp counts into
// its own histogram (shared-memory atomics), then the warps' counts are summed.
template <typename KeyT, typename Get>
__device__ KeyT block_kth_largest(Get getkey, int n, int k, RadixSmem& rs, int* krem_out) {
    constexpr int BITS = sizeof(KeyT) * 8;
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    int* wh = rs.whist + (threadIdx.x >> 5) * 256;
    // ---- key range
    if (threadIdx.x == 0) {
        rs.kmin = ~0ull;
        rs.kmax = 0ull;
    }
    __syncthreads();
    {
        KeyT lo = (KeyT)~(KeyT)0, hi = 0;
        for (int t0 = threadIdx.x; t0 < n; t0 += 8 * blockDim.x) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = t0 + u * blockDim.x;
                KeyT key;
                if (t < n && getkey(t, key)) {
                    lo = key < lo ? key : lo;
                    hi = key > hi ? key : hi;
                }
            }
        }
        lo = warp_min_key(lo);
        hi = warp_max_key(hi);
        if (lane == 0) {
            atomicMin(&rs.kmin, (unsigned long long)lo);
            atomicMax(&rs.kmax, (unsigned long long)hi);
        }
    }
    __syncthreads();
    const KeyT kmin = (KeyT)rs.kmin, kmax = (KeyT)rs.kmax;
    const KeyT diff = kmin ^ kmax;
    int krem = k;
    if (diff == 0 || kmin > kmax) {               // one distinct key (or nothing takes part)
        __syncthreads();
        *krem_out = krem;
        return kmax;
    }
    int top = BITS - 1;                           // highest bit not yet fixed
    while (((diff >> top) & 1) == 0) --top;
    const KeyT common = top == BITS - 1 ? (KeyT)0 : (KeyT)(~(KeyT)0) << (top + 1);
    KeyT prefix = kmin & common, mask = common;
    while (top >= 0) {
        const int width = top + 1 < 8 ? top + 1 : 8;
        const int shift = top - width + 1;
        const KeyT dmask = (KeyT)((1u << width) - 1u);
        for (int i = threadIdx.x; i < nw * 256; i += blockDim.x) rs.whist[i] = 0;
        __syncthreads();
        // keys fetched 8 at a time ahead of the atomics, so their loads overlap
        for (int t0 = threadIdx.x; t0 < n; t0 += 8 * blockDim.x) {
            KeyT kk[8];
            bool in[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = t0 + u * blockDim.x;
                in[u] = t < n && getkey(t, kk[u]);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (in[u] && (kk[u] & mask) == prefix) atomicAdd(&wh[(int)((kk[u] >> shift) & dmask)], 1);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < 256; i += blockDim.x) {
            int c = 0;
            for (int w = 0; w < nw; ++w) c += rs.whist[w * 256 + i];
            rs.hist[i] = c;
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            int c = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) c += rs.hist[255 - 8 * lane - i];   // lane 0 holds the top bins
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= krem);
            const int L = __ffs(hit) - 1;
            if (lane == L) {
                int cum = incl - c;
                for (int i = 0; i < 8; ++i) {
                    const int d = 255 - 8 * lane - i;
                    if (cum + rs.hist[d] >= krem) {
                        rs.ctl[1] = d;
                        rs.ctl[2] = krem - cum;
                        break;
                    }
                    cum += rs.hist[d];
                }
            }
        }
        __syncthreads();
        prefix |= (KeyT)rs.ctl[1] << shift;
        mask |= dmask << shift;
        krem = rs.ctl[2];
        __syncthreads();
        top = shift - 1;
    }
    *krem_out = krem;
    return prefix;
}

// the float whose order-preserving key (f32_key) is k
__device__ __forceinline__ float key_value(unsigned int k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// A band [lo, hi] of keys that holds the k-th largest of the keys
// (order-preserving images of finite floats, 1 <= k <= number of finite ones
// taking part): every key above hi is among the k largest, every key below lo
// is not.  The value range of the keys is
// cut into 256 buckets of equal width in value (the bucket index never
// decreases as the value grows, so every key of a higher bucket is larger);
// the bucket holding the k-th largest is found from the top; while it still
// holds more than 64 keys its own range is cut again (at most four levels).
// The band is the smallest and largest key of the last bucket.  Non-finite keys
// (an empty slot's -inf) stay below every bucket.  Used where the caller only
// filters with it: even buckets spread the shared-memory atomics (one
// histogram for the block), and the refinement keeps the band to a few dozen keys.
// The band search from a known range: lo / hi are the smallest and largest
// finite keys taking part, rs.hist is zero and a block barrier has passed since
// both were set.  Each level is three block phases: histogram, scan (warp 0),
// then the range of the chosen bucket (which also clears the histogram for the
// next level).
template <typename Get>
__device__ uint2 block_kth_band_from(Get getkey, int n, int k, unsigned int lo, unsigned int hi, RadixSmem& rs) {
    const int lane = threadIdx.x & 31;
    auto bucket_of = [](unsigned int key, float vlo, float scale) {
        return min((int)((key_value(key) - vlo) * scale), 255);
    };
    int need = k;
    for (int level = 0; level < 4 && lo < hi; ++level) {
        const float vlo = key_value(lo);
        float scale = 256.0f / (key_value(hi) - vlo);
        if (!(scale > 0.0f && scale < INFINITY)) scale = 0.0f;       // degenerate range: one bucket
        for (int t0 = threadIdx.x; t0 < n; t0 += 8 * blockDim.x) {
            unsigned int kk[8];
            bool in[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = t0 + u * blockDim.x;
                in[u] = t < n && getkey(t, kk[u]);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (in[u] && kk[u] >= lo && kk[u] <= hi) atomicAdd(&rs.hist[bucket_of(kk[u], vlo, scale)], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            int c = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) c += rs.hist[255 - 8 * lane - i];   // lane 0 holds the top bins
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
            const int L = hit ? __ffs(hit) - 1 : 31;
            if (lane == L) {
                int cum = incl - c, d = 255 - 8 * lane - 7;
                for (int i = 0; i < 8; ++i) {
                    const int dd = 255 - 8 * lane - i;
                    if (cum + rs.hist[dd] >= need) {
                        d = dd;
                        break;
                    }
                    cum += rs.hist[dd];
                }
                rs.ctl[1] = d;
                rs.ctl[2] = need - cum;
                rs.ctl[3] = rs.hist[d];
            }
            if (lane == 0) {
                rs.kmin32 = ~0u;
                rs.kmax32 = 0u;
            }
        }
        __syncthreads();
        const int bstar = rs.ctl[1], cnt = rs.ctl[3];
        need = rs.ctl[2];
        for (int i = threadIdx.x; i < 256; i += blockDim.x) rs.hist[i] = 0;
        // min / max of the keys of bucket bstar
        unsigned int mn = ~0u, mx = 0u;
        for (int t0 = threadIdx.x; t0 < n; t0 += 8 * blockDim.x) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = t0 + u * blockDim.x;
                unsigned int key;
                if (t < n && getkey(t, key) && key >= lo && key <= hi && isfinite(key_value(key)) &&
                    bucket_of(key, vlo, scale) == bstar) {
                    mn = min(mn, key);
                    mx = max(mx, key);
                }
            }
        }
        mn = __reduce_min_sync(0xffffffffu, mn);
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (lane == 0) {
            atomicMin(&rs.kmin32, mn);
            atomicMax(&rs.kmax32, mx);
        }
        __syncthreads();
        lo = rs.kmin32;
        hi = rs.kmax32;
        if (cnt <= 64 || scale == 0.0f) break;
    }
    __syncthreads();
    return make_uint2(lo, hi);
}

// A band [lo, hi] of keys that holds the k-th largest of the keys
// (order-preserving images of finite floats, 1 <= k <= number of finite ones
// taking part): every key above hi is among the k largest, every key below lo
// is not.  The value range of the keys is
// cut into 256 buckets of equal width in value (the bucket index never
// decreases as the value grows, so every key of a higher bucket is larger);
// the bucket holding the k-th largest is found from the top; while it still
// holds more than 64 keys its own range is cut again (at most four levels).
// The band is the smallest and largest key of the last bucket.  Non-finite keys
// (an empty slot's -inf) stay below every bucket.  Used where the caller only
// filters with it: even buckets spread the shared-memory atomics (one
// histogram for the block), and the refinement keeps the band to a few dozen keys.
template <typename Get>
__device__ uint2 block_kth_band(Get getkey, int n, int k, RadixSmem& rs) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        rs.kmin32 = ~0u;
        rs.kmax32 = 0u;
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x) rs.hist[i] = 0;
    __syncthreads();
    unsigned int mn = ~0u, mx = 0u;
    for (int t0 = threadIdx.x; t0 < n; t0 += 8 * blockDim.x) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int t = t0 + u * blockDim.x;
            unsigned int key;
            if (t < n && getkey(t, key) && isfinite(key_value(key))) {
                mn = min(mn, key);
                mx = max(mx, key);
            }
        }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
        atomicMin(&rs.kmin32, mn);
        atomicMax(&rs.kmax32, mx);
    }
    __syncthreads();
    return block_kth_band_from(getkey, n, k, rs.kmin32, rs.kmax32, rs);
}

// the band's lower end (a key <= the k-th largest) or upper end (>= it)
template <typename Get>
__device__ unsigned int block_kth_bound(Get getkey, int n, int k, bool upper, RadixSmem& rs) {
    const uint2 band = block_kth_band(getkey, n, k, rs);
    return upper ? band.y : band.x;
}

// The smallest key of the bucket that holds the k-th largest of the keys, cutting their value range
// into 2048 buckets of equal width: at least k keys are >= it, so it never exceeds the k-th largest
// (1 <= k <= the number of finite keys taking part; non-finite keys are ignored).  One pass for the
// range, one for the histogram (rs.whist: 2048 counters), one block scan from the top bucket down,
// one pass for the bucket's smallest key.  Used where the caller only filters with it.
template <typename Get>
__device__ unsigned int block_kth_floor(Get getkey, int n, int k, RadixSmem& rs) {
    constexpr int NB = 2048;
    int* hist = rs.whist;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        rs.kmin32 = ~0u;
        rs.kmax32 = 0u;
        rs.ctl[1] = 0;
    }
    for (int i = threadIdx.x; i < NB; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    unsigned int mn = ~0u, mx = 0u;
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
        unsigned int key;
        if (getkey(t, key) && isfinite(key_value(key))) {
            mn = min(mn, key);
            mx = max(mx, key);
        }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
        atomicMin(&rs.kmin32, mn);
        atomicMax(&rs.kmax32, mx);
    }
    __syncthreads();
    const unsigned int lo = rs.kmin32, hi = rs.kmax32;
    if (lo > hi) return 0u;                                    // no finite key: keep everything
    const float vlo = key_value(lo);
    float scale = (float)NB / (key_value(hi) - vlo);
    if (!(scale > 0.0f && scale < INFINITY)) return lo;         // one value (or too narrow to cut): lo
    auto bucket_of = [&](unsigned int key) { return min((int)((key_value(key) - vlo) * scale), NB - 1); };
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
        unsigned int key;
        if (getkey(t, key) && key >= lo && key <= hi) atomicAdd(&hist[bucket_of(key)], 1);
    }
    if (threadIdx.x == 0) rs.kmax32 = ~0u;                      // (every thread has read hi)
    __syncthreads();
    // thread i sums buckets NB-1-PB*i down to NB-PB*(i+1); an inclusive scan over the threads counts
    // from the top bucket down
    const int PB = NB / (int)blockDim.x;
    int c = 0;
    for (int j = 0; j < PB; ++j) c += hist[NB - 1 - PB * (int)threadIdx.x - j];
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) rs.hist[warp] = incl;
    __syncthreads();
    for (int w = 0; w < warp; ++w) incl += rs.hist[w];
    const int excl = incl - c;
    if (excl < k && incl >= k) {
        int cum = excl;
        for (int j = 0; j < PB; ++j) {
            const int b = NB - 1 - PB * (int)threadIdx.x - j;
            cum += hist[b];
            if (cum >= k) {
                rs.ctl[1] = b;
                break;
            }
        }
    }
    __syncthreads();
    const int bstar = rs.ctl[1];
    mn = ~0u;
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
        unsigned int key;
        if (getkey(t, key) && key >= lo && key <= hi && bucket_of(key) == bstar) mn = min(mn, key);
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    if (lane == 0) atomicMin(&rs.kmax32, mn);
    __syncthreads();
    const unsigned int r = rs.kmax32;
    __syncthreads();                                          // rs is reused by the caller
    return r == ~0u ? lo : r;
}

// block_kth_bound over the keys of an array: the largest of keys32[st t .. st t + st - 1] (st >= 1;
// the array holds at least st n keys), or (keys32 null) the high word of keys64[t].  Not inlined:
// the selections that take it share one copy of the band search.
// known_range: the caller passes the smallest and largest finite key as lo / hi, and rs.hist is zero
// and a block barrier has passed since both were set (the range pass is skipped).
static __device__ __noinline__ unsigned int block_kth_bound_arr(const unsigned int* keys32, const unsigned long long* keys64,
                                                         int n, int k, bool upper, RadixSmem& rs, int st = 1,
                                                         bool known_range = false, unsigned int lo = 0u,
                                                         unsigned int hi = 0u) {
    auto getkey = [&](int t, unsigned int& key) {
        if (keys32) {
            key = keys32[st * t];
            for (int i = 1; i < st; ++i) key = max(key, keys32[st * t + i]);
        } else {
            key = (unsigned int)(keys64[t] >> 32);
        }
        return true;
    };
    if (!known_range) {
        const int lane = threadIdx.x & 31;
        if (threadIdx.x == 0) {
            rs.kmin32 = ~0u;
            rs.kmax32 = 0u;
        }
        for (int i = threadIdx.x; i < 256; i += blockDim.x) rs.hist[i] = 0;
        __syncthreads();
        unsigned int mn = ~0u, mx = 0u;
        for (int t = threadIdx.x; t < n; t += blockDim.x) {
            unsigned int key;
            if (getkey(t, key) && isfinite(key_value(key))) {
                mn = min(mn, key);
                mx = max(mx, key);
            }
        }
        mn = __reduce_min_sync(0xffffffffu, mn);
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (lane == 0) {
            atomicMin(&rs.kmin32, mn);
            atomicMax(&rs.kmax32, mx);
        }
        __syncthreads();
        lo = rs.kmin32;
        hi = rs.kmax32;
    }
    const uint2 band = block_kth_band_from(getkey, n, k, lo, hi, rs);
    return upper ? band.y : band.x;
}

// warp-aggregated append to a list whose counter lives at *ctr (shared or global)
__device__ __forceinline__ int append_slot(bool flag, int* ctr) {
    const unsigned m = __ballot_sync(0xffffffffu, flag);
    if (!m) return -1;
    const int lane = threadIdx.x & 31, leader = __ffs(m) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(ctr, __popc(m));
    base = __shfl_sync(0xffffffffu, base, leader);
    return flag ? base + __popc(m & ((1u << lane) - 1u)) : -1;
}


// Block-wide append of the items i in [0, n) with flag(i) to a list in global
// memory whose length counter is *gctr: the block counts its items per warp,
// reserves them with ONE global atomic, then every warp places its items
// (put(slot, i)) in order from its own offset, by ballots (no atomics).
// Every thread of the block calls it; rs.hist serves as scratch (the band
// searches clear it before use).
template <typename Flag, typename Put>
__device__ void block_append_global(int n, Flag flag, Put put, int* gctr, RadixSmem& rs) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int c = 0;
    for (int i0 = 0; i0 < n; i0 += blockDim.x) {
        const int i = i0 + threadIdx.x;
        c += (i < n && flag(i)) ? 1 : 0;
    }
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) rs.hist[warp] = c;
    __syncthreads();
    if (warp == 0) {
        const int v = lane < nw ? rs.hist[lane] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int tot = __shfl_sync(0xffffffffu, incl, 31);
        int g = 0;
        if (lane == 0 && tot) g = atomicAdd(gctr, tot);
        g = __shfl_sync(0xffffffffu, g, 0);
        if (lane < nw) rs.hist[32 + lane] = g + incl - v;
    }
    __syncthreads();
    int pos = rs.hist[32 + warp];
    for (int i0 = 0; i0 < n; i0 += blockDim.x) {
        const int i = i0 + threadIdx.x;
        const bool f = i < n && flag(i);
        const unsigned m = __ballot_sync(0xffffffffu, f);
        if (f) put(pos + __popc(m & ((1u << lane) - 1u)), i);
        pos += __popc(m);
    }
    __syncthreads();
}

// After a scan block has the (S~-E, S~+E) bounds of its chunk in shared memory
// (lu[0..E), entries c0..c0+E-1), forward to the query's global lists every
// entry whose upper bound reaches (a lower bound of) the chunk's k-th largest
// lower bound, and
// likewise for HSI blocks (bounds = max over members; the newest block, which
// is always kept, is not forwarded).  The global k-th lower bound is never
// smaller than a chunk's, so nothing the exact selection needs is dropped.
static __device__ void forward_candidates(const float2* lu, int c0, int E, int n_elig, int k, int pool_blocks, int bs,
                                   int64_t slab, int list_len, int* counts, int* cid, float2* clu, int* bid,
                                   float2* blu, RadixSmem& rs) {
    const int n_loc = min(max(n_elig - c0, 0), E);
    if (n_loc == 0) return;                       // uniform
    if (threadIdx.x == 0) rs.ctl[4] = 0;
    __syncthreads();
    unsigned int lam = 0u;                        // <= the chunk's k-th largest lower bound
    if (n_loc > k)
        lam = block_kth_floor(
            [&](int i, unsigned int& key) {
                key = f32_key(lu[i].x);
                return true;
            },
            n_loc, k, rs);
    block_append_global(
        n_loc, [&](int i) { return f32_key(lu[i].y) >= lam; },
        [&](int pos, int i) {
            cid[slab * list_len + pos] = c0 + i;
            clu[slab * list_len + pos] = lu[i];
        },
        counts + 2 * slab, rs);
    if (pool_blocks > 1) {
        const int nb = (n_elig + bs - 1) / bs;           // blocks of this query
        const int forced = nb - 1;
        const int g0 = c0 / bs;                           // first block of the chunk (E is a multiple of bs)
        const int nbl = min(E / bs, nb - g0);             // blocks of this chunk that exist
        const int nvalid = nbl - ((forced >= g0 && forced < g0 + nbl) ? 1 : 0);
        if (nb > pool_blocks && nvalid > 0) {
            // block bounds (max over members) computed once and written over lu[0..nbl) when
            // every thread holds at most four blocks (each reads its members before any is
            // overwritten); otherwise taken from the members at each use
            float2* lub = const_cast<float2*>(lu);
            const bool cached = nbl <= 4 * (int)blockDim.x;
            auto members = [&](int bl) {
                float2 m2 = make_float2(-INFINITY, -INFINITY);
                for (int i = 0; i < bs; ++i) {
                    const int e = bl * bs + i;
                    if (e < n_loc) {
                        m2.x = fmaxf(m2.x, lu[e].x);
                        m2.y = fmaxf(m2.y, lu[e].y);
                    }
                }
                return m2;
            };
            if (cached) {
                float2 mine[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int bl = threadIdx.x + q * blockDim.x;
                    mine[q] = bl < nbl ? members(bl) : make_float2(-INFINITY, -INFINITY);
                }
                __syncthreads();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int bl = threadIdx.x + q * blockDim.x;
                    if (bl < nbl) lub[bl] = mine[q];
                }
                __syncthreads();
            }
            auto blk = [&](int bl, bool upper) {
                const float2 m2 = cached ? lub[bl] : members(bl);
                return upper ? m2.y : m2.x;
            };
            unsigned int lamb = 0u;
            if (nvalid > pool_blocks - 1)
                lamb = block_kth_floor(
                    [&](int bl, unsigned int& key) {
                        key = f32_key(blk(bl, false));
                        return g0 + bl != forced;
                    },
                    nbl, pool_blocks - 1, rs);
            block_append_global(
                nbl, [&](int bl) { return g0 + bl != forced && f32_key(blk(bl, true)) >= lamb; },
                [&](int pos, int bl) {
                    bid[slab * list_len + pos] = g0 + bl;
                    blu[slab * list_len + pos] = make_float2(blk(bl, false), blk(bl, true));
                },
                counts + 2 * slab + 1, rs);
        }
    }
}

}  // namespace csa2

// Multi-query Full indexer scan on the tensor cores, for a chunked prefill
// ("DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる", §2.3.1 lightweight
// indexer over FP4 keys; §2.3.4 a Full layer scores every causally visible entry).
//
// One block takes MQ_QB = 4 consecutive queries of the chunk and every entry
// any of them may read, 128 entries a tile:
//   A = key codes  [128 entries x 128 dims] FP4 E2M1 (kind::f8f6f4 layout: each
//       16-value group is 8 packed bytes followed by 8 pad bytes)
//   B = block-diagonal queries [4 queries x 8 heads x 8 groups = 256 rows x 128]:
//       row (q, h, g) holds query q's head-h codes of group g, zeros elsewhere
//   D = A . B^T   M = 128, N = 256, K = 128   (fp32 in TMEM, two accumulators)
// D[e][(q,h,g)] is an exact group sum, so the epilogue forms every (entry,
// query) score S~ and its rounding bound E exactly as the single-query scans do.
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
// Warps (384 threads): 0-7 epilogue (warp w: TMEM lane quarter w%4, queries
// 2(w/4) and 2(w/4)+1), 8 lane 0 issues the MMAs, 9 lane 0 the 1-D bulk copies
// of each tile's contiguous key rows (four tiles in flight), 10-11 expand the
// packed codes into the MMA layout.
#include "indexer_common.cuh"
#include "umma.cuh"

namespace csa2 {

constexpr int MQ_QB = 4;
constexpr int MQ_TILE = 128;
constexpr int MQ_DI = 128;
constexpr int MQ_G = MQ_DI / 16;
constexpr int MQ_H = 8;
constexpr int MQ_N = MQ_QB * MQ_H * MQ_G;                 // 256
constexpr int MQ_NR = 4;                                  // raw staging slots
constexpr int MQ_NA = 2;                                  // MMA-layout A slots
constexpr int MQ_SAMPLE_TILES = 32;
constexpr int MQ_THREADS = 384;
constexpr int MQ_EPI = 256;
constexpr int MQ_XF = 64;
constexpr uint32_t MQ_RAW_SLOT = MQ_TILE * (MQ_DI / 2) + MQ_TILE * 8;          // codes 8 KB + scales 1 KB
constexpr uint32_t MQS_B = 0;                                                   // 256 rows x 128 B
constexpr uint32_t MQS_A = MQ_N * 128;                                          // 2 x 16 KB
constexpr uint32_t MQS_RAW = MQS_A + MQ_NA * MQ_TILE * 128;                     // 4 x 9 KB
constexpr uint32_t MQS_SAMP = MQS_RAW + MQ_NR * MQ_RAW_SLOT;                    // [QB][32 x 128] lower bounds
constexpr uint32_t MQS_Q = MQS_SAMP + MQ_QB * MQ_SAMPLE_TILES * MQ_TILE * 4;    // sq [QB][64], w [QB][8]
constexpr uint32_t MQS_END = MQS_Q + MQ_QB * (MQ_H * MQ_G + MQ_H) * 4;
constexpr uint32_t MQS_DYN = MQS_END + 1024;

__device__ __forceinline__ uint32_t mq_swz(uint32_t row, uint32_t unit) { return row * 128 + ((unit ^ (row & 7)) << 4); }

__global__ void __launch_bounds__(MQ_THREADS, 1) k_scan_mq_tc(
    const uint8_t* __restrict__ kc_all, const uint8_t* __restrict__ ks_all, int capacity,
    const uint8_t* __restrict__ iq_codes, const uint8_t* __restrict__ iq_scales, const float* __restrict__ w_head,
    const int64_t* __restrict__ q_pos, int n_q, int q0, int n_qc, int k, int* __restrict__ counts,
    int* __restrict__ cid, float2* __restrict__ clu, int list_len, int* __restrict__ err, int ratio) {
    pdl_wait();
    extern __shared__ uint8_t dyn[];
    __shared__ __align__(8) unsigned long long bar_rfull[MQ_NR], bar_rfree[MQ_NR], bar_afull[MQ_NA], bar_afree[MQ_NA],
        bar_dfull[2], bar_dfree[2];
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
    // query operand: row n = (q, h, g) -> unit g holds query q's 8 code bytes of head h, group g
    for (int i = tid; i < MQ_N * 8; i += MQ_THREADS) {
        const int n = i >> 3, u = i & 7;
        const int q = n >> 6, h = (n >> 3) & 7, g = n & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (u == g && q < nqb) {
            const int64_t gq = (int64_t)b * n_q + q0 + qa + q;
            const uint2 c = *reinterpret_cast<const uint2*>(iq_codes + (gq * MQ_H + h) * (MQ_DI / 2) + g * 8);
            v.x = c.x;
            v.y = c.y;
        }
        *reinterpret_cast<uint4*>(sm + MQS_B + mq_swz(n, u)) = v;
    }
    float* sq = reinterpret_cast<float*>(sm + MQS_Q);               // [QB][64]
    float* ww = sq + MQ_QB * MQ_H * MQ_G;                            // [QB][8]
    for (int i = tid; i < MQ_QB * MQ_H * MQ_G; i += MQ_THREADS) {
        const int q = i >> 6;
        sq[i] = q < nqb ? e4m3_to_f32(iq_scales[((int64_t)b * n_q + q0 + qa + q) * (MQ_H * MQ_G) + (i & 63)]) : 0.0f;
    }
    for (int i = tid; i < MQ_QB * MQ_H; i += MQ_THREADS) {
        const int q = i >> 3;
        ww[i] = q < nqb ? w_head[((int64_t)b * n_q + q0 + qa + q) * MQ_H + (i & 7)] : 0.0f;
    }
    // the pad half of every 16-byte unit of the A slots stays zero
    for (int i = tid; i < MQ_NA * MQ_TILE * 8; i += MQ_THREADS)
        reinterpret_cast<uint4*>(sm + MQS_A)[i] = make_uint4(0, 0, 0, 0);
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
    const float fac = bound_factor(MQ_H, MQ_DI);
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
        if (warp == 9) {
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
        } else if (warp >= 10) {
            // ---- expand packed codes into the data half of each 16-byte unit
            const int xt = tid - 320;
            for (int v = v0; v < v_end && ok; ++v) {
                const int r = v % MQ_NR, a = v % MQ_NA;
                ok &= umma::mbar_wait(umma::smem_u32(&bar_rfull[r]), (v / MQ_NR) & 1);
                if (v >= MQ_NA) ok &= umma::mbar_wait(umma::smem_u32(&bar_afree[a]), ((v / MQ_NA) - 1) & 1);
                if (!ok) break;
                const uint4* rw = reinterpret_cast<const uint4*>(sm + MQS_RAW + r * MQ_RAW_SLOT);
                uint8_t* as = sm + MQS_A + a * (MQ_TILE * 128);
#pragma unroll 4
                for (int c = xt; c < MQ_TILE * 4; c += MQ_XF) {
                    const int row = c >> 2, q4 = c & 3;
                    const uint4 x = rw[c];
                    *reinterpret_cast<uint2*>(as + mq_swz(row, 2 * q4)) = make_uint2(x.x, x.y);
                    *reinterpret_cast<uint2*>(as + mq_swz(row, 2 * q4 + 1)) = make_uint2(x.z, x.w);
                }
                umma::fence_proxy_async();
                umma::mbar_arrive(umma::smem_u32(&bar_afull[a]));
            }
        } else if (warp == 8) {
            // ---- MMA issuer
            if (lane == 0) {
                const uint32_t idesc = (1u << 4) | (5u << 7) | (5u << 10) | ((uint32_t)(MQ_N >> 3) << 17) |
                                       ((uint32_t)(MQ_TILE >> 4) << 24);
                for (int v = v0; v < v_end && ok; ++v) {
                    const int s = v % MQ_NA, d = v & 1;
                    ok &= umma::mbar_wait(umma::smem_u32(&bar_afull[s]), (v / MQ_NA) & 1);
                    if (v >= 2) ok &= umma::mbar_wait(umma::smem_u32(&bar_dfree[d]), ((v >> 1) - 1) & 1);
                    if (!ok) break;
                    umma::fence_after();
#pragma unroll
                    for (int ks = 0; ks < MQ_DI / 32; ++ks) {
                        const uint64_t ad = umma::desc(base + MQS_A + s * (MQ_TILE * 128) + ks * 32, 16, 1024,
                                                       umma::LAYOUT_SW128);
                        const uint64_t bd = umma::desc(base + MQS_B + ks * 32, 16, 1024, umma::LAYOUT_SW128);
                        asm volatile(
                            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                            " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(tmem + 256 * d),
                            "l"(ad), "l"(bd), "r"(idesc), "r"(ks));
                    }
                    umma::commit(umma::smem_u32(&bar_dfull[d]));
                    umma::commit(umma::smem_u32(&bar_afree[s]));
                }
            }
        } else {
            // ---- epilogue: one entry (TMEM lane) and two queries per thread
            const int qd = warp & 3, qp = warp >> 2;
            const int r = qd * 32 + lane;
            int cge[2] = {0, 0};
            for (int v = v0; v < v_end && ok; ++v) {
                const int rs = v % MQ_NR, d = v & 1;
                const int e0 = tile_of(v) * MQ_TILE;
                const int rows = min(MQ_TILE, nmax - e0);
                const int e = e0 + r;
                ok &= umma::mbar_wait(umma::smem_u32(&bar_dfull[d]), (v >> 1) & 1);
                // the scales landed with this slot's bulk copy: observe that barrier phase too
                if (bulk_scales) ok &= umma::mbar_wait(umma::smem_u32(&bar_rfull[rs]), (v / MQ_NR) & 1);
                if (!ok) break;
                umma::fence_after();
                uint2 skw = make_uint2(0, 0);
                if (bulk_scales && r < (rows & ~1))
                    skw = *reinterpret_cast<const uint2*>(sm + MQS_RAW + rs * MQ_RAW_SLOT + MQ_TILE * (MQ_DI / 2) + r * 8);
                else if (r < rows)
                    skw = __ldg(reinterpret_cast<const uint2*>(ks_all + ((int64_t)b * capacity + e) * MQ_G));
                umma::mbar_arrive(umma::smem_u32(&bar_rfree[rs]));
                float skf[MQ_G];
#pragma unroll
                for (int g = 0; g < MQ_G; ++g) skf[g] = e4m3_to_f32(((g < 4 ? skw.x : skw.y) >> (8 * (g & 3))) & 255u);
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int qi = 2 * qp + qq;
                    float dv[64];
                    const uint32_t tb = tmem + ((uint32_t)(qd * 32) << 16) + 256 * d + 64 * qi;
#pragma unroll
                    for (int c = 0; c < 64; c += 16) umma::tmem_ld16(tb + c, dv + c);
                    umma::tmem_wait_ld();
                    if (qq == 1) {
                        umma::fence_before();
                        umma::mbar_arrive(umma::smem_u32(&bar_dfree[d]));
                    }
                    if (qi >= nqb) continue;                   // warp-uniform
                    const float* sqq = sq + qi * 64;
                    const float* wq = ww + qi * MQ_H;
                    float S = 0.0f, Bs = 0.0f;
#pragma unroll
                    for (int h = 0; h < MQ_H; ++h) {
                        float dd = 0.0f, A = 0.0f;
#pragma unroll
                        for (int g = 0; g < MQ_G; ++g) {
                            // dv * sq is exact (a multiple of 1/4 below 2^10 times an E4M3 value), and
                            // so is its product with the key scale inside the fma: the same sums as
                            // adding t = dv * (sq * sk) one by one
                            const float x = dv[h * MQ_G + g] * sqq[h * MQ_G + g];
                            dd = __fmaf_rn(skf[g], x, dd);
                            A = __fmaf_rn(skf[g], fabsf(x), A);
                        }
                        S = __fmaf_rn(wq[h], fmaxf(dd, 0.0f), S);
                        Bs = __fmaf_rn(fabsf(wq[h]), A, Bs);
                    }
                    const float E = Bs * fac;
                    const float L = S - E, U = S + E;
                    const bool elig = e < s_nel[qi];
                    const int64_t slab = (int64_t)b * n_qc + qa + qi;
                    if (phase == 0) {
                        samp[qi * (MQ_SAMPLE_TILES * MQ_TILE) + (v - v0) * MQ_TILE + r] = elig ? L : -INFINITY;
                    } else {
                        const uint32_t tau = s_tau[qi];
                        const bool fwd = elig && (phase == 1 ? f32_key(U) >= tau : s_retry[qi] != 0);
                        if (phase == 1) cge[qq] += (elig && f32_key(L) >= tau) ? 1 : 0;
                        const int pos = append_slot(fwd, counts + 2 * slab);
                        if (fwd) {
                            cid[slab * list_len + pos] = e;
                            clu[slab * list_len + pos] = make_float2(L, U);
                        }
                    }
                }
            }
            if (phase == 1) {
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int c = __reduce_add_sync(0xffffffffu, cge[qq]);
                    if (lane == 0 && c) atomicAdd(&s_cnt[2 * qp + qq], c);
                }
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
    if (warp == 9 && lane == 0 && !ok) {
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

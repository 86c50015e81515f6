/*
 * CSA2 decode oracle: plain, slow, fp64 CPU restatement of what the hot path
 * computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg use it; the library never does.  It shares no
 * code, header, table or constant with the CUDA sources.
 *
 * Sources (page titles and sections):
 *  [P1] "DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる" (hackernews.jp):
 *       §1.1 (512-dim shared latent, encoder 2:1 channel-wise merge, FP4 KV),
 *       §2.3.1 (indexer Q x indexer K scores main-KV entries, top-k per query,
 *       each Q also attends to the local SWA window; compressor without overlap
 *       or absolute position embedding), §2.3.2 (Full / Reindex / Reuse),
 *       §2.3.4 (HSI: per-block max of the Full layer's scores, newest block
 *       forced in, blocks expanded to a candidate pool).
 *  [P2] ai.freelance-job.com summary, spec table (latent 512, window 128) and
 *       the CSA2 paragraph (top-k 512).
 *  [P3] "DeepSeek V4.1 Flash architecture: making a giant AI faster through
 *       reuse" (yasmorita.com): causal mask; Q·K scores turned into weights
 *       that sum to 1, then a weighted sum of V; MQA shares one K/V set.
 *
 * The pages fix no number format, score formula or tie rule; the readings used
 * here (E2M1 codes with one E4M3 scale per 16 values, score = sum_h w_h *
 * ReLU(q_h . k_j), ties to the lower index, fp32 merge by one fused
 * multiply-add) are listed with the rest of the design notes.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off (no fused contractions other than
 * the explicit fma()/fmaf() calls below).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* ------------------------------------------------------------------------ */
/* number formats                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1 (FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * Magnitudes written out from the bit fields: exponent 0 is subnormal
 * (mantissa * 0.5), exponent e>0 gives (1 + m/2) * 2^(e-1). */
double orc_e2m1_value(int nibble) {
    int s = (nibble >> 3) & 1, e = (nibble >> 1) & 3, m = nibble & 1;
    double mag = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (OCP FP8, "fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinity. */
double orc_e4m3_value(int byte) {
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? (m / 8.0) * ldexp(1.0, -6) : (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest non-negative finite E4M3 value to v >= 0, ties to the even code,
 * values beyond the largest finite value (448) saturate to it.  Written as a
 * scan over all 127 non-negative finite codes in increasing order. */
int orc_e4m3_encode(float v) {
    double x = (double)v;
    if (x >= 448.0) return 0x7e;       /* saturate: nothing larger is finite */
    int best = 0;
    double best_err = fabs(orc_e4m3_value(0) - x);
    for (int c = 1; c <= 0x7e; ++c) {
        double err = fabs(orc_e4m3_value(c) - x);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return best;
}

/* FP4 code of x for scale s > 0: the magnitude m in {0,.5,1,1.5,2,3,4,6} whose
 * m*s is nearest to |x| (ties to the even code, |x| > 6s saturates to 6); the
 * sign bit is set only for a nonzero magnitude (zero is always written +0). */
int orc_e2m1_encode(float x, double s) {
    double ax = fabs((double)x);
    if (ax >= 6.0 * s) return (x < 0.0f) ? 15 : 7;   /* saturate at the largest magnitude */
    int best = 0;
    double best_err = ax;  /* distance to magnitude 0 */
    for (int c = 1; c <= 7; ++c) {
        double err = fabs(orc_e2m1_value(c) * s - ax);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    if (best != 0 && x < 0.0f) best |= 8;
    return best;
}

/* Quantise rows of d floats (d a multiple of 16): per group of 16 consecutive
 * values, scale byte = E4M3(float(amax / 6)), codes = E2M1(x / scale); a scale
 * that encodes to zero makes every code of its group zero.  Codes are packed
 * two per byte: element 2i in the low nibble, element 2i+1 in the high one. */
void orc_quantize_rows(const float* x, int64_t rows, int d, uint8_t* codes, uint8_t* scales) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * d;
        uint8_t* cr = codes + r * (d / 2);
        uint8_t* sr = scales + r * (d / 16);
        for (int g = 0; g < d / 16; ++g) {
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(xr[g * 16 + i]);
                if (a > amax) amax = a;
            }
            float v = amax / 6.0f;
            int sb = orc_e4m3_encode(v);
            double s = orc_e4m3_value(sb);
            sr[g] = (uint8_t)sb;
            for (int i = 0; i < 16; i += 2) {
                int lo = (s > 0.0) ? orc_e2m1_encode(xr[g * 16 + i], s) : 0;
                int hi = (s > 0.0) ? orc_e2m1_encode(xr[g * 16 + i + 1], s) : 0;
                cr[(g * 16 + i) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* Dequantise rows back to doubles: value = E2M1(code) * E4M3(scale), exact. */
void orc_dequant_rows(const uint8_t* codes, const uint8_t* scales, int64_t rows, int d, double* out) {
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < d; ++i) {
            uint8_t byte = codes[r * (d / 2) + i / 2];
            int nib = (i & 1) ? (byte >> 4) : (byte & 15);
            out[r * d + i] = orc_e2m1_value(nib) * orc_e4m3_value(scales[r * (d / 16) + i / 16]);
        }
}

static float bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------------ */
/* cache write: 2:1 channel-wise merge, then FP4 quantisation                */
/* [P1] §1.1 and §2.3.1: two adjacent positions merge into one entry with    */
/* learned channel-wise weights, no overlap between entries, no absolute     */
/* position embedding; main KV and indexer keys are stored in FP4.           */
/* ------------------------------------------------------------------------ */

/* e[i][c] = fmaf(w1[c], h[2i+1][c], float(w0[c] * h[2i][c])) */
void orc_merge_pairs(const uint16_t* h, int64_t n_entries, int d, const float* w0, const float* w1, float* e) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n_entries; ++i)
        for (int c = 0; c < d; ++c) {
            float h0 = bf16_value(h[(2 * i) * d + c]);
            float h1 = bf16_value(h[(2 * i + 1) * d + c]);
            float p0 = w0[c] * h0;
            e[i * d + c] = fmaf(w1[c], h1, p0);
        }
}

/* One sequence: n_pos raw positions (even) -> n_pos/2 entries of latent codes
 * and scales; the raw indexer-key rows (bf16, one per entry) are quantised with
 * the same codec. */
void orc_cache_write(const uint16_t* h, int64_t n_pos, int d_lat, const float* w0, const float* w1,
                     const uint16_t* kraw, int d_idx,
                     uint8_t* lat_codes, uint8_t* lat_scales, uint8_t* ikey_codes, uint8_t* ikey_scales) {
    int64_t n = n_pos / 2;
    float* e = (float*)malloc(sizeof(float) * n * d_lat);
    orc_merge_pairs(h, n, d_lat, w0, w1, e);
    orc_quantize_rows(e, n, d_lat, lat_codes, lat_scales);
    free(e);
    float* k = (float*)malloc(sizeof(float) * n * d_idx);
    for (int64_t i = 0; i < n * d_idx; ++i) k[i] = bf16_value(kraw[i]);
    orc_quantize_rows(k, n, d_idx, ikey_codes, ikey_scales);
    free(k);
}

/* Decoder cache (compression ratio 1, [P1] §1.1 and §2.3.3: one global entry
 * per position, kept for addressability): entry i is raw position i, its bf16
 * hidden state quantised as it is. */
void orc_cache_write_r1(const uint16_t* h, int64_t n_pos, int d_lat, uint8_t* lat_codes, uint8_t* lat_scales) {
    float* e = (float*)malloc(sizeof(float) * n_pos * d_lat);
    for (int64_t i = 0; i < n_pos * d_lat; ++i) e[i] = bf16_value(h[i]);
    orc_quantize_rows(e, n_pos, d_lat, lat_codes, lat_scales);
    free(e);
}

/* Indexer keys projected from the main KV entry ([P1] §2.3.1: the indexer K is
 * a projection of the main KV, which replaces CSA's separate path):
 *     k[d] = sum_c W[d][c] * L[c]
 * over the stored entry L (dequantised FP4 latent) and the projection W, itself
 * stored in the same FP4 format (E2M1, one E4M3 scale per 16 inputs).  Every
 * product is exact in fp64 and a multiple of 2^-20, and every partial sum stays
 * below 2^52 in magnitude, so the fp64 sum below is the exact value; it is
 * rounded once to fp32 and quantised with the cache's codec. */
void orc_project_ikeys(const uint8_t* lat_codes, const uint8_t* lat_scales, int64_t n, int d_lat,
                       const uint8_t* w_codes, const uint8_t* w_scales, int d_idx,
                       uint8_t* ikey_codes, uint8_t* ikey_scales) {
    double* W = (double*)malloc(sizeof(double) * d_idx * d_lat);
    orc_dequant_rows(w_codes, w_scales, d_idx, d_lat, W);
    float* k = (float*)malloc(sizeof(float) * n * d_idx);
    #pragma omp parallel
    {
        double* L = (double*)malloc(sizeof(double) * d_lat);
        #pragma omp for schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            orc_dequant_rows(lat_codes + i * (d_lat / 2), lat_scales + i * (d_lat / 16), 1, d_lat, L);
            for (int d = 0; d < d_idx; ++d) {
                double acc = 0.0;
                for (int c = 0; c < d_lat; ++c) acc += W[(int64_t)d * d_lat + c] * L[c];
                k[i * d_idx + d] = (float)acc;
            }
        }
        free(L);
    }
    orc_quantize_rows(k, n, d_idx, ikey_codes, ikey_scales);
    free(k);
    free(W);
}

/* ------------------------------------------------------------------------ */
/* indexer: score_j = sum_h w_h * ReLU(q_h . k_j)                            */
/* [P1] §2.3.1: indexer Q and indexer K score the main-KV entries and the    */
/* top-k entries of each query are selected.  q and k are the dequantised    */
/* FP4 values; their dot product is exact in fp64 (all products are integer  */
/* multiples of 2^-20 and every partial sum stays below 2^33).  The head sum */
/* is the fp64 chain S = fma(w_h, r_h, S) for h = 0, 1, ..., H-1.           */
/* ------------------------------------------------------------------------ */

/* scores of the entries ids[0..n) (ids == NULL: entries 0..n-1); entries whose
 * id is negative get -inf. */
void orc_index_scores(const uint8_t* kcodes, const uint8_t* kscales, int d, const int32_t* ids, int64_t n,
                      const uint8_t* qcodes, const uint8_t* qscales, const float* w, int H, double* S) {
    double* qh = (double*)malloc(sizeof(double) * H * d);
    orc_dequant_rows(qcodes, qscales, H, d, qh);
    #pragma omp parallel
    {
        double* kh = (double*)malloc(sizeof(double) * d);
        #pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            int64_t j = ids ? ids[t] : t;
            if (j < 0) { S[t] = -INFINITY; continue; }
            orc_dequant_rows(kcodes + j * (d / 2), kscales + j * (d / 16), 1, d, kh);
            double acc = 0.0;
            for (int hh = 0; hh < H; ++hh) {
                double dot = 0.0;
                for (int i = 0; i < d; ++i) dot += qh[hh * d + i] * kh[i];
                double r = dot > 0.0 ? dot : 0.0;
                acc = fma((double)w[hh], r, acc);
            }
            S[t] = acc;
        }
        free(kh);
    }
    free(qh);
}

typedef struct { double s; int32_t id; } scored;

/* rank: larger score first, then smaller id */
static int by_score_desc_id_asc(const void* a, const void* b) {
    const scored* x = (const scored*)a;
    const scored* y = (const scored*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->id < y->id) ? -1 : (x->id > y->id);
}

static int by_id_asc(const void* a, const void* b) {
    const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Top-k: the k best entries by a full sort of (score desc, id asc); entries
 * with negative id are not candidates.  The selection is a set of positions:
 * it is written in ascending entry order (as the pages print the read
 * positions of their toy example), missing slots -1 at the end. */
void orc_topk(const double* S, const int32_t* ids, int64_t n, int k, int32_t* out) {
    scored* v = (scored*)malloc(sizeof(scored) * (n > 0 ? n : 1));
    int64_t m = 0;
    for (int64_t t = 0; t < n; ++t) {
        int32_t id = ids ? ids[t] : (int32_t)t;
        if (id < 0) continue;
        v[m].s = S[t];
        v[m].id = id;
        ++m;
    }
    qsort(v, (size_t)m, sizeof(scored), by_score_desc_id_asc);
    int64_t kept = m < k ? m : k;
    for (int64_t i = 0; i < kept; ++i) out[i] = v[i].id;
    qsort(out, (size_t)kept, sizeof(int32_t), by_id_asc);
    for (int64_t i = kept; i < k; ++i) out[i] = -1;
    free(v);
}

/* HSI candidate pool ([P1] §2.3.4).  The eligible scores (width n_elig) are cut
 * into blocks of bs entries, the tail block padded with -inf; each block keeps
 * its maximum; the block that holds the newest eligible entry (n_elig-1) is
 * set to +inf so that it always takes one of the slots; the n_sel best blocks
 * (max desc, block asc) are kept and every eligible entry of a kept block goes
 * into the pool, in ascending order.  Unused pool slots are -1. */
void orc_hsi_pool(const double* S, int64_t n_elig, int bs, int n_sel, int32_t* pool) {
    int64_t nb = (n_elig + bs - 1) / bs;
    scored* blk = (scored*)malloc(sizeof(scored) * (nb > 0 ? nb : 1));
    for (int64_t b = 0; b < nb; ++b) {
        double mx = -INFINITY;
        for (int i = 0; i < bs; ++i) {
            int64_t j = b * bs + i;
            double v = (j < n_elig) ? S[j] : -INFINITY;
            if (v > mx) mx = v;
        }
        blk[b].s = mx;
        blk[b].id = (int32_t)b;
    }
    if (nb > 0) blk[(n_elig - 1) / bs].s = INFINITY;
    qsort(blk, (size_t)nb, sizeof(scored), by_score_desc_id_asc);
    int64_t keep = nb < n_sel ? nb : n_sel;
    unsigned char* mark = (unsigned char*)calloc((size_t)(nb > 0 ? nb : 1), 1);
    for (int64_t t = 0; t < keep; ++t) mark[blk[t].id] = 1;
    int64_t w = 0;
    for (int64_t b = 0; b < nb; ++b)
        if (mark[b])
            for (int i = 0; i < bs; ++i) {
                int64_t j = b * bs + i;
                if (j < n_elig) pool[w++] = (int32_t)j;
            }
    for (; w < (int64_t)n_sel * bs; ++w) pool[w] = -1;
    free(mark);
    free(blk);
}

/* ------------------------------------------------------------------------ */
/* attention over the selected entries plus the window                       */
/* [P1] §2.3.1: each Q attends to its top-k entries and to the local window  */
/* KV; §1.1: every head reads one shared 512-dim latent (MQA).  [P3]: scores */
/* Q·K become weights summing to 1 (softmax), output = weighted sum of V.    */
/* With one latent L_j serving as key and value: s_hj = scale * (q_h . L_j), */
/* p_h = softmax over J of s_h, o_h = sum_j p_hj L_j.                        */
/* ------------------------------------------------------------------------ */

static void attend_rows(const uint16_t* q, int H, int d, const double* keys, int64_t n_keys, double scale,
                        double* out, double* lse) {
    double* s = (double*)malloc(sizeof(double) * (n_keys > 0 ? n_keys : 1));
    for (int hh = 0; hh < H; ++hh) {
        double qd[1024];
        for (int i = 0; i < d; ++i) qd[i] = (double)bf16_value(q[hh * d + i]);
        double mx = -INFINITY;
        for (int64_t j = 0; j < n_keys; ++j) {
            double dot = 0.0;
            for (int i = 0; i < d; ++i) dot += qd[i] * keys[j * d + i];
            s[j] = dot * scale;
            if (s[j] > mx) mx = s[j];
        }
        double sum = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) {
            s[j] = exp(s[j] - mx);
            sum += s[j];
        }
        for (int i = 0; i < d; ++i) out[hh * d + i] = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) {
            double p = s[j] / sum;
            for (int i = 0; i < d; ++i) out[hh * d + i] += p * keys[j * d + i];
        }
        if (lse) lse[hh] = mx + log(sum);
    }
    free(s);
}

/* Sparse attention of one query.  Keys: the entries idx[0..k) that are >= 0
 * (dequantised latent rows of this sequence) followed by the window rows
 * win[0..n_win) (bf16). */
void orc_sparse_attention(const uint16_t* q, int H, int d, const int32_t* idx, int k,
                          const uint8_t* lat_codes, const uint8_t* lat_scales,
                          const uint16_t* win, int64_t n_win, double scale, double* out, double* lse) {
    int64_t n_sel = 0;
    for (int i = 0; i < k; ++i) n_sel += idx[i] >= 0;
    int64_t n_keys = n_sel + n_win;
    double* keys = (double*)malloc(sizeof(double) * (n_keys > 0 ? n_keys : 1) * d);
    int64_t r = 0;
    for (int i = 0; i < k; ++i)
        if (idx[i] >= 0) {
            orc_dequant_rows(lat_codes + (int64_t)idx[i] * (d / 2), lat_scales + (int64_t)idx[i] * (d / 16), 1, d,
                             keys + r * d);
            ++r;
        }
    for (int64_t j = 0; j < n_win; ++j, ++r)
        for (int i = 0; i < d; ++i) keys[r * d + i] = (double)bf16_value(win[j * d + i]);
    attend_rows(q, H, d, keys, n_keys, scale, out, lse);
    free(keys);
}

/* Textbook dense attention of one query over every eligible entry 0..n_elig-1
 * and every window row: written separately from the sparse path (its own
 * loops, no index list) so that "sparse with k >= n_elig equals dense" checks
 * the sparse path against something other than itself. */
void orc_dense_attention(const uint16_t* q, int H, int d, int64_t n_elig,
                         const uint8_t* lat_codes, const uint8_t* lat_scales,
                         const uint16_t* win, int64_t n_win, double scale, double* out, double* lse) {
    for (int hh = 0; hh < H; ++hh) {
        double num[1024];
        for (int i = 0; i < d; ++i) num[i] = 0.0;
        /* two passes: max, then exp-weighted sums */
        double mx = -INFINITY;
        for (int64_t j = 0; j < n_elig + n_win; ++j) {
            double dot = 0.0;
            for (int i = 0; i < d; ++i) {
                double kv;
                if (j < n_elig) {
                    uint8_t byte = lat_codes[j * (d / 2) + i / 2];
                    kv = orc_e2m1_value((i & 1) ? byte >> 4 : byte & 15) * orc_e4m3_value(lat_scales[j * (d / 16) + i / 16]);
                } else {
                    kv = (double)bf16_value(win[(j - n_elig) * d + i]);
                }
                dot += (double)bf16_value(q[hh * d + i]) * kv;
            }
            double s = dot * scale;
            if (s > mx) mx = s;
        }
        double den = 0.0;
        for (int64_t j = 0; j < n_elig + n_win; ++j) {
            double dot = 0.0;
            double kv[1024];
            for (int i = 0; i < d; ++i) {
                if (j < n_elig) {
                    uint8_t byte = lat_codes[j * (d / 2) + i / 2];
                    kv[i] = orc_e2m1_value((i & 1) ? byte >> 4 : byte & 15) * orc_e4m3_value(lat_scales[j * (d / 16) + i / 16]);
                } else {
                    kv[i] = (double)bf16_value(win[(j - n_elig) * d + i]);
                }
                dot += (double)bf16_value(q[hh * d + i]) * kv[i];
            }
            double wgt = exp(dot * scale - mx);
            den += wgt;
            for (int i = 0; i < d; ++i) num[i] += wgt * kv[i];
        }
        for (int i = 0; i < d; ++i) out[hh * d + i] = num[i] / den;
        if (lse) lse[hh] = mx + log(den);
    }
}

/*
 * libcsa2 — CSA2 sparse-attention decode over an FP4 global KV cache, for
 * NVIDIA GB300 (sm_103a).  C ABI.
 *
 * What the library computes is described in "DeepSeek-v4.1 Flash:
 * KVキャッシュ圧縮の限界を押し広げる" (hackernews.jp), §1.1 and §2.3 (CSA2), in the
 * spec table of the ai.freelance-job.com summary of the same report, and in
 * "DeepSeek V4.1 Flash architecture: making a giant AI faster through reuse"
 * (yasmorita.com), CSA2 and storage sections.  The pages fix neither a number
 * format nor a score formula; this library uses:
 *   - FP4 = E2M1 codes, two per byte (element 2i in the low nibble), with one
 *     E4M3 scale byte per 16 consecutive values, scale = E4M3_rn_satfinite(
 *     amax/6), code = round-to-nearest-even of x/scale (zero written as +0);
 *   - indexer score_j = sum_h w_h * ReLU(q_h . k_j) over dequantised FP4 q and
 *     k, q.k exact, the head sum an fp64 fused multiply-add chain in ascending h;
 *     ranking by (score desc, entry index asc);
 *   - a query at raw position p sees global entries i < n_elig(p) =
 *     floor((p-127)/ratio) (entries lying wholly before its window; ratio 2
 *     for an encoder copy, 1 for the decoder's) and the window rows of raw
 *     positions max(0, p-127) .. p.
 *
 * Conventions (all entry points):
 *   - Every array argument is DEVICE memory allocated and owned by the caller;
 *     the library allocates nothing, frees nothing and never synchronises.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued on it; results are valid once the stream reaches them.
 *   - Arguments are validated on the host before anything is enqueued; a bad
 *     argument returns CSA2_ERR_INVALID_ARG and enqueues nothing.  A launch
 *     failure returns CSA2_ERR_CUDA (cudaGetLastError after the launch).
 *   - Index value -1 marks an empty slot in every index list.
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - Threading: calls are re-entrant; calls on one stream run in order.
 *   - Kernels are launched with programmatic stream serialisation: a kernel of
 *     this library may be scheduled while the kernel just before it in the
 *     stream still runs, and waits for that kernel's completion before it
 *     reads what the stream produced; it lets its own successor start only
 *     after that wait, so it never overlaps any earlier work.  Before the wait
 *     the attention reads only caller inputs that no kernel of this library
 *     writes (the queries q and their positions q_pos, the window rows swa); a
 *     caller that writes those with a kernel of its own that itself lets its
 *     successor start early must make that kernel complete first.  Kernels not
 *     launched this way (any caller kernel by default) are waited for as usual.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CSA2_OK = 0,
    CSA2_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or mode; nothing enqueued */
    CSA2_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d_lat != 512) */
    CSA2_ERR_CUDA = 3,          /* a CUDA call or launch failed */
    CSA2_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than csa2_workspace_size() */
    CSA2_ERR_TIMEOUT = 5        /* a kernel gave up on a bounded wait (reported by csa2_poll_error) */
} csa2_status;

/* cross-layer modes, "DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる" §2.3.2 */
enum { CSA2_FULL = 0, CSA2_REINDEX = 1, CSA2_REUSE = 2 };

/* operations that take a workspace */
enum { CSA2_OP_INDEXER_TOPK = 1, CSA2_OP_REINDEX = 2, CSA2_OP_SPARSE_ATTN = 3 };

/*
 * The global KV cache shared by the layers of one block ("DeepSeek-v4.1 Flash"
 * §1.1: main KV and indexer keys shared across layers, FP4).  Four dense
 * planes, sequence-major, entry i of sequence b at row b*capacity + i:
 *   lat_codes   [batch][capacity][d_lat/2]   E2M1 codes of the 512-dim latent
 *   lat_scales  [batch][capacity][d_lat/16]  E4M3 scales of the latent
 *   ikey_codes  [batch][capacity][d_idx/2]   E2M1 codes of the indexer key
 *   ikey_scales [batch][capacity][d_idx/16]  E4M3 scales of the indexer key
 * ratio is the number of raw positions per entry: 2 for an encoder copy
 * (entry i merges raw positions 2i and 2i+1, §1.1), 1 for the decoder's copy
 * (entry i is raw position i, kept per position for addressability, §2.3.3);
 * a query at raw position p may read entries i < n_elig(p) = floor((p-127) /
 * ratio), those lying wholly before its window.
 * lat_codes, lat_scales and ikey_codes must be 16-byte aligned, ikey_scales
 * d_idx/16-byte aligned (so a batch-1 view of one sequence of a larger cache
 * is always valid).  d_lat must be 512; d_idx must be 64 or 128; ratio 1 or 2.
 * With ikey_codes 32-byte aligned (as any cudaMalloc'd plane is), the decode
 * Full scan reads the keys by tensor copy; otherwise it takes a CUDA-core scan
 * with the same results.
 */
typedef struct {
    uint8_t* lat_codes;
    uint8_t* lat_scales;
    uint8_t* ikey_codes;
    uint8_t* ikey_scales;
    int32_t batch;
    int32_t capacity;
    int32_t d_lat;
    int32_t d_idx;
    int32_t ratio;
} csa2_cache;

/*
 * Cache write: the encoder's 2:1 channel-wise merge fused with FP4
 * quantisation ("DeepSeek-v4.1 Flash" §1.1 sequence dimension; §2.3.1: the
 * CSA2 compressor merges without overlap and without absolute position
 * embedding).  For a ratio-2 cache, every sequence b and entry i in
 * [pos0/2, pos0/2 + n_pos/2):
 *     e[c] = fmaf(w1[c], h[2i+1][c], float(w0[c] * h[2i][c]))   (fp32)
 * quantised to FP4 into lat_codes / lat_scales; for a ratio-1 cache (the
 * decoder's, §2.3.3) entry i is raw position i, h[i] quantised as it is (w0 and
 * w1 are not read and may be NULL).  If ikey_raw is not NULL its rows (one per
 * entry) are quantised into ikey_codes / ikey_scales.
 *   h        bf16 [batch][n_pos][d_lat], raw positions pos0 .. pos0+n_pos-1
 *   w0, w1   fp32 [d_lat]
 *   ikey_raw bf16 [batch][n_pos/ratio][d_idx] or NULL
 * Ratio 2: pos0 and n_pos even.  pos0/ratio + n_pos/ratio <= capacity.  Inputs
 * must be finite.
 */
csa2_status csa2_cache_write(const csa2_cache* cache, const uint16_t* h, int64_t pos0, int32_t n_pos,
                             const float* w0, const float* w1, const uint16_t* ikey_raw, void* stream);

/*
 * Cache write with the indexer keys projected from the entries ("DeepSeek-v4.1
 * Flash" §2.3.1: the indexer K is a projection of the main KV entry, which
 * replaces CSA's separate compression path): the latent as csa2_cache_write
 * writes it, and for every entry
 *     k[d] = sum_c W[d][c] * L[c],   d < d_idx
 * over the stored entry L (the dequantised FP4 latent just written) and the
 * projection W, given in the same FP4 format; the exact sum is rounded once to
 * fp32 and quantised into ikey_codes / ikey_scales with the cache's codec.  One
 * kernel does both per entry.
 *   wik_codes  uint8 [d_idx][d_lat/2] E2M1 codes of W (16-byte aligned)
 *   wik_scales uint8 [d_idx][d_lat/16] E4M3 scales of W (4-byte aligned)
 * Other arguments and conditions as csa2_cache_write (ikey_raw not taken).
 */
csa2_status csa2_cache_write_projected(const csa2_cache* cache, const uint16_t* h, int64_t pos0, int32_t n_pos,
                                       const float* w0, const float* w1, const uint8_t* wik_codes,
                                       const uint8_t* wik_scales, void* stream);

/*
 * FP4 quantisation of fp32 rows (the same codec as the cache): used for the
 * indexer queries, which the indexer takes in FP4 ("DeepSeek-v4.1 Flash"
 * TL;DR: FP4 KV cache; the indexer is optimised together with it).
 *   x      fp32 [n_rows][d], d a multiple of 16
 *   codes  uint8 [n_rows][d/2], scales uint8 [n_rows][d/16]
 */
csa2_status csa2_quantize_fp4(const float* x, int64_t n_rows, int32_t d, uint8_t* codes, uint8_t* scales,
                              void* stream);

/*
 * Full-mode indexer: scores every eligible entry and keeps the top k
 * ("DeepSeek-v4.1 Flash" §2.3.1 lightweight indexer, §2.3.2 Full mode), and
 * optionally the HSI candidate pool (§2.3.4): per-block maxima of the same
 * scores over blocks of pool_block_size entries (tail block padded with
 * -inf), the block holding entry n_elig-1 forced to +inf, the best
 * pool_blocks blocks (ties to the lower block), expanded to their eligible
 * entries in ascending order.
 *   iq_codes  uint8 [batch][n_q][n_heads][d_idx/2]   FP4 indexer queries (16-byte aligned)
 *   iq_scales uint8 [batch][n_q][n_heads][d_idx/16]
 *   w_head    fp32  [batch][n_q][n_heads]
 *   q_pos     int64 [batch][n_q]  raw position of each query (device memory);
 *             n_elig is clamped to capacity
 *   idx_out   int32 [batch][n_q][k]  the chosen entry ids in ascending order, -1 padded
 *   pool_out  int32 [batch][n_q][pool_blocks*pool_block_size] or NULL when
 *             pool_blocks == 0; -1 padded
 * pool_block_size == 0 asks for the other reading of the candidate pool: the
 * pool_blocks best entries by the same score and order as the top k (no block
 * structure, nothing forced in), ascending, -1 padded; pool_out then has
 * pool_blocks slots per query.
 * 1 <= k <= 2048; 1 <= n_heads <= 32; pool_blocks <= 2048;
 * pool_blocks*pool_block_size <= 16384.
 * workspace: csa2_workspace_size(CSA2_OP_INDEXER_TOPK, ...) bytes.
 */
csa2_status csa2_indexer_topk(const csa2_cache* cache, const uint8_t* iq_codes, const uint8_t* iq_scales,
                              const float* w_head, int32_t n_q, const int64_t* q_pos, int32_t n_heads, int32_t k,
                              int32_t* idx_out, int32_t pool_blocks, int32_t pool_block_size, int32_t* pool_out,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * Reindex / Reuse ("DeepSeek-v4.1 Flash" §2.3.2 and §2.3.4).
 *   mode CSA2_REINDEX: score only the pool entries with this layer's indexer
 *     queries and keep the top k inside the pool (ascending entry order, -1 padded);
 *     pool int32 [batch][n_q][pool_len] (-1 slots ignored, entries distinct as
 *     in an HSI pool), pool_len <= 16384.
 *   mode CSA2_REUSE: idx_out = prev_idx, bit for bit (a device copy); the
 *     indexer arguments and the pool may be NULL.
 *   prev_idx, idx_out int32 [batch][n_q][k].
 * workspace: csa2_workspace_size(CSA2_OP_REINDEX, ...) bytes (may be 0 for REUSE).
 */
csa2_status csa2_reindex(int32_t mode, const csa2_cache* cache, const uint8_t* iq_codes, const uint8_t* iq_scales,
                         const float* w_head, int32_t n_q, int32_t n_heads, const int32_t* pool, int32_t pool_len,
                         const int32_t* prev_idx, int32_t k, int32_t* idx_out, void* workspace, size_t ws_bytes,
                         void* stream);

/*
 * Reindex from unquantised indexer queries: the same results as
 * csa2_quantize_fp4(iq -> codes, scales) followed by csa2_reindex(CSA2_REINDEX,
 * codes, scales, ...), bit for bit, with the FP4 quantisation of the queries
 * done by the Reindex kernels as they stage each query, so a Reindex layer
 * takes one launch fewer.  The pages have no separate counterpart: it is the
 * Reindex step with its query quantisation fused.
 *   iq fp32 [batch][n_q][n_heads][d_idx], 16-byte aligned; the other arguments
 *   as for csa2_reindex(CSA2_REINDEX, ...), same workspace size.
 */
csa2_status csa2_reindex_f32(const csa2_cache* cache, const float* iq, const float* w_head, int32_t n_q,
                             int32_t n_heads, const int32_t* pool, int32_t pool_len, int32_t k, int32_t* idx_out,
                             void* workspace, size_t ws_bytes, void* stream);

/*
 * Sparse attention over the selected entries plus the sliding window
 * ("DeepSeek-v4.1 Flash" §2.3.1: each query attends to its top-k entries and
 * to the local SWA window; §1.1: all heads share one 512-dim latent, which is
 * both key and value).  Per query and head h:
 *     s_j = scale * (q_h . L_j) for j in J = {idx >= 0} U window
 *     o_h = sum_j softmax_J(s)_j L_j,   lse_h = log sum_j exp(s_j)
 * L_j is the dequantised FP4 latent of entry j, or the bf16 window row.
 *   q     bf16 [batch][n_q][n_heads][d_lat]
 *   q_pos int64 [batch][n_q] raw positions (device)
 *   idx   int32 [batch][n_q][k]
 *   swa   bf16 [batch][swa_len][d_lat], row r = raw position swa_pos0 + r; the
 *         window of a query is clipped to the rows present
 *   out   fp32 [batch][n_q][n_heads][d_lat]
 *   lse   fp32 [batch][n_q][n_heads] or NULL
 * 1 <= n_heads <= 128, k <= 2048.  q, swa and out 16-byte aligned, q_pos 8, idx
 * and lse 4 (CSA2_ERR_INVALID_ARG otherwise).
 * workspace: csa2_workspace_size(CSA2_OP_SPARSE_ATTN, ...) bytes (may be 0).
 */
csa2_status csa2_sparse_attn(const csa2_cache* cache, const uint16_t* q, int32_t n_q, int32_t n_heads,
                             const int64_t* q_pos, const int32_t* idx, int32_t k, const uint16_t* swa,
                             int64_t swa_pos0, int32_t swa_len, float scale, float* out, float* lse,
                             void* workspace, size_t ws_bytes, void* stream);

/*
 * Reindex without a workspace, for callers that cannot allocate device memory:
 * for instance a plug-in inside a host application that owns and budgets all
 * device memory, or a real-time decode loop that must not hit the implicit
 * device-wide synchronisation of cudaMalloc / cudaFree.  The pages have no
 * counterpart of this entry point; it is a deployment convenience.
 *
 * Same arguments, checks and results as csa2_reindex(CSA2_REINDEX, ...) minus
 * the workspace (and minus prev_idx, which only Reuse reads).  The scratch is a
 * fixed 8 MiB array inside the library's device image: every GPU that loads
 * the library holds those 8 MiB until the process exits.  Requests needing
 * more (batch * n_q * pool_len above about 233,000 pool slots) return
 * CSA2_ERR_WORKSPACE and enqueue nothing.  The call allocates and frees
 * nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: do not use this entry point across cudaDeviceReset.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents.  No part of it needs to start at zero.  Calls that can
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on it: order them, or give one of them a workspace via csa2_reindex.
 */
csa2_status csa2_reindex_noalloc(const csa2_cache* cache, const uint8_t* iq_codes, const uint8_t* iq_scales,
                                 const float* w_head, int32_t n_q, int32_t n_heads, const int32_t* pool,
                                 int32_t pool_len, int32_t k, int32_t* idx_out, void* stream);

/*
 * Failure detection.  Every wait of the library's kernels on an asynchronous
 * event (a copy landing, a tensor-core operation completing, the other CTA of
 * a pair) is bounded: after about 2^24 polls it gives up, the kernel records
 * the failure in the first 32-bit word of the workspace it was given and
 * returns with its outputs unspecified (the attention writes NaN), so the
 * context stays usable.  No call reports this itself, since calls are
 * asynchronous.
 *
 * csa2_poll_error reads that word of `workspace` (a workspace given to any
 * operation, at least 16 bytes), clears it, and returns CSA2_ERR_TIMEOUT if it
 * was set, CSA2_OK otherwise.  The library never clears the word otherwise:
 * zero the first 16 bytes of a new workspace (or poll it once) before relying
 * on it.  It synchronises `stream` (it waits for the work
 * enqueued on it), so call it between steps, never during stream capture.
 * Returns CSA2_ERR_INVALID_ARG for a NULL or too small workspace,
 * CSA2_ERR_CUDA if the copy fails.
 */
csa2_status csa2_poll_error(void* workspace, size_t ws_bytes, void* stream);

/*
 * Self-test of the bounded waits: one kernel waits, with at most `max_polls`
 * polls, on a barrier that nothing ever signals, gives up, and records the
 * failure in `workspace` exactly as the library's kernels do; a following
 * csa2_poll_error returns CSA2_ERR_TIMEOUT.  It exercises the waiting helper,
 * the error word and the poll without a fault or a hang.  max_polls >= 1;
 * workspace at least 16 bytes.
 */
csa2_status csa2_selftest_wait_timeout(uint32_t max_polls, void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes an operation needs (0 if none).  capacity = entries per
 * sequence of the cache; for CSA2_OP_REINDEX pass pool_len as `capacity`. */
size_t csa2_workspace_size(int32_t op, int32_t batch, int32_t n_q, int32_t n_heads, int32_t k, int64_t capacity);

/* Static string for a status code. */
const char* csa2_status_string(csa2_status s);

/* Number of kernel launches this library has enqueued in this process so far
 * (all devices, all streams; a launch recorded into a CUDA graph counts once,
 * when it is recorded).  Instrumentation for benchmarks; never fails. */
int64_t csa2_launch_count(void);

/* ABI version of this header (major * 100 + minor). */
int32_t csa2_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H */

"""CUDA path vs the fp64 oracle, through the C ABI.

Bar: cache bytes, FP4 codes, scales, top-k index lists and HSI pools
bit-exact; attention outputs within a max relative error of 2e-3 per
(sequence, query, head) row: max_i |o_i - o*_i| / max_i |o*_i|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.workloads import WORKLOADS, scaled

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_decode_gb300 as m
    from compressed_sparse_attention_decode_gb300 import build as b
    b.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def bf16_t(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def rel_err_rows(out, ref):
    num = np.abs(out.astype(np.float64) - ref).max(-1)
    den = np.abs(ref).max(-1)
    return float((num / den).max())


def host_cache(csa, planes, d_idx):
    """upload host cache planes (numpy [B, n, ...]) into a Cache"""
    lc, ls, kc, ks = planes
    c = csa.Cache(lc.shape[0], lc.shape[1], d_idx)
    for t, a in zip((c.lat_codes, c.lat_scales, c.ikey_codes, c.ikey_scales), planes):
        t.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return c


# ---------------------------------------------------------------- cache write / codec

def wide_range_rows(seed, rows, d):
    """normal values times 2^e, e drawn per 16-group over [-40, 14]: E4M3
    scales from subnormal to saturated, plus exact midpoints and zero groups"""
    x = synth.normal_f32(seed, 1, (rows, d)).astype(np.float64)
    e = np.floor(synth.uniform_f32(seed, 2, (rows, d // 16), -40, 14)).astype(np.float64)
    x = x * np.repeat(2.0 ** e, 16, axis=1)
    x[0, :16] = 0.0
    s = 2.0 ** -3
    x[1, :16] = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5, 5.5]) * s
    return x


def test_quantize_fp4_bit_exact(csa):
    x = wide_range_rows(31, 512, 128).astype(np.float32)
    codes, scales = csa.csa2_quantize_fp4(torch.from_numpy(x).cuda())
    rc, rs = oracle.quantize_rows(x)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("d_idx", [64, 128])
def test_cache_write_bit_exact_wide_range(csa, d_idx):
    B, n_pos = 2, 256
    h = wide_range_rows(32, B * n_pos, 512)
    # round to bf16 (RNE) on the host
    u = h.astype(np.float32).view(np.uint32).astype(np.uint64)
    hb = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16).reshape(B, n_pos, 512)
    kr = wide_range_rows(33, B * n_pos // 2, d_idx).astype(np.float32).view(np.uint32).astype(np.uint64)
    kb = ((kr + 0x7FFF + ((kr >> 16) & 1)) >> 16).astype(np.uint16).reshape(B, n_pos // 2, d_idx)
    w0 = synth.uniform_f32(33, 3, (512,), 0.3, 0.7)
    w1 = synth.uniform_f32(33, 4, (512,), 0.3, 0.7)
    cache = csa.Cache(B, n_pos // 2 + 10, d_idx)
    csa.csa2_cache_write(cache, bf16_t(hb[:, :128]), 0, torch.from_numpy(w0).cuda(), torch.from_numpy(w1).cuda(),
                         bf16_t(kb[:, :64]))
    csa.csa2_cache_write(cache, bf16_t(hb[:, 128:]), 128, torch.from_numpy(w0).cuda(), torch.from_numpy(w1).cuda(),
                         bf16_t(kb[:, 64:]))
    for b in range(B):
        lc, ls, kc, ks = oracle.cache_write(hb[b], w0, w1, kb[b])
        n = n_pos // 2
        assert np.array_equal(cache.lat_codes[b, :n].cpu().numpy(), lc)
        assert np.array_equal(cache.lat_scales[b, :n].cpu().numpy(), ls)
        assert np.array_equal(cache.ikey_codes[b, :n].cpu().numpy(), kc)
        assert np.array_equal(cache.ikey_scales[b, :n].cpu().numpy(), ks)
        assert not cache.lat_codes[b, n:].any()          # untouched rows stay zero


# ---------------------------------------------------------------- whole walks on small workloads

def check_walk(csa, wl, seqs, queries=None, layers=None):
    from compressed_sparse_attention_decode_gb300.synthetic import build_step
    step = build_step(wl, want_lse=True)
    step.enqueue()
    torch.cuda.synchronize()
    for bi, b in enumerate(seqs):
        lc, ls, kc, ks = (p.cpu().numpy()[bi] for p in (step.cache.lat_codes, step.cache.lat_scales,
                                                          step.cache.ikey_codes, step.cache.ikey_scales))
        ref_cache = oracle.sequence_cache(wl, b)
        for got, want in zip((lc, ls, kc, ks), ref_cache):
            assert np.array_equal(got, want)
        ref = oracle.run_sequence(wl, b, cache=ref_cache, queries=queries, layers=layers)
        qs = list(range(wl.n_q)) if queries is None else list(queries)
        for l in ref["idx"]:
            got = step.layer_idx(l)[bi].cpu().numpy()[qs]
            assert np.array_equal(got, ref["idx"][l]), (wl.name, b, l)
        for l in ref["pool"]:
            assert np.array_equal(step.pool[bi].cpu().numpy()[qs], ref["pool"][l]), (wl.name, b, l)
        for l in ref["out"]:
            got = step.out[l, bi].cpu().numpy()[qs]
            err = rel_err_rows(got, ref["out"][l])
            assert err <= ATTN_TOL, (wl.name, b, l, err)
            lse = step.lse[l, bi].cpu().numpy()[qs]
            assert np.abs(lse - ref["lse"][l]).max() <= 1e-4 * max(1.0, np.abs(ref["lse"][l]).max())
    return step


@pytest.mark.parametrize("ratio,d_idx", [(1, 128), (1, 64), (2, 128)])
def test_projected_cache_write_bit_exact(csa, ratio, d_idx):
    """indexer keys projected from the stored entries (FP4 W times the FP4 entry,
    exact sum, then the FP4 codec) in the same launch as the entry write: every byte
    of all four planes against the oracle; two writes (a prefix, then a ragged tail
    at a nonzero position) so that the position offset is exercised"""
    wl = scaled(WORKLOADS[2], B=1, T=2 * 1000 + 2 * 37, d_I=d_idx, ratio=ratio, ikey_proj=True)
    cache = csa.Cache(1, wl.n_entries, d_idx, ratio=ratio)
    w0, w1 = (torch.from_numpy(w).cuda() for w in wl.merge_weights())
    wc, ws = csa.csa2_quantize_fp4(torch.from_numpy(wl.w_ik()).cuda())
    h = bf16_t(wl.h(0, 0, wl.T))[None]
    csa.csa2_cache_write_projected(cache, h[:, :2000].contiguous(), 0, w0, w1, wc, ws)
    csa.csa2_cache_write_projected(cache, h[:, 2000:].contiguous(), 2000, w0, w1, wc, ws)
    torch.cuda.synchronize()
    want = oracle.sequence_cache(wl, 0)
    got = (cache.lat_codes, cache.lat_scales, cache.ikey_codes, cache.ikey_scales)
    for name, g, w in zip(("lat_codes", "lat_scales", "ikey_codes", "ikey_scales"), got, want):
        assert np.array_equal(g[0].cpu().numpy(), w), name
    # W is the library's own quantisation of the same rows
    wc_ref, ws_ref = oracle.quantize_rows(wl.w_ik())
    assert np.array_equal(wc.cpu().numpy(), wc_ref) and np.array_equal(ws.cpu().numpy(), ws_ref)


def test_ratio_mismatch_is_rejected(csa):
    """a ratio-1 cache write whose raw rows do not cover whole entries of the
    cache's ratio, or a ratio outside {1, 2}, is refused before any launch"""
    cache = csa.Cache(1, 64, 128, ratio=3)
    h = torch.zeros((1, 8, 512), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(512, dtype=torch.float32, device="cuda")
    kr = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        csa.csa2_cache_write(cache, h, 0, w, w, kr)
    cache2 = csa.Cache(1, 64, 128, ratio=2)
    with pytest.raises(RuntimeError):
        csa.csa2_cache_write(cache2, h[:, :7].contiguous(), 0, w, w, kr)
    torch.cuda.synchronize()


def test_decoder_ratio1_projected_schedule(csa):
    """the decoder's cache (one entry per raw position, indexer keys projected):
    Full (+HSI pool) -> Reuse x3 -> Reindex -> Reuse x3, every index and output"""
    wl = scaled(WORKLOADS[2], B=2, T=9000 + 77, ratio=1, ikey_proj=True, pool_blocks=256,
                layers=("full", "reuse", "reuse", "reuse", "reindex", "reuse", "reuse", "reuse"))
    check_walk(csa, wl, [0, 1])


def test_decoder_ratio1_short_contexts(csa):
    """ratio 1 near the start of a sequence: fewer eligible entries than k,
    none at all, exactly k"""
    for T in (100, 128, 129, 200, 128 + 64):
        wl = scaled(WORKLOADS[2], B=1, T=T, k=64, H=16, ratio=1, ikey_proj=True, layers=("full", "reuse"))
        check_walk(csa, wl, [0])


def test_decoder_ratio1_chunked_prefill(csa):
    """a 512-position chunk written in the step (projected keys), per-query
    causal top-k over the ratio-1 cache"""
    wl = scaled(WORKLOADS[4], T=4096 + 512, chunk=512, ratio=1, ikey_proj=True)
    check_walk(csa, wl, [0], queries=[0, 1, 2, 255, 511])


def test_tiny_workload(csa):
    check_walk(csa, WORKLOADS[0], [0])


def test_decode_32k_all_sequences(csa):
    check_walk(csa, WORKLOADS[1], list(range(WORKLOADS[1].B)))


def test_decode_scan_on_a_key_plane_off_32_byte_alignment(csa):
    """a key-code plane that starts 16 bytes past a 32-byte boundary (allowed: the planes need
    16-byte alignment) cannot be read by the tensor copy, so the decode Full layer takes the
    CUDA-core scan and the candidate-list selection: the same top k and HSI pool as the
    tensor-core path, which the walks check against the oracle"""
    import copy
    from compressed_sparse_attention_decode_gb300.synthetic import build_step
    wl = scaled(WORKLOADS[2], B=4, T=16384, layers=("full",))
    step = build_step(wl)
    step.enqueue()
    torch.cuda.synchronize()
    c = step.cache
    n = c.ikey_codes.numel()
    buf = torch.zeros(n + 64, dtype=torch.uint8, device="cuda")
    off = (16 - buf.data_ptr() % 32) % 32
    c2 = copy.copy(c)
    c2.ikey_codes = buf[off:off + n].view(c.ikey_codes.shape)
    c2.ikey_codes.copy_(c.ikey_codes)
    assert c2.ikey_codes.data_ptr() % 32 == 16
    idx2 = torch.full_like(step.idx[0], -7)
    pool2 = torch.full_like(step.pool, -7)
    ws2 = csa.workspace(csa.OP_INDEXER_TOPK, wl.B, 1, wl.H_I, wl.k, c.capacity)
    csa.csa2_indexer_topk(c2, step.iq_codes, step.iq_scales, step.w_head[0], step.q_pos, step.k, step.pool_blocks,
                          step.bs, idx_out=idx2, pool_out=pool2, ws=ws2)
    torch.cuda.synchronize()
    assert csa.csa2_poll_error(ws2) == csa.OK
    assert torch.equal(idx2, step.idx[0])
    assert torch.equal(pool2, step.pool)


def test_layer_schedule_small(csa):
    """Full (+HSI pool) -> Reindex x3 -> Reuse x3 on a small context, 3 sequences"""
    wl = scaled(WORKLOADS[2], B=3, T=16384, layers=("full",) + ("reindex",) * 3 + ("reuse",) * 3)
    step = check_walk(csa, wl, [0, 1, 2])
    for l in (5, 6):
        assert step.layer_idx(l).data_ptr() == step.idx[3].data_ptr()


def test_pool_edge_cases(csa):
    """fewer blocks than pool slots; a pool that is the whole context; k > n_elig"""
    for T, pb, k in [(512, 256, 64), (2048 + 256, 64, 512), (4096 + 254, 16, 32)]:
        wl = scaled(WORKLOADS[2], B=2, T=T, k=k, pool_blocks=pb, H=16,
                    layers=("full", "reindex", "reuse"))
        check_walk(csa, wl, [0, 1])


def test_pages_hsi_example_pool_of_16384(csa):
    """the pool size of the pages' own example: 2048 blocks x 8 entries"""
    wl = scaled(WORKLOADS[2], B=2, T=65536, pool_blocks=2048, layers=("full", "reindex", "reuse"))
    check_walk(csa, wl, [0, 1])


@pytest.mark.parametrize("T,P,k", [(16384, 2048, 512), (4096, 2048, 512), (16384, 300, 512)])
def test_pure_top_entries_pool(csa, T, P, k):
    """the other reading of the candidate pool: the P best entries of the Full layer's scores
    (no blocks, nothing forced in); a pool covering every entry; a pool smaller than k"""
    wl = scaled(WORKLOADS[2], B=2, T=T, k=k, pool_blocks=P, pool_block_size=0, layers=("full", "reindex", "reuse"))
    check_walk(csa, wl, [0, 1])


def test_short_contexts_pad_with_minus_one(csa):
    for T in (128, 130, 200, 256):
        wl = scaled(WORKLOADS[0], T=T, k=64)
        step = check_walk(csa, wl, [0])
        n = oracle.n_elig(T - 1)
        idx = step.idx[0, 0, 0].cpu().numpy()
        assert (idx[n:] == -1).all() and sorted(idx[:n].tolist()) == list(range(n))


# ---------------------------------------------------------------- adversarial top-k

def test_topk_ties_duplicates_and_zero_keys(csa):
    n, d = 3000, 128
    rng = np.random.default_rng(7)
    base = synth.normal_f32(40, 1, (n, d))
    base[1000:1500] = base[0:500]           # exact duplicates of lower rows
    base[2000:2600] = 0.0                   # all-zero keys: score exactly 0
    kc, ks = oracle.quantize_rows(base)
    lat = oracle.quantize_rows(synth.normal_f32(40, 2, (n, 512)))
    planes = [a[None] for a in (lat[0], lat[1], kc, ks)]
    cache = host_cache(csa, planes, d)
    iq = synth.normal_f32(40, 3, (1, 1, 8, d))
    w = synth.uniform_f32(40, 4, (1, 1, 8), 0.0, 1.0)
    for wv in (w, np.zeros_like(w)):        # zero head weights: every score ties at 0
        qc, qs = oracle.quantize_rows(iq)
        p = n * 2 + 127
        for k in (512, 2048):
            idx, _ = csa.csa2_indexer_topk(cache, torch.from_numpy(qc).cuda(), torch.from_numpy(qs).cuda(),
                                           torch.from_numpy(wv).cuda(),
                                           torch.tensor([[p]], dtype=torch.int64).cuda(), k)
            S = oracle.index_scores(kc, ks, qc[0, 0], qs[0, 0], wv[0, 0], n=n)
            assert np.array_equal(idx.cpu().numpy()[0, 0], oracle.topk(S, k))


# ---------------------------------------------------------------- multi-query scan (chunked prefill)

def _mq_check(csa, kc, ks, lat, iq, w, qpos, k):
    """n_q queries of one sequence through csa2_indexer_topk (the multi-query
    tensor scan for n_q >= 4) against the oracle's exact top-k, query by query"""
    cache = host_cache(csa, [a[None] for a in (lat[0], lat[1], kc, ks)], kc.shape[1] * 2)
    qc, qs = oracle.quantize_rows(iq)
    qp = torch.tensor(np.asarray(qpos, np.int64)[None], dtype=torch.int64).cuda()
    idx, _ = csa.csa2_indexer_topk(cache, torch.from_numpy(qc).cuda(), torch.from_numpy(qs).cuda(),
                                   torch.from_numpy(w).cuda(), qp, k)
    got = idx.cpu().numpy()[0]
    for t, p in enumerate(qpos):
        S = oracle.index_scores(kc, ks, qc[0, t], qs[0, t], w[0, t], n=oracle.n_elig(p))
        assert np.array_equal(got[t], oracle.topk(S, k)), (t, p)


def test_multi_query_scan_ties_and_mixed_eligibility(csa):
    """six queries (a ragged group of four), duplicated rows and all-zero keys,
    zero head weights; eligible ranges above and below 4k (with and without a
    sampled threshold), one shorter than k and one empty"""
    n, d = 3000, 128
    base = synth.normal_f32(41, 1, (n, d))
    base[1000:1500] = base[0:500]
    base[2000:2600] = 0.0
    kc, ks = oracle.quantize_rows(base)
    lat = oracle.quantize_rows(synth.normal_f32(41, 2, (n, 512)))
    qpos = [2 * 3000 + 127, 2 * 2900 + 127, 2 * 1500 + 127, 2 * 300 + 127, 100, 2 * 2049 + 127]
    iq = synth.normal_f32(41, 3, (1, len(qpos), 8, d))
    w = synth.uniform_f32(41, 4, (1, len(qpos), 8), 0.0, 1.0)
    for wv in (w, np.zeros_like(w)):
        for k in (512, 64):
            _mq_check(csa, kc, ks, lat, iq, wv, qpos, k)


def test_multi_query_scan_unrepresentative_sample(csa):
    """keys whose large scores sit only in the sampled tiles (every eighth
    128-entry tile of 32,768): the sampled threshold is then too high for
    every query, fewer than k lower bounds reach it, and each query must be
    scanned again without one"""
    n, d = 32768, 128
    base = synth.normal_f32(42, 1, (n, d)) * np.float32(0.01)
    tiles = np.arange(n) // 128
    hot = tiles % 8 == 0
    base[hot] = np.abs(synth.normal_f32(42, 2, (int(hot.sum()), d))) * np.float32(4.0)
    kc, ks = oracle.quantize_rows(base)
    lat = oracle.quantize_rows(synth.normal_f32(42, 3, (n, 512)))
    qpos = [2 * n + 127, 2 * n + 126, 2 * n + 125, 2 * n + 124, 2 * n + 123]
    iq = np.abs(synth.normal_f32(42, 4, (1, len(qpos), 8, d)))
    w = synth.uniform_f32(42, 5, (1, len(qpos), 8), 0.1, 1.0)
    _mq_check(csa, kc, ks, lat, iq, w, qpos, 512)


def test_chunked_prefill_around_the_sampling_switch(csa):
    """a 64-position chunk whose queries see 2,029 to 2,061 entries: both
    sides of the 4k = 2,048 point where the scan starts to sample a threshold"""
    wl = scaled(WORKLOADS[4], T=4250, chunk=64)
    check_walk(csa, wl, [0])


def test_reindex_pool_with_holes_and_reuse(csa):
    n, d = 5000, 128
    lat = oracle.quantize_rows(synth.normal_f32(41, 2, (n, 512)))
    kc, ks = oracle.quantize_rows(synth.normal_f32(41, 1, (n, d)))
    cache = host_cache(csa, [a[None] for a in (lat[0], lat[1], kc, ks)], d)
    pool = np.full((1, 1, 2048), -1, np.int32)
    ids = np.sort(np.random.default_rng(3).choice(n, 1500, replace=False)).astype(np.int32)
    pool[0, 0, :1500] = ids
    iq = synth.normal_f32(41, 3, (1, 1, 8, d))
    w = synth.uniform_f32(41, 4, (1, 1, 8), 0.0, 1.0)
    qc, qs = oracle.quantize_rows(iq)
    for k in (512, 1500, 2000):
        idx = csa.csa2_reindex(csa.REINDEX, cache, k, torch.from_numpy(qc).cuda(), torch.from_numpy(qs).cuda(),
                               torch.from_numpy(w).cuda(), torch.from_numpy(pool).cuda())
        S = oracle.index_scores(kc, ks, qc[0, 0], qs[0, 0], w[0, 0], ids=pool[0, 0])
        want = oracle.topk(S, k, ids=pool[0, 0])
        assert np.array_equal(idx.cpu().numpy()[0, 0], want)
        again = csa.csa2_reindex(csa.REUSE, cache, k, prev_idx=idx)
        assert torch.equal(again, idx)
        # the same from the unquantised queries (quantised inside the Reindex kernels)
        idx32 = csa.csa2_reindex_f32(cache, k, torch.from_numpy(iq).cuda(), torch.from_numpy(w).cuda(),
                                     torch.from_numpy(pool).cuda())
        assert torch.equal(idx32, idx)


@pytest.mark.parametrize("d,H,pool_len", [(128, 8, 2048), (128, 8, 700), (64, 4, 2048), (128, 16, 1024),
                                          (64, 8, 3000)])
def test_reindex_paths_ties_holes_and_unordered_pools(csa, d, H, pool_len):
    """every Reindex path (tensor-core group sums for d_idx 128 with 8 heads, the CUDA-core
    kernel otherwise, bounds + selection above 2,048 slots) on pools with empty slots, in
    ascending and in shuffled order, over keys with exact duplicates and all-zero rows, with
    random and with all-zero head weights (every score ties)"""
    n, B, n_q = 6000, 2, 3
    base = synth.normal_f32(44, 1, (B * n, d))
    base[700:900] = base[100:300]             # duplicated rows: equal scores, lower entry first
    base[1200:1800] = 0.0                     # zero rows: score exactly 0
    kc, ks = oracle.quantize_rows(base)
    lat = oracle.quantize_rows(synth.normal_f32(44, 2, (B * n, 512)))
    planes = [a.reshape(B, n, -1) for a in (lat[0], lat[1], kc, ks)]
    cache = host_cache(csa, planes, d)
    rng = np.random.default_rng(9)
    pool = np.full((B, n_q, pool_len), -1, np.int32)
    for b in range(B):
        for q in range(n_q):
            m = pool_len - 37 * q
            ids = rng.choice(np.arange(0, max(2100, m + 100) if q == 0 else n), m, replace=False).astype(np.int32)
            if q == 1:
                ids = np.sort(ids)                # an ascending pool (as the HSI pool is) ...
            pool[b, q, :m] = ids                  # ... and two in no order
            if q == 2:
                rng.shuffle(pool[b, q])           # empty slots anywhere
    iq = synth.normal_f32(45, 3, (B, n_q, H, d))
    w = synth.uniform_f32(45, 4, (B, n_q, H), 0.0, 1.0)
    qc, qs = oracle.quantize_rows(iq)
    for wv in (w, np.zeros_like(w)):
        for k in (64, 512):
            idx = csa.csa2_reindex_f32(cache, k, torch.from_numpy(iq).cuda(), torch.from_numpy(wv).cuda(),
                                       torch.from_numpy(pool).cuda())
            got = idx.cpu().numpy()
            for b in range(B):
                for q in range(n_q):
                    ids = pool[b, q]
                    S = oracle.index_scores(kc.reshape(B, n, -1)[b], ks.reshape(B, n, -1)[b], qc[b, q], qs[b, q],
                                            wv[b, q], ids=ids)
                    assert np.array_equal(got[b, q], oracle.topk(S, k, ids=ids)), (d, H, pool_len, k, b, q)


def test_reindex_from_fp32_queries_large_pool(csa):
    """csa2_reindex_f32 through the bounds + selection path (pool above 2,048 slots), against the
    oracle and against csa2_quantize_fp4 + csa2_reindex"""
    n, d = 9000, 128
    lat = oracle.quantize_rows(synth.normal_f32(43, 2, (n, 512)))
    kc, ks = oracle.quantize_rows(synth.normal_f32(43, 1, (n, d)))
    cache = host_cache(csa, [a[None] for a in (lat[0], lat[1], kc, ks)], d)
    pool = np.full((1, 2, 6000), -1, np.int32)
    rng = np.random.default_rng(5)
    for q in range(2):
        pool[0, q, :5800] = rng.choice(n, 5800, replace=False).astype(np.int32)
    iq = synth.normal_f32(43, 3, (1, 2, 8, d))
    w = synth.uniform_f32(43, 4, (1, 2, 8), 0.0, 1.0)
    qc, qs = oracle.quantize_rows(iq)
    k = 512
    idx32 = csa.csa2_reindex_f32(cache, k, torch.from_numpy(iq).cuda(), torch.from_numpy(w).cuda(),
                                 torch.from_numpy(pool).cuda())
    codes = torch.empty((1, 2, 8, d // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((1, 2, 8, d // 16), dtype=torch.uint8, device="cuda")
    csa.csa2_quantize_fp4(torch.from_numpy(iq).cuda(), codes, scales)
    idx = csa.csa2_reindex(csa.REINDEX, cache, k, codes, scales, torch.from_numpy(w).cuda(),
                           torch.from_numpy(pool).cuda())
    assert torch.equal(idx32, idx)
    for q in range(2):
        S = oracle.index_scores(kc, ks, qc[0, q], qs[0, q], w[0, q], ids=pool[0, q])
        assert np.array_equal(idx32.cpu().numpy()[0, q], oracle.topk(S, k, ids=pool[0, q]))


def _scaled_bf16(a, e):
    """bf16 bit patterns times 2^e (exact: only the exponent field moves)"""
    f = synth.bf16_to_f32(a).astype(np.float64) * 2.0 ** e
    u = f.astype(np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16)


@pytest.mark.parametrize("H", [64])
def test_attention_inputs_far_outside_fp16_range(csa, H):
    """q heads and window rows scaled by 2^20 and 2^-30 (far outside fp16's range) must still
    match the fp64 oracle"""
    n, k = 2000, 512
    lat = oracle.quantize_rows(synth.normal_f32(46, 2, (n, 512)))
    kc, ks = oracle.quantize_rows(synth.normal_f32(46, 1, (n, 128)))
    cache = host_cache(csa, [a[None] for a in (lat[0], lat[1], kc, ks)], 128)
    p = 2 * n + 127
    idx = np.sort(np.random.default_rng(11).choice(n, k, replace=False)).astype(np.int32)[None, None]
    q0 = synth.normal_bf16(46, 3, (H, 512))
    w0 = synth.normal_bf16(46, 4, (128, 512))
    cases = []
    qa = q0.copy()
    qa[: H // 2] = _scaled_bf16(q0[: H // 2], 20)
    qa[H // 2:] = _scaled_bf16(q0[H // 2:], -30)
    cases.append((qa, w0))
    cases.append((q0, _scaled_bf16(w0, 20)))
    cases.append((q0, _scaled_bf16(w0, -30)))
    wm = w0.copy()
    wm[:64] = _scaled_bf16(w0[:64], 20)          # one CTA's half of the window far up, the other as drawn
    cases.append((_scaled_bf16(q0, 12), wm))
    for qb, win in cases:
        out, lse = csa.csa2_sparse_attn(cache, bf16_t(qb[None, None]), torch.tensor([[p]], dtype=torch.int64).cuda(),
                                        torch.from_numpy(idx).cuda(), bf16_t(win[None]), p - 127, want_lse=True)
        ro, rl = oracle.sparse_attention(qb, idx[0, 0], lat[0], lat[1], win)
        assert np.isfinite(out.cpu().numpy()).all()
        assert rel_err_rows(out.cpu().numpy()[0, 0], ro) <= ATTN_TOL


def test_bounded_wait_runs_out_and_is_reported(csa):
    """a wait on a barrier that nothing signals gives up after its poll limit; the
    failure comes back from csa2_poll_error once (the word is cleared), and the
    context stays usable: a real call afterwards runs and reports no failure"""
    wl = WORKLOADS[0]
    ws = csa.workspace(csa.OP_SPARSE_ATTN, 1, 1, wl.H, wl.k, wl.T // 2)
    assert csa.csa2_poll_error(ws) == csa.OK
    csa.csa2_selftest_wait_timeout(64, ws)
    assert csa.csa2_poll_error(ws) == csa.ERR_TIMEOUT
    assert csa.csa2_poll_error(ws) == csa.OK
    lc, ls, kc, ks = oracle.sequence_cache(wl, 0)
    cache = host_cache(csa, [a[None] for a in (lc, ls, kc, ks)], wl.d_I)
    q = wl.q(0, 0)
    idx = np.arange(0, 3 * 64, 3, dtype=np.int32)[None, None]
    out, _ = csa.csa2_sparse_attn(cache, bf16_t(q[None]), torch.tensor([[wl.T - 1]], dtype=torch.int64).cuda(),
                                  torch.from_numpy(idx).cuda(), bf16_t(wl.window(0, 0)[None]), wl.T - 128, ws=ws)
    assert csa.csa2_poll_error(ws) == csa.OK
    ro, _ = oracle.sparse_attention(q[0], idx[0, 0], lc, ls, wl.window(0, 0))
    assert rel_err_rows(out.cpu().numpy()[0, 0], ro) <= ATTN_TOL


def test_attention_window_clipping_and_empty_selection(csa):
    wl = WORKLOADS[0]
    lc, ls, kc, ks = oracle.sequence_cache(wl, 0)
    cache = host_cache(csa, [a[None] for a in (lc, ls, kc, ks)], wl.d_I)
    q = wl.q(0, 0)
    win = wl.window(0, 0)
    p = wl.T - 1
    for k_valid, clip in [(0, 0), (10, 0), (64, 100), (0, 127)]:
        idx = np.full((1, 1, 64), -1, np.int32)
        idx[0, 0, :k_valid] = np.arange(0, 3 * k_valid, 3)
        swa = win[clip:]
        out, lse = csa.csa2_sparse_attn(cache, bf16_t(q[None]), torch.tensor([[p]], dtype=torch.int64).cuda(),
                                        torch.from_numpy(idx).cuda(), bf16_t(swa[None]), wl.T - 128 + clip,
                                        want_lse=True)
        ro, rl = oracle.sparse_attention(q[0], idx[0, 0], lc, ls, swa)
        assert rel_err_rows(out.cpu().numpy()[0, 0], ro) <= ATTN_TOL
        assert np.abs(lse.cpu().numpy()[0, 0] - rl).max() < 1e-4 * max(1, np.abs(rl).max())


# ---------------------------------------------------------------- writes stay inside the outputs
# (in place of a memory checker, which this pool does not run: guard regions of a known pattern
# around every output, checked after the call; indices outside the cache are skipped, not read)

def _guarded(shape, dtype, fill, pad=256):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), fill, dtype=dtype, device="cuda")
    return buf, buf[pad:pad + n].view(shape), pad


def _guards_intact(buf, pad, fill):
    return bool((buf[:pad] == fill).all()) and bool((buf[-pad:] == fill).all())


def test_calls_write_only_their_outputs(csa):
    """a cache write touches only its entries; the scan, Reindex and attention
    write nothing past the ends of their index, pool, output and lse buffers"""
    wl = scaled(WORKLOADS[2], B=2, T=8192, pool_blocks=64)
    n, d = wl.n_entries, wl.d_I
    cache = csa.Cache(2, n, d)
    for t in (cache.lat_codes, cache.lat_scales, cache.ikey_codes, cache.ikey_scales):
        t.fill_(0xA5)
    w0, w1 = (torch.from_numpy(w).cuda() for w in wl.merge_weights())
    e0, ne = 1000, 37
    h = torch.stack([bf16_t(wl.h(b, 2 * e0, 2 * ne)) for b in range(2)])
    kr = torch.stack([bf16_t(wl.kraw(b, e0, ne)) for b in range(2)])
    csa.csa2_cache_write(cache, h, 2 * e0, w0, w1, kr)
    torch.cuda.synchronize()
    for t in (cache.lat_codes, cache.lat_scales, cache.ikey_codes, cache.ikey_scales):
        a = t.cpu().numpy()
        assert (a[:, :e0] == 0xA5).all() and (a[:, e0 + ne:] == 0xA5).all()
        assert not (a[:, e0:e0 + ne] == 0xA5).all()
    # full context for the rest
    from compressed_sparse_attention_decode_gb300.synthetic import seq_view
    for b in range(2):
        csa.csa2_cache_write(seq_view(cache, b), bf16_t(wl.h(b, 0, wl.T))[None], 0, w0, w1,
                             bf16_t(wl.kraw(b, 0, n))[None])
    k, P = wl.k, wl.pool_len
    sent = 0x5A5A5A5A
    for nq in (1, 6):                         # the decode scan and the multi-query scan
        qpos = torch.tensor([[wl.T - 1 - i for i in range(nq)]] * 2, dtype=torch.int64).cuda()
        iq = torch.from_numpy(synth.normal_f32(43, 1, (2, nq, 8, d))).cuda()
        w = torch.from_numpy(synth.uniform_f32(43, 2, (2, nq, 8), 0.0, 1.0)).cuda()
        qc, qs = csa.csa2_quantize_fp4(iq)
        ibuf, idx, pi = _guarded((2, nq, k), torch.int32, sent)
        pbuf, pool, pp = _guarded((2, nq, P), torch.int32, sent)
        pb = wl.pool_blocks if nq == 1 else 0
        csa.csa2_indexer_topk(cache, qc, qs, w, qpos, k, pb, 8, idx_out=idx, pool_out=pool if pb else None)
        torch.cuda.synchronize()
        assert _guards_intact(ibuf, pi, sent) and _guards_intact(pbuf, pp, sent)
        if pb:
            rbuf, ridx, pr = _guarded((2, nq, k), torch.int32, sent)
            csa.csa2_reindex_f32(cache, k, iq, w, pool, idx_out=ridx)
            torch.cuda.synchronize()
            assert _guards_intact(rbuf, pr, sent)
        q = torch.stack([bf16_t(wl.q(0, b)) for b in range(2)])[:, :1].repeat(1, nq, 1, 1)
        first, count = wl.swa_range()
        win = torch.stack([bf16_t(wl.window(0, b)) for b in range(2)])
        obuf, out, po = _guarded((2, nq, wl.H, 512), torch.float32, 12345.0)
        lbuf, lse, pl = _guarded((2, nq, wl.H), torch.float32, 12345.0)
        csa.csa2_sparse_attn(cache, q.contiguous(), qpos, idx, win, first, out=out, lse=lse)
        torch.cuda.synchronize()
        assert _guards_intact(obuf, po, 12345.0) and _guards_intact(lbuf, pl, 12345.0)


def test_indices_outside_the_cache_are_skipped(csa):
    """attention indices and Reindex pool entries at or past the capacity, or
    negative, are empty slots: the results equal the oracle's with -1 there"""
    wl = WORKLOADS[0]
    lc, ls, kc, ks = oracle.sequence_cache(wl, 0)
    cache = host_cache(csa, [a[None] for a in (lc, ls, kc, ks)], wl.d_I)
    n = lc.shape[0]
    q = wl.q(0, 0)
    win = wl.window(0, 0)
    p = wl.T - 1
    idx = np.arange(0, 3 * 64, 3, dtype=np.int32)[None, None].copy()
    bad = [n, n + 5, 2**31 - 1, -7, -2**31]
    idx[0, 0, 10:15] = bad
    out, _ = csa.csa2_sparse_attn(cache, bf16_t(q[None]), torch.tensor([[p]], dtype=torch.int64).cuda(),
                                  torch.from_numpy(idx).cuda(), bf16_t(win[None]), wl.T - 128)
    clean = idx[0, 0].copy()
    clean[10:15] = -1
    ro, _ = oracle.sparse_attention(q[0], clean, lc, ls, win)
    assert rel_err_rows(out.cpu().numpy()[0, 0], ro) <= ATTN_TOL
    # a Reindex pool with entries outside the cache
    pool = np.full((1, 1, 512), -1, np.int32)
    pool[0, 0, :400] = np.arange(0, 800, 2)
    pool[0, 0, 400:405] = bad
    iq = synth.normal_f32(44, 1, (1, 1, wl.H_I, wl.d_I))
    w = synth.uniform_f32(44, 2, (1, 1, wl.H_I), 0.0, 1.0)
    qc, qs = oracle.quantize_rows(iq)
    got = csa.csa2_reindex(csa.REINDEX, cache, 64, torch.from_numpy(qc).cuda(), torch.from_numpy(qs).cuda(),
                           torch.from_numpy(w).cuda(), torch.from_numpy(pool).cuda())
    cp = pool[0, 0].copy()
    cp[400:405] = -1
    S = oracle.index_scores(kc, ks, qc[0, 0], qs[0, 0], w[0, 0], ids=cp)
    assert np.array_equal(got.cpu().numpy()[0, 0], oracle.topk(S, 64, ids=cp))


# ---------------------------------------------------------------- full sizes, sampled outputs

def test_decode_128k_20_layers_full_size_sampled(csa):
    """the benchmark's workload and launch configuration (one CUDA graph per
    step), checked on three sequences across all 20 layers"""
    from compressed_sparse_attention_decode_gb300.synthetic import build_step
    wl = WORKLOADS[2]
    step = build_step(wl)
    step.capture()
    step.run()
    step.run()
    torch.cuda.synchronize()
    for b in (0, 37, 63):
        ref = oracle.run_sequence(wl, b)
        for l in range(len(wl.layers)):
            assert np.array_equal(step.layer_idx(l)[b].cpu().numpy(), ref["idx"][l]), (b, l)
            err = rel_err_rows(step.out[l, b].cpu().numpy(), ref["out"][l])
            assert err <= ATTN_TOL, (b, l, err)
        assert np.array_equal(step.pool[b].cpu().numpy(), ref["pool"][0])


def test_decode_1m_full_size_sampled(csa):
    from compressed_sparse_attention_decode_gb300.synthetic import build_step
    wl = WORKLOADS[3]
    step = build_step(wl)
    step.enqueue()
    torch.cuda.synchronize()
    for b in (0, 3):
        ref = oracle.run_sequence(wl, b)
        assert np.array_equal(step.idx[0, b].cpu().numpy(), ref["idx"][0])
        assert rel_err_rows(step.out[0, b].cpu().numpy(), ref["out"][0]) <= ATTN_TOL


def test_chunked_prefill_full_size_sampled(csa):
    """cache write of the 8,192-position chunk plus per-query causal top-512
    and attention; queries checked: every 64th plus the first and the last"""
    from compressed_sparse_attention_decode_gb300.synthetic import build_step
    wl = WORKLOADS[4]
    step = build_step(wl)
    step.enqueue()
    torch.cuda.synchronize()
    ref_cache = oracle.sequence_cache(wl, 0)
    for got, want in zip((step.cache.lat_codes, step.cache.lat_scales, step.cache.ikey_codes,
                          step.cache.ikey_scales), ref_cache):
        assert np.array_equal(got[0].cpu().numpy(), want)
    qs = sorted(set(list(range(0, wl.n_q, 64)) + [1, wl.n_q - 1]))
    ref = oracle.run_sequence(wl, 0, cache=ref_cache, queries=qs)
    assert np.array_equal(step.idx[0, 0].cpu().numpy()[qs], ref["idx"][0])
    assert rel_err_rows(step.out[0, 0].cpu().numpy()[qs], ref["out"][0]) <= ATTN_TOL

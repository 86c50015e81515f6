"""csa2_reindex_noalloc: the Reindex entry point for callers that cannot
allocate device memory (it uses a fixed scratch array inside the library
instead of a caller workspace).  Its results must equal those of
csa2_reindex, bit for bit, call after call.  This file is collected last so
that a run stopping at the first failure has run every other test first; it
also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_decode_gb300 as m
    from compressed_sparse_attention_decode_gb300 import build as b
    b.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def _case(csa, seed, B, n_q, n, pool_len):
    """a cache of B sequences x n entries and one pool per query, all drawn on the host"""
    d = 128
    lat = oracle.quantize_rows(synth.normal_f32(seed, 1, (B * n, 512)))
    kc, ks = oracle.quantize_rows(synth.normal_f32(seed, 2, (B * n, d)))
    cache = csa.Cache(B, n, d)
    for t, a in zip((cache.lat_codes, cache.lat_scales, cache.ikey_codes, cache.ikey_scales),
                    (lat[0], lat[1], kc, ks)):
        t.copy_(torch.from_numpy(a.reshape(B, n, -1)))
    iq = synth.normal_f32(seed, 3, (B, n_q, 8, d))
    qc, qs = oracle.quantize_rows(iq)
    w = synth.uniform_f32(seed, 4, (B, n_q, 8), 0.0, 1.0)
    rng = np.random.default_rng(seed)
    pool = np.full((B, n_q, pool_len), -1, np.int32)
    for b in range(B):
        for q in range(n_q):
            m = pool_len - (q % 3) * 17                # a few empty slots at the end of some pools
            pool[b, q, :m] = np.sort(rng.choice(n, m, replace=False))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return cache, dev(qc), dev(qs), dev(w), dev(pool)


def test_noalloc_reindex_matches_workspace_reindex_twice(csa):
    lib = csa.load()
    for seed, (B, n_q, n, pool_len, k) in enumerate([(4, 2, 6000, 2048, 512), (2, 1, 3000, 700, 64)]):
        cache, qc, qs, w, pool = _case(csa, 50 + seed, B, n_q, n, pool_len)
        ref = csa.csa2_reindex(csa.REINDEX, cache, k, qc, qs, w, pool)
        for _ in range(2):                            # two calls in a row through the C ABI
            out = torch.full((B, n_q, k), -7, dtype=torch.int32, device="cuda")
            c = cache.struct()
            st = lib.csa2_reindex_noalloc(ctypes.byref(c), ctypes.c_void_p(qc.data_ptr()),
                                          ctypes.c_void_p(qs.data_ptr()), ctypes.c_void_p(w.data_ptr()), n_q, 8,
                                          ctypes.c_void_p(pool.data_ptr()), pool_len, k,
                                          ctypes.c_void_p(out.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == csa.OK
            torch.cuda.synchronize()
            assert torch.equal(out, ref)
    # the same through the binding
    cache, qc, qs, w, pool = _case(csa, 60, 2, 1, 3000, 1024)
    assert torch.equal(csa.csa2_reindex_noalloc(cache, 128, qc, qs, w, pool),
                       csa.csa2_reindex(csa.REINDEX, cache, 128, qc, qs, w, pool))


def _noalloc(csa, cache, qc, qs, w, pool, k):
    lib = csa.load()
    B, n_q, pool_len = pool.shape
    out = torch.full((B, n_q, k), -7, dtype=torch.int32, device="cuda")
    c = cache.struct()
    st = lib.csa2_reindex_noalloc(ctypes.byref(c), ctypes.c_void_p(qc.data_ptr()), ctypes.c_void_p(qs.data_ptr()),
                                  ctypes.c_void_p(w.data_ptr()), n_q, 8, ctypes.c_void_p(pool.data_ptr()), pool_len,
                                  k, ctypes.c_void_p(out.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == csa.OK
    torch.cuda.synchronize()
    return out


def test_noalloc_large_pool_after_a_differently_shaped_call_matches_the_oracle(csa):
    """a pool above 2048 slots takes the bounds + selection kernels; run it right
    after a small call, so it finds the scratch holding another call's data"""
    cache, qc, qs, w, pool = _case(csa, 70, 2, 3, 3000, 300)
    _noalloc(csa, cache, qc, qs, w, pool, 32)
    B, n_q, n, pool_len, k = 2, 2, 9000, 5000, 512
    cache, qc, qs, w, pool = _case(csa, 71, B, n_q, n, pool_len)
    for _ in range(2):
        out = _noalloc(csa, cache, qc, qs, w, pool, k)
        assert torch.equal(out, csa.csa2_reindex(csa.REINDEX, cache, k, qc, qs, w, pool))
    kc = cache.ikey_codes.cpu().numpy()
    ks = cache.ikey_scales.cpu().numpy()
    qcn, qsn, wn, pn = qc.cpu().numpy(), qs.cpu().numpy(), w.cpu().numpy(), pool.cpu().numpy()
    for b in range(B):
        for q in range(n_q):
            ids = pn[b, q]
            S = oracle.index_scores(kc[b], ks[b], qcn[b, q], qsn[b, q], wn[b, q], ids=ids)
            S = np.where(ids >= 0, S, -np.inf)
            assert np.array_equal(out[b, q].cpu().numpy(), oracle.topk(S, k, ids=ids))


def test_noalloc_reindex_rejects_requests_beyond_its_scratch(csa):
    lib = csa.load()
    c = csa._CacheStruct(256, 256, 256, 256, 64, 100000, 512, 128, 2)
    p = ctypes.c_void_p(256)
    # 64 sequences x 4 queries x 16384 pool slots needs far more than 8 MiB
    assert lib.csa2_reindex_noalloc(ctypes.byref(c), p, p, p, 4, 8, p, 16384, 512, p, None) == csa.ERR_WORKSPACE

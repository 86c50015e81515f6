"""Pins for the indexer score, top-k, HSI pool and the Full/Reindex/Reuse walk."""
import heapq
from fractions import Fraction

import numpy as np
import torch

import oracle
import synth
from conftest import read_golden
from exact import rn_f64
from synth.workloads import WORKLOADS, scaled

E2M1 = {int(k, 16): float(v) for k, v in read_golden("e2m1_values.txt").items()}
FP8 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _frac_rows(codes, scales):
    """decode with the standard table and torch's float8 (not oracle.c)"""
    d = codes.shape[-1] * 2
    out = []
    for r in range(codes.shape[0]):
        row = []
        for i in range(d):
            b = int(codes[r, i // 2])
            nib = (b >> 4) if i & 1 else (b & 15)
            row.append(Fraction(E2M1[nib]) * Fraction(float(FP8[scales[r, i // 16]])))
        out.append(row)
    return out


def _score_exact(qrows, krow, w):
    S = 0.0
    for h, qr in enumerate(qrows):
        d = sum(a * b for a, b in zip(qr, krow))      # exact rational
        r = d if d > 0 else Fraction(0)
        S = rn_f64(Fraction(float(w[h])) * r + Fraction(S))   # one fp64 fma
    return S


def test_scores_equal_exact_rational_evaluation():
    rng = np.random.default_rng(0)
    for d, H in [(64, 4), (128, 8)]:
        kc, ks = oracle.quantize_rows(rng.normal(size=(40, d)).astype(np.float32)
                                      * np.exp(rng.uniform(-8, 6, (40, 1))).astype(np.float32))
        qc, qs = oracle.quantize_rows(rng.normal(size=(H, d)).astype(np.float32)
                                      * np.exp(rng.uniform(-8, 6, (H, 1))).astype(np.float32))
        w = rng.uniform(0, 1, H).astype(np.float32)
        S = oracle.index_scores(kc, ks, qc, qs, w, n=40)
        qf = _frac_rows(qc, qs)
        kf = _frac_rows(kc, ks)
        for j in range(40):
            assert S[j] == _score_exact(qf, kf[j], w), j


def test_score_invariants():
    rng = np.random.default_rng(1)
    kc, ks = oracle.quantize_rows(rng.normal(size=(300, 128)).astype(np.float32))
    qc, qs = oracle.quantize_rows(rng.normal(size=(8, 128)).astype(np.float32))
    w = rng.uniform(0, 1, 8).astype(np.float32)
    S = oracle.index_scores(kc, ks, qc, qs, w, n=300)
    assert np.all(S >= 0)
    # doubling every head weight doubles every score exactly
    assert np.array_equal(oracle.index_scores(kc, ks, qc, qs, 2 * w, n=300), 2 * S)
    # zero weights, or a query whose heads all see negative dots, score 0
    assert not oracle.index_scores(kc, ks, qc, qs, 0 * w, n=300).any()
    # flipping the key's sign turns ReLU(d) into ReLU(-d): S(k) + S(-k) = sum_h w_h |d_h|
    kneg = kc ^ np.where((kc & 0x07) != 0, 0x08, 0).astype(np.uint8) ^ np.where((kc & 0x70) != 0, 0x80, 0).astype(np.uint8)
    Sn = oracle.index_scores(kneg, ks, qc, qs, w, n=300)
    qd = oracle.dequant_rows(qc, qs)
    kd = oracle.dequant_rows(kc, ks)
    absdot = np.abs(kd @ qd.T) @ w.astype(np.float64)
    assert np.allclose(S + Sn, absdot, rtol=1e-12)
    # ids select entries; negative ids score -inf
    ids = np.array([5, -1, 299, 0], np.int32)
    Si = oracle.index_scores(kc, ks, qc, qs, w, ids=ids)
    assert Si[0] == S[5] and Si[1] == -np.inf and Si[2] == S[299] and Si[3] == S[0]


def test_topk_brute_force_and_heap_select():
    rng = np.random.default_rng(2)
    for n, k in [(10, 3), (100, 100), (50, 64), (1000, 17), (0, 4)]:
        S = np.round(rng.normal(size=n), 1)           # many exact ties
        got = oracle.topk(S, k)
        ref = sorted(range(n), key=lambda j: (-S[j], j))[:k]
        heap = [j for _, j in heapq.nsmallest(k, [(-S[j], j) for j in range(n)])]
        want = sorted(ref) + [-1] * (k - len(ref))        # the chosen set, ascending
        assert got.tolist() == want and heap == ref


def test_topk_duplicate_rows_prefer_lower_index():
    rng = np.random.default_rng(3)
    base = rng.normal(size=(8, 64)).astype(np.float32)
    rows = np.concatenate([base, base, base])          # entries j, j+8, j+16 identical
    kc, ks = oracle.quantize_rows(rows)
    qc, qs = oracle.quantize_rows(rng.normal(size=(4, 64)).astype(np.float32))
    w = rng.uniform(0, 1, 4).astype(np.float32)
    S = oracle.index_scores(kc, ks, qc, qs, w, n=24)
    top = oracle.topk(S, 12)
    for j in top:
        for dup in (j - 8, j - 16):
            if dup >= 0:
                assert dup in top   # a copy is taken only after the lower-index original
    # all scores equal (all-zero keys): the k lowest indices
    zc = np.zeros_like(kc)
    zs = np.zeros_like(ks)
    S0 = oracle.index_scores(zc, zs, qc, qs, w, n=24)
    assert oracle.topk(S0, 5).tolist() == [0, 1, 2, 3, 4]


def _hsi_tensor_ops(S, bs, n_sel):
    """the block pipeline written with tensor ops: pad to whole blocks with
    -inf, max per block, newest block to +inf, best blocks, block flags
    expanded back to entry width"""
    x = torch.tensor(S, dtype=torch.float64)
    width = x.shape[0]
    pad = (-width) % bs
    x = torch.cat([x, torch.full((pad,), -float("inf"), dtype=torch.float64)])
    bmax = x.view(-1, bs).max(dim=1).values
    bmax[(width - 1) // bs] = float("inf")
    keep = torch.topk(bmax, min(n_sel, bmax.shape[0])).indices
    flag = torch.zeros(bmax.shape[0], dtype=torch.bool)
    flag[keep] = True
    bitmap = flag.repeat_interleave(bs)[:width]
    pool = torch.nonzero(bitmap).flatten().tolist()
    return pool + [-1] * (n_sel * bs - len(pool))


def test_hsi_pool_against_tensor_ops():
    rng = np.random.default_rng(4)
    for n, bs, nsel in [(100, 8, 4), (97, 8, 5), (64, 8, 8), (30, 8, 16), (1000, 8, 25), (24, 1, 10), (5, 4, 1)]:
        S = rng.permutation(n).astype(np.float64)       # distinct scores
        got = oracle.hsi_pool(S, bs, nsel)
        assert got.tolist() == _hsi_tensor_ops(S, bs, nsel), (n, bs, nsel)


def test_hsi_pool_invariants_and_ties():
    rng = np.random.default_rng(5)
    for n in [1, 7, 8, 9, 2047, 2048, 2049, 65472]:
        S = np.floor(rng.uniform(0, 50, n))             # ties between blocks
        pool = oracle.hsi_pool(S, 8, 256)
        valid = pool[pool >= 0]
        assert n - 1 in valid                             # newest block always in
        assert np.all(np.diff(valid) > 0) and valid.max() < n
        if n <= 2048:
            assert np.array_equal(valid, np.arange(n))
        else:
            # 256 whole blocks, one of them the (full or partial) newest block
            assert len(valid) == 255 * 8 + (n - 8 * ((n - 1) // 8))
    # equal block maxima: the lower block wins
    S = np.zeros(80)
    assert oracle.hsi_pool(S, 8, 3).tolist() == list(range(16)) + list(range(72, 80))
    assert oracle.hsi_pool(np.zeros(0), 8, 2).tolist() == [-1] * 16


def test_toy_full_reindex_reuse_example():
    """24 positions, pool of 10 (block size 1), 4 read positions 2, 10, 15, 23
    kept unchanged by Reuse.  Scores are built by hand so that Full's pool is
    {0, 2, 4, 7, 10, 11, 15, 18, 20, 23} (23 is the newest, forced in) and the
    Reindex layer picks 2, 10, 15, 23 inside it."""
    g = read_golden("toy_reuse.txt")
    n, P = int(g["positions"]), int(g["pool_size"])
    read = [int(x) for x in g["read"].split(",")]
    full = np.zeros(n)
    for rank, j in enumerate([10, 2, 15, 20, 4, 0, 18, 7, 11]):
        full[j] = 100 - rank
    pool = oracle.hsi_pool(full, 1, P)
    assert sorted(pool.tolist()) == [0, 2, 4, 7, 10, 11, 15, 18, 20, 23]
    re = np.zeros(n)
    for j, v in zip(read, [5.0, 9.0, 7.0, 8.0]):
        re[j] = v
    re[3] = 50.0                                        # not in the pool: must not be picked
    S_pool = re[pool]
    idx = oracle.topk(S_pool, 4, ids=pool)
    assert idx.tolist() == read                         # the pages' read positions, in their order
    reuse = idx.copy()                                  # Reuse: same entries, new weights
    assert reuse.tolist() == idx.tolist()


def test_walk_reuse_copies_and_reindex_stays_in_pool():
    wl = scaled(WORKLOADS[2], B=1, T=4096, H=4, layers=("full", "reindex", "reindex", "reuse", "reuse"),
                pool_blocks=16, k=32)
    res = oracle.run_sequence(wl, 0, want_out=False)
    pool = res["pool"][0][0]
    assert len(pool) == 128 and (pool >= 0).all()
    for l in (1, 2):
        assert set(res["idx"][l][0].tolist()) <= set(pool.tolist())
    assert np.array_equal(res["idx"][3], res["idx"][2]) and np.array_equal(res["idx"][4], res["idx"][2])
    n_elig = oracle.n_elig(wl.T - 1)
    assert res["idx"][0].max() < n_elig


def test_pure_pool_is_the_best_entries_and_reindex_stays_in_it():
    """pool_block_size 0: the Full layer's pool is its P best entries by (score desc, entry asc),
    ascending, by brute force over the exact scores; Reindex layers choose inside it"""
    wl = scaled(WORKLOADS[2], B=1, T=4096, H=4, k=32, pool_blocks=100, pool_block_size=0,
                layers=("full", "reindex", "reuse"))
    res = oracle.run_sequence(wl, 0, want_out=False)
    lc, ls, kc, ks = oracle.sequence_cache(wl, 0)
    qc, qs = oracle.quantize_rows(wl.iq(0, 0))
    n = oracle.n_elig(wl.T - 1)
    S = oracle.index_scores(kc, ks, qc[0], qs[0], wl.w_head(0, 0)[0], n=n)
    best = sorted(range(n), key=lambda j: (-S[j], j))[:100]
    assert res["pool"][0][0].tolist() == sorted(best)
    assert set(res["idx"][1][0].tolist()) <= set(best)
    assert np.array_equal(res["idx"][2], res["idx"][1])


def test_walk_takes_each_layer_own_query_and_the_latest_full_pool():
    """Each layer of the walk, re-derived by brute force: a Full layer's k best entries (score desc,
    entry asc) under its own query and head weights; a Reindex layer's k best inside the pool of the
    latest Full layer, under its own query; a Reuse layer repeats the layer before it ([P1] §2.3.2,
    §2.3.4).  Two Full layers with different pools, so that taking a stale pool or another layer's
    query fails."""
    layers = ("full", "reindex", "reuse", "full", "reindex", "reuse")
    wl = scaled(WORKLOADS[2], B=1, T=4096, H=4, layers=layers, pool_blocks=16, k=32)
    res = oracle.run_sequence(wl, 0, want_out=False)
    lc, ls, kc, ks = oracle.sequence_cache(wl, 0)
    qpos = wl.q_positions()

    def best(S, ids, k):
        order = sorted(range(len(ids)), key=lambda i: (-S[i], ids[i]))[:k]
        got = sorted(int(ids[i]) for i in order)
        return got + [-1] * (k - len(got))

    assert not np.array_equal(res["pool"][0], res["pool"][3])
    pool = None
    for l, mode in enumerate(layers):
        qc, qs = oracle.quantize_rows(wl.iq(l, 0)) if mode != "reuse" else (None, None)
        for t in range(wl.n_q):
            if mode == "full":
                n = oracle.n_elig(int(qpos[t]))
                S = oracle.index_scores(kc, ks, qc[t], qs[t], wl.w_head(l, 0)[t], n=n)
                assert res["idx"][l][t].tolist() == best(S, list(range(n)), wl.k)
            elif mode == "reindex":
                ids = res["pool"][pool][t]
                S = oracle.index_scores(kc, ks, qc[t], qs[t], wl.w_head(l, 0)[t], ids=ids)
                assert res["idx"][l][t].tolist() == best(S, ids.tolist(), wl.k)
            else:
                assert res["idx"][l][t].tolist() == res["idx"][l - 1][t].tolist()
        if mode == "full":
            pool = l

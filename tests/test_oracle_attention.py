"""Pins for the oracle's sparse attention over selected entries + window."""
import numpy as np
import torch

import oracle
import synth

D = 512


def _cache(n, seed):
    h = synth.normal_bf16(seed, 1, (2 * n, D))
    kraw = synth.normal_bf16(seed, 2, (n, 64))
    w0 = synth.uniform_f32(seed, 3, (D,), 0.3, 0.7)
    w1 = synth.uniform_f32(seed, 4, (D,), 0.3, 0.7)
    return oracle.cache_write(h, w0, w1, kraw)


def _sdpa(q, keys, scale):
    """torch's scaled_dot_product_attention in float64, K = V = keys (MQA)"""
    qt = torch.from_numpy(synth.bf16_to_f32(q).astype(np.float64))[None, :, None, :]
    kt = torch.from_numpy(keys)[None, None].expand(1, q.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, kt, scale=scale)
    s = (qt @ kt.transpose(-1, -2))[0, :, 0, :] * scale
    return o[0, :, 0].numpy(), torch.logsumexp(s, dim=-1).numpy()


def test_matches_torch_sdpa_float64():
    lc, ls, _, _ = _cache(300, 21)
    q = synth.normal_bf16(21, 5, (8, D))
    win = synth.normal_bf16(21, 6, (128, D))
    idx = np.array([5, 17, 299, 0, -1, 42, 42 + 100, -1], np.int32)
    o, lse = oracle.sparse_attention(q, idx, lc, ls, win)
    keys = np.concatenate([oracle.dequant_rows(lc[idx[idx >= 0]], ls[idx[idx >= 0]]),
                           synth.bf16_to_f32(win).astype(np.float64)])
    ro, rl = _sdpa(q, keys, oracle.SCALE)
    assert np.allclose(o, ro, rtol=1e-12, atol=1e-13) and np.allclose(lse, rl, rtol=1e-13)


def test_weights_sum_to_one_and_special_cases():
    lc, ls, _, _ = _cache(64, 22)
    win = synth.normal_bf16(22, 6, (1, D))
    # one key only: output equals that key exactly
    q = synth.normal_bf16(22, 5, (4, D))
    o, lse = oracle.sparse_attention(q, np.array([-1, -1], np.int32), lc, ls, win)
    assert np.array_equal(o, np.repeat(synth.bf16_to_f32(win).astype(np.float64), 4, 0))
    o, _ = oracle.sparse_attention(q, np.array([7], np.int32), lc, ls, win[:0])
    assert np.allclose(o, oracle.dequant_rows(lc[7:8], ls[7:8]).repeat(4, 0), rtol=0, atol=1e-15)
    # zero query: every weight 1/n, output = plain mean of the keys, lse = log n
    zq = np.zeros((2, D), np.uint16)
    idx = np.arange(0, 64, 3, dtype=np.int32)
    win2 = synth.normal_bf16(22, 7, (128, D))
    o, lse = oracle.sparse_attention(zq, idx, lc, ls, win2)
    keys = np.concatenate([oracle.dequant_rows(lc[idx], ls[idx]), synth.bf16_to_f32(win2).astype(np.float64)])
    assert np.allclose(o, keys.mean(0)[None], rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, np.log(len(keys)), rtol=1e-14)
    # softmax weights sum to one: sum_j exp(s_j - lse) = 1
    q = synth.normal_bf16(22, 8, (3, D))
    o, lse = oracle.sparse_attention(q, idx, lc, ls, win2)
    s = synth.bf16_to_f32(q).astype(np.float64) @ keys.T * oracle.SCALE
    assert np.allclose(np.exp(s - lse[:, None]).sum(1), 1.0, rtol=1e-12)


def test_order_of_indices_does_not_matter():
    lc, ls, _, _ = _cache(200, 23)
    q = synth.normal_bf16(23, 5, (4, D))
    win = synth.normal_bf16(23, 6, (128, D))
    idx = np.arange(10, 190, 7, dtype=np.int32)
    a, la = oracle.sparse_attention(q, idx, lc, ls, win)
    b, lb = oracle.sparse_attention(q, idx[::-1].copy(), lc, ls, win)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14) and np.allclose(la, lb, rtol=1e-14)


def test_sparse_with_k_covering_all_entries_equals_dense():
    n = 200
    lc, ls, _, _ = _cache(n, 24)
    q = synth.normal_bf16(24, 5, (4, D))
    win = synth.normal_bf16(24, 6, (128, D))
    n_elig = 150
    idx = np.concatenate([np.arange(n_elig), [-1] * 10]).astype(np.int32)
    a, la = oracle.sparse_attention(q, idx, lc, ls, win)
    b, lb = oracle.dense_attention(q, n_elig, lc, ls, win)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14) and np.allclose(la, lb, rtol=1e-13)


def test_eligibility_rule_and_window_are_disjoint_and_cover_the_context():
    """global entry i covers raw positions 2i, 2i+1; a query at p reads entries
    lying wholly before its window [p-127, p] and the window rows themselves"""
    # the decode queries of the workloads: T - 1 for T = 2048, 131072, 1048576
    assert [oracle.n_elig(T - 1) for T in (2048, 131072, 1048576)] == [960, 65472, 524224]
    assert oracle.n_elig(0) == 0 and oracle.n_elig(126) == 0 and oracle.n_elig(128) == 0
    for p in [127, 128, 129, 130, 255, 2047, 131071]:
        n = oracle.n_elig(p)
        covered = set(range(0, 2 * n))
        window = set(range(max(0, p - 127), p + 1))
        assert not covered & window
        # entry n (the next one) would reach into the window
        assert 2 * n - 1 < p - 127 and 2 * (n + 1) - 1 >= p - 127
        missing = set(range(0, p + 1)) - covered - window
        # decode queries sit at an odd raw position (T-1, T even): nothing is missed;
        # otherwise only the half entry straddling the window edge is unread
        assert missing == (set() if (p - 127) % 2 == 0 else {p - 128})


def test_tiny_workload_walk_and_dense_agreement():
    from synth.workloads import WORKLOADS, scaled
    wl = WORKLOADS[0]
    res = oracle.run_sequence(wl, 0)
    idx = res["idx"][0][0]
    assert len(set(idx.tolist())) == 64 and idx.min() >= 0 and idx.max() < 960
    # with k covering every eligible entry the walk's output equals dense attention
    small = scaled(wl, T=512, k=256)
    res = oracle.run_sequence(small, 0)
    n_elig = oracle.n_elig(small.T - 1)
    assert sorted(res["idx"][0][0][:n_elig].tolist()) == list(range(n_elig))
    lc, ls, _, _ = oracle.sequence_cache(small, 0)
    dense, _ = oracle.dense_attention(small.q(0, 0)[0], n_elig, lc, ls, small.window(0, 0))
    assert np.allclose(res["out"][0][0], dense, rtol=1e-12, atol=1e-14)

"""fp64 CPU oracle for CSA2 decode.  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the library never does.  It shares no
code with the CUDA path: the arithmetic lives in ``oracle.c`` (plain C, fp64
loops) and this wrapper only marshals numpy arrays and walks the layers of a
workload.  Inputs come from the seeded generator in ``synth``.

Every function of oracle.c is pinned by a ``-m "not gpu"`` test
(tests/test_oracle_*.py) against closed forms, brute force on tiny inputs,
invariants or values printed on the pages.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

SCALE = 1.0 / np.sqrt(512.0)
WINDOW = 128


def n_elig(p, ratio=2):
    """Global entries a query at raw position p may attend to besides its window:
    the entries lying wholly before the window [p-127, p] ("DeepSeek-v4.1 Flash"
    §2.3.1: each query reads its selected global entries plus the local window;
    §2.3.4: the indexer scores the causally visible entries).  Entry i covers raw
    positions [ratio*i, ratio*i + ratio - 1], so it is eligible when
    ratio*i + ratio - 1 < p - 127."""
    p = int(p)
    if p < WINDOW - 1:
        return 0
    return (p - (WINDOW - 1)) // ratio


def build(force=False):
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i64, i32, f64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.orc_e2m1_value.argtypes = [i32]
        lib.orc_e2m1_value.restype = f64
        lib.orc_e4m3_value.argtypes = [i32]
        lib.orc_e4m3_value.restype = f64
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_e4m3_encode.restype = i32
        lib.orc_e2m1_encode.argtypes = [ctypes.c_float, f64]
        lib.orc_e2m1_encode.restype = i32
        lib.orc_quantize_rows.argtypes = [vp, i64, i32, vp, vp]
        lib.orc_dequant_rows.argtypes = [vp, vp, i64, i32, vp]
        lib.orc_merge_pairs.argtypes = [vp, i64, i32, vp, vp, vp]
        lib.orc_cache_write.argtypes = [vp, i64, i32, vp, vp, vp, i32, vp, vp, vp, vp]
        lib.orc_cache_write_r1.argtypes = [vp, i64, i32, vp, vp]
        lib.orc_project_ikeys.argtypes = [vp, vp, i64, i32, vp, vp, i32, vp, vp]
        lib.orc_index_scores.argtypes = [vp, vp, i32, vp, i64, vp, vp, vp, i32, vp]
        lib.orc_topk.argtypes = [vp, vp, i64, i32, vp]
        lib.orc_hsi_pool.argtypes = [vp, i64, i32, i32, vp]
        lib.orc_sparse_attention.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, i64, f64, vp, vp]
        lib.orc_dense_attention.argtypes = [vp, i32, i32, i64, vp, vp, vp, i64, f64, vp, vp]
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ---------------------------------------------------------------- formats
def e2m1_value(nibble):
    return _load().orc_e2m1_value(int(nibble))


def e4m3_value(byte):
    return _load().orc_e4m3_value(int(byte))


def e4m3_encode(v):
    return _load().orc_e4m3_encode(float(v))


def e2m1_encode(x, s):
    return _load().orc_e2m1_encode(float(x), float(s))


def quantize_rows(x):
    """float32 [..., d] -> (codes uint8 [..., d/2], scales uint8 [..., d/16])"""
    x = np.ascontiguousarray(x, np.float32)
    d = x.shape[-1]
    rows = x.size // d
    codes = np.empty(x.shape[:-1] + (d // 2,), np.uint8)
    scales = np.empty(x.shape[:-1] + (d // 16,), np.uint8)
    _load().orc_quantize_rows(x.ctypes.data, rows, d, codes.ctypes.data, scales.ctypes.data)
    return codes, scales


def dequant_rows(codes, scales):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    d = codes.shape[-1] * 2
    rows = codes.size // (d // 2)
    out = np.empty(codes.shape[:-1] + (d,), np.float64)
    _load().orc_dequant_rows(codes.ctypes.data, scales.ctypes.data, rows, d, out.ctypes.data)
    return out


# ---------------------------------------------------------------- cache write
def merge_pairs(h, w0, w1):
    """bf16 (uint16) [2n, d] -> float32 [n, d]"""
    h, hp = _c(h, np.uint16)
    n, d = h.shape[0] // 2, h.shape[1]
    w0, w0p = _c(w0, np.float32)
    w1, w1p = _c(w1, np.float32)
    e = np.empty((n, d), np.float32)
    _load().orc_merge_pairs(hp, n, d, w0p, w1p, e.ctypes.data)
    return e


def cache_write(h, w0, w1, kraw):
    """One sequence: h bf16 [n_pos, 512], kraw bf16 [n_pos/2, d_I] ->
    (lat_codes [n,256], lat_scales [n,32], ikey_codes [n,d_I/2], ikey_scales [n,d_I/16])"""
    h, hp = _c(h, np.uint16)
    kraw, kp = _c(kraw, np.uint16)
    n_pos, d_lat = h.shape
    n = n_pos // 2
    d_idx = kraw.shape[1]
    assert kraw.shape[0] == n
    w0, w0p = _c(w0, np.float32)
    w1, w1p = _c(w1, np.float32)
    lc = np.empty((n, d_lat // 2), np.uint8)
    ls = np.empty((n, d_lat // 16), np.uint8)
    kc = np.empty((n, d_idx // 2), np.uint8)
    ks = np.empty((n, d_idx // 16), np.uint8)
    _load().orc_cache_write(hp, n_pos, d_lat, w0p, w1p, kp, d_idx, lc.ctypes.data, ls.ctypes.data,
                            kc.ctypes.data, ks.ctypes.data)
    return lc, ls, kc, ks


def cache_write_r1(h):
    """Decoder cache (one entry per raw position): h bf16 [n_pos, 512] ->
    (lat_codes [n_pos, 256], lat_scales [n_pos, 32])"""
    h, hp = _c(h, np.uint16)
    n, d = h.shape
    lc = np.empty((n, d // 2), np.uint8)
    ls = np.empty((n, d // 16), np.uint8)
    _load().orc_cache_write_r1(hp, n, d, lc.ctypes.data, ls.ctypes.data)
    return lc, ls


def project_ikeys(lat_codes, lat_scales, w_codes, w_scales):
    """indexer keys projected from the stored entries: FP4(fp32(W . L)) ->
    (ikey_codes [n, d_idx/2], ikey_scales [n, d_idx/16])"""
    lat_codes, lcp = _c(lat_codes, np.uint8)
    lat_scales, lsp = _c(lat_scales, np.uint8)
    w_codes, wcp = _c(w_codes, np.uint8)
    w_scales, wsp = _c(w_scales, np.uint8)
    n, d_lat = lat_codes.shape[0], lat_codes.shape[1] * 2
    d_idx = w_codes.shape[0]
    kc = np.empty((n, d_idx // 2), np.uint8)
    ks = np.empty((n, d_idx // 16), np.uint8)
    _load().orc_project_ikeys(lcp, lsp, n, d_lat, wcp, wsp, d_idx, kc.ctypes.data, ks.ctypes.data)
    return kc, ks


# ---------------------------------------------------------------- indexer
def index_scores(kcodes, kscales, qcodes, qscales, w, ids=None, n=None):
    """exact scores S[t] of entry ids[t] (or entries 0..n-1) for one query.
    qcodes [H, d/2], qscales [H, d/16], w [H] float32."""
    kcodes, kcp = _c(kcodes, np.uint8)
    kscales, ksp = _c(kscales, np.uint8)
    qcodes, qcp = _c(qcodes, np.uint8)
    qscales, qsp = _c(qscales, np.uint8)
    w, wp = _c(w, np.float32)
    H, d = qcodes.shape[0], qcodes.shape[1] * 2
    if ids is not None:
        ids, idp = _c(ids, np.int32)
        n = ids.shape[0]
    else:
        idp = None
    S = np.empty(n, np.float64)
    _load().orc_index_scores(kcp, ksp, d, idp, n, qcp, qsp, wp, H, S.ctypes.data)
    return S


def topk(S, k, ids=None):
    """the k best ids by (S desc, id asc), written in ascending id order, -1 padded"""
    S, sp = _c(S, np.float64)
    if ids is not None:
        ids, idp = _c(ids, np.int32)
    else:
        idp = None
    out = np.empty(k, np.int32)
    _load().orc_topk(sp, idp, S.shape[0], k, out.ctypes.data)
    return out


def hsi_pool(S, block_size, n_blocks):
    S, sp = _c(S, np.float64)
    pool = np.empty(n_blocks * block_size, np.int32)
    _load().orc_hsi_pool(sp, S.shape[0], block_size, n_blocks, pool.ctypes.data)
    return pool


# ---------------------------------------------------------------- attention
def sparse_attention(q, idx, lat_codes, lat_scales, win, scale=SCALE):
    """q bf16 [H, 512]; idx int32 [k]; win bf16 [n_win, 512] -> (o float64 [H,512], lse [H])"""
    q, qp = _c(q, np.uint16)
    idx, ip = _c(idx, np.int32)
    lat_codes, lcp = _c(lat_codes, np.uint8)
    lat_scales, lsp = _c(lat_scales, np.uint8)
    win, wp = _c(win, np.uint16)
    H, d = q.shape
    out = np.empty((H, d), np.float64)
    lse = np.empty(H, np.float64)
    _load().orc_sparse_attention(qp, H, d, ip, idx.shape[0], lcp, lsp, wp, win.shape[0], float(scale),
                                 out.ctypes.data, lse.ctypes.data)
    return out, lse


def dense_attention(q, n_elig, lat_codes, lat_scales, win, scale=SCALE):
    q, qp = _c(q, np.uint16)
    lat_codes, lcp = _c(lat_codes, np.uint8)
    lat_scales, lsp = _c(lat_scales, np.uint8)
    win, wp = _c(win, np.uint16)
    H, d = q.shape
    out = np.empty((H, d), np.float64)
    lse = np.empty(H, np.float64)
    _load().orc_dense_attention(qp, H, d, int(n_elig), lcp, lsp, wp, win.shape[0], float(scale),
                                out.ctypes.data, lse.ctypes.data)
    return out, lse


# ---------------------------------------------------------------- one sequence of a workload
def sequence_cache(wl, b):
    """cache planes of sequence b of workload wl (whole context): merged 2:1
    (ratio 2) or one entry per position (ratio 1, the decoder's); indexer keys
    from the raw rows, or projected from the entries when wl.ikey_proj"""
    if wl.ratio == 1:
        lc, ls = cache_write_r1(wl.h(b, 0, wl.T))
        kc, ks = quantize_rows(synth_bf16_to_f32(wl.kraw(b, 0, wl.n_entries))) if not wl.ikey_proj else (None, None)
    else:
        w0, w1 = wl.merge_weights()
        lc, ls, kc, ks = cache_write(wl.h(b, 0, wl.T), w0, w1, wl.kraw(b, 0, wl.n_entries))
    if wl.ikey_proj:
        wc, ws = quantize_rows(wl.w_ik())
        kc, ks = project_ikeys(lc, ls, wc, ws)
    return lc, ls, kc, ks


def synth_bf16_to_f32(a):
    """bf16 bit patterns -> float32 (exact)"""
    return (np.ascontiguousarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)


def run_sequence(wl, b, cache=None, queries=None, layers=None, want_out=True):
    """Walk the layers of workload wl for sequence b (Full -> Reindex -> Reuse),
    exactly as the pages describe the three modes ([P1] §2.3.2, §2.3.4), plus
    window-only ("swa") layers.
    queries: which query slots (default all); layers: which layer indices.
    Returns dict with per-layer idx [nq, k], pool [nq, P] (Full with pool),
    out [nq, H, 512], lse [nq, H]."""
    lc, ls, kc, ks = cache if cache is not None else sequence_cache(wl, b)
    qpos = wl.q_positions()
    queries = list(range(wl.n_q)) if queries is None else list(queries)
    layers = list(range(len(wl.layers))) if layers is None else list(layers)
    first, count = wl.swa_range()
    res = {"idx": {}, "pool": {}, "out": {}, "lse": {}}
    prev_idx = None
    pool = None
    for l in range(max(layers) + 1):
        mode = wl.layers[l]
        need_out = want_out and l in layers
        idx_l = np.empty((len(queries), wl.k), np.int32)
        if mode in ("full", "reindex"):
            iq = wl.iq(l, b)
            wh = wl.w_head(l, b)
            qc, qs = quantize_rows(iq[queries])
            if mode == "full" and wl.pool_blocks:
                pool = np.empty((len(queries), wl.pool_len), np.int32)
            for t, qi in enumerate(queries):
                ne = n_elig(qpos[qi], wl.ratio)
                if mode == "full":
                    S = index_scores(kc, ks, qc[t], qs[t], wh[qi], n=ne)
                    idx_l[t] = topk(S, wl.k)
                    if wl.pool_blocks and wl.pool_block_size:
                        pool[t] = hsi_pool(S, wl.pool_block_size, wl.pool_blocks)
                    elif wl.pool_blocks:
                        # the other reading of the candidate pool: the best pool_blocks entries
                        pool[t] = topk(S, wl.pool_blocks)
                else:
                    S = index_scores(kc, ks, qc[t], qs[t], wh[qi], ids=pool[t])
                    idx_l[t] = topk(S, wl.k, ids=pool[t])
            if mode == "full" and wl.pool_blocks:
                res["pool"][l] = pool
        elif mode == "swa":
            # a sliding-window layer ([P1] §2.3.3: the encoder's first two layers):
            # no global entry is selected, and the latest indices stay as they are
            idx_l = np.empty((len(queries), 0), np.int32)
        else:  # reuse: the latest indices, unchanged
            idx_l[:] = prev_idx
        if mode != "swa":
            prev_idx = idx_l
        res["idx"][l] = idx_l
        if need_out:
            win_all = wl.window(l, b)
            o = np.empty((len(queries), wl.H, 512), np.float64)
            lse = np.empty((len(queries), wl.H), np.float64)
            for t, qi in enumerate(queries):
                p = int(qpos[qi])
                lo = max(0, p - 127)
                win = win_all[lo - first:p - first + 1]
                o[t], lse[t] = sparse_attention(wl.q(l, b, qi, 1)[0], idx_l[t], lc, ls, win)
            res["out"][l] = o
            res["lse"][l] = lse
    return res

"""CSA2 sparse-attention decode over an FP4 global KV cache, GB300 (sm_103a).

Thin binding over the C ABI of ``libcsa2.so`` (declared in include/csa2.h):
argument marshalling only.  Every step runs in the library's CUDA kernels;
PyTorch supplies device memory and the current stream.  There is no CPU
fallback: if the library is not built, every call raises.

Entry points (same names as the C ABI):
    csa2_cache_write, csa2_quantize_fp4, csa2_indexer_topk, csa2_reindex, csa2_reindex_f32,
    csa2_sparse_attn, csa2_workspace_size, csa2_poll_error, csa2_selftest_wait_timeout
plus ``Cache``, which owns the four cache planes as torch tensors.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_TIMEOUT = 0, 1, 2, 3, 4, 5
FULL, REINDEX, REUSE = 0, 1, 2
OP_INDEXER_TOPK, OP_REINDEX, OP_SPARSE_ATTN = 1, 2, 3
D_LAT = 512


class Csa2Error(RuntimeError):
    def __init__(self, status, fn):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (fn, _status_string(status), status))


class _CacheStruct(ctypes.Structure):
    _fields_ = [("lat_codes", ctypes.c_void_p), ("lat_scales", ctypes.c_void_p),
                ("ikey_codes", ctypes.c_void_p), ("ikey_scales", ctypes.c_void_p),
                ("batch", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("d_lat", ctypes.c_int32), ("d_idx", ctypes.c_int32), ("ratio", ctypes.c_int32)]


_lib = None
EXPORTS = ("csa2_cache_write", "csa2_quantize_fp4", "csa2_indexer_topk", "csa2_reindex", "csa2_sparse_attn",
           "csa2_workspace_size", "csa2_status_string", "csa2_abi_version", "csa2_launch_count",
           "csa2_reindex_noalloc", "csa2_reindex_f32", "csa2_poll_error", "csa2_selftest_wait_timeout",
           "csa2_cache_write_projected")


def load(path=None):
    """Load libcsa2.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("libcsa2.so is not built (%s); run __graft_entry__.build()" % p)
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    cp = ctypes.POINTER(_CacheStruct)
    lib.csa2_cache_write.argtypes = [cp, vp, i64, i32, vp, vp, vp, vp]
    lib.csa2_cache_write_projected.argtypes = [cp, vp, i64, i32, vp, vp, vp, vp, vp]
    lib.csa2_cache_write_projected.restype = ctypes.c_int
    lib.csa2_quantize_fp4.argtypes = [vp, i64, i32, vp, vp, vp]
    lib.csa2_indexer_topk.argtypes = [cp, vp, vp, vp, i32, vp, i32, i32, vp, i32, i32, vp, vp, sz, vp]
    lib.csa2_reindex.argtypes = [i32, cp, vp, vp, vp, i32, i32, vp, i32, vp, i32, vp, vp, sz, vp]
    lib.csa2_reindex_f32.argtypes = [cp, vp, vp, i32, i32, vp, i32, i32, vp, vp, sz, vp]
    lib.csa2_sparse_attn.argtypes = [cp, vp, i32, i32, vp, vp, i32, vp, i64, i32, ctypes.c_float, vp, vp, vp, sz, vp]
    lib.csa2_reindex_noalloc.argtypes = [cp, vp, vp, vp, i32, i32, vp, i32, i32, vp, vp]
    lib.csa2_reindex_noalloc.restype = ctypes.c_int
    lib.csa2_poll_error.argtypes = [vp, sz, vp]
    lib.csa2_poll_error.restype = ctypes.c_int
    lib.csa2_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp, sz, vp]
    lib.csa2_selftest_wait_timeout.restype = ctypes.c_int
    lib.csa2_workspace_size.argtypes = [i32, i32, i32, i32, i32, i64]
    lib.csa2_workspace_size.restype = sz
    lib.csa2_status_string.argtypes = [ctypes.c_int]
    lib.csa2_status_string.restype = ctypes.c_char_p
    lib.csa2_abi_version.restype = i32
    lib.csa2_launch_count.restype = i64
    for name in ("csa2_cache_write", "csa2_quantize_fp4", "csa2_indexer_topk", "csa2_reindex", "csa2_reindex_f32",
                 "csa2_sparse_attn"):
        getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _status_string(s):
    try:
        return load().csa2_status_string(s).decode()
    except Exception:
        return "status %d" % s


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, fn):
    if status != OK:
        raise Csa2Error(status, fn)


class Cache:
    """The four planes of the FP4 global KV cache (device tensors, uint8); ratio
    raw positions per entry (2: an encoder copy, 1: the decoder's)."""

    def __init__(self, batch, capacity, d_idx=128, device="cuda", ratio=2):
        self.batch, self.capacity, self.d_idx, self.ratio = batch, capacity, d_idx, ratio
        self.lat_codes = torch.zeros((batch, capacity, D_LAT // 2), dtype=torch.uint8, device=device)
        self.lat_scales = torch.zeros((batch, capacity, D_LAT // 16), dtype=torch.uint8, device=device)
        self.ikey_codes = torch.zeros((batch, capacity, d_idx // 2), dtype=torch.uint8, device=device)
        self.ikey_scales = torch.zeros((batch, capacity, d_idx // 16), dtype=torch.uint8, device=device)

    def struct(self):
        return _CacheStruct(self.lat_codes.data_ptr(), self.lat_scales.data_ptr(), self.ikey_codes.data_ptr(),
                            self.ikey_scales.data_ptr(), self.batch, self.capacity, D_LAT, self.d_idx,
                            getattr(self, "ratio", 2))

    def nbytes(self):
        return sum(t.numel() for t in (self.lat_codes, self.lat_scales, self.ikey_codes, self.ikey_scales))


def csa2_launch_count():
    return load().csa2_launch_count()


def csa2_workspace_size(op, batch, n_q, n_heads, k, capacity):
    return load().csa2_workspace_size(op, batch, n_q, n_heads, k, capacity)


def workspace(op, batch, n_q, n_heads, k, capacity, device="cuda"):
    """a workspace for the operation, its error word cleared"""
    n = csa2_workspace_size(op, batch, n_q, n_heads, k, capacity)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=device)
    ws[:16].zero_()
    return ws


def csa2_poll_error(ws, stream=None):
    """reads and clears the error word of a workspace: OK, or ERR_TIMEOUT if a
    kernel that used it gave up on a bounded wait (synchronises the stream)"""
    return load().csa2_poll_error(_ptr(ws), ws.numel(), _stream(stream))


def csa2_selftest_wait_timeout(max_polls, ws, stream=None):
    """a kernel waits on a barrier nothing signals, with at most max_polls polls,
    gives up and records it in ws's error word"""
    _check(load().csa2_selftest_wait_timeout(int(max_polls), _ptr(ws), ws.numel(), _stream(stream)),
           "csa2_selftest_wait_timeout")


def csa2_cache_write(cache, h, pos0, w0, w1, ikey_raw=None, stream=None):
    """h: bf16 [B, n_pos, 512] (as torch.bfloat16 or int16 bits); w0/w1 fp32 [512];
    ikey_raw bf16 [B, n_pos/2, d_idx] or None."""
    c = cache.struct()
    st = load().csa2_cache_write(ctypes.byref(c), _ptr(h), int(pos0), int(h.shape[1]), _ptr(w0), _ptr(w1),
                                 _ptr(ikey_raw), _stream(stream))
    _check(st, "csa2_cache_write")


def csa2_cache_write_projected(cache, h, pos0, w0, w1, wik_codes, wik_scales, stream=None):
    """as csa2_cache_write, with the indexer keys projected from the entries:
    wik_codes uint8 [d_idx, 256], wik_scales uint8 [d_idx, 32] (FP4 W)"""
    c = cache.struct()
    st = load().csa2_cache_write_projected(ctypes.byref(c), _ptr(h), int(pos0), int(h.shape[1]), _ptr(w0), _ptr(w1),
                                           _ptr(wik_codes), _ptr(wik_scales), _stream(stream))
    _check(st, "csa2_cache_write_projected")


def csa2_quantize_fp4(x, codes=None, scales=None, stream=None):
    """fp32 [..., d] -> (codes uint8 [..., d/2], scales uint8 [..., d/16])"""
    d = x.shape[-1]
    if codes is None:
        codes = torch.empty(x.shape[:-1] + (d // 2,), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (d // 16,), dtype=torch.uint8, device=x.device)
    st = load().csa2_quantize_fp4(_ptr(x), x.numel() // d, d, _ptr(codes), _ptr(scales), _stream(stream))
    _check(st, "csa2_quantize_fp4")
    return codes, scales


def csa2_indexer_topk(cache, iq_codes, iq_scales, w_head, q_pos, k, pool_blocks=0, pool_block_size=8,
                      idx_out=None, pool_out=None, ws=None, stream=None):
    """Full-mode indexer + top-k (+ HSI pool).  iq_codes [B, n_q, H_I, d_idx/2] ...
    Returns (idx [B, n_q, k] int32, pool [B, n_q, P] int32 or None)."""
    B, n_q, H = iq_codes.shape[0], iq_codes.shape[1], iq_codes.shape[2]
    dev = iq_codes.device
    if idx_out is None:
        idx_out = torch.empty((B, n_q, k), dtype=torch.int32, device=dev)
    if pool_blocks and pool_out is None:
        P = pool_blocks * pool_block_size if pool_block_size else pool_blocks   # 0: the pure pool
        pool_out = torch.empty((B, n_q, P), dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(OP_INDEXER_TOPK, cache.batch, n_q, H, k, cache.capacity, dev)
    c = cache.struct()
    st = load().csa2_indexer_topk(ctypes.byref(c), _ptr(iq_codes), _ptr(iq_scales), _ptr(w_head), n_q, _ptr(q_pos),
                                  H, k, _ptr(idx_out), pool_blocks, pool_block_size,
                                  _ptr(pool_out) if pool_blocks else None, _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "csa2_indexer_topk")
    return idx_out, (pool_out if pool_blocks else None)


def csa2_reindex(mode, cache, k, iq_codes=None, iq_scales=None, w_head=None, pool=None, prev_idx=None,
                 idx_out=None, ws=None, stream=None, n_q=None):
    """mode REINDEX: top-k inside the pool with this layer's indexer queries;
    mode REUSE: copy prev_idx."""
    if n_q is None:
        n_q = (iq_codes if iq_codes is not None else prev_idx).shape[1]
    dev = (iq_codes if iq_codes is not None else prev_idx).device
    if idx_out is None:
        idx_out = torch.empty((cache.batch, n_q, k), dtype=torch.int32, device=dev)
    H = iq_codes.shape[2] if iq_codes is not None else 0
    pool_len = pool.shape[-1] if pool is not None else 0
    if mode == REINDEX and ws is None:
        ws = workspace(OP_REINDEX, cache.batch, n_q, H, k, pool_len, dev)
    c = cache.struct()
    st = load().csa2_reindex(mode, ctypes.byref(c), _ptr(iq_codes), _ptr(iq_scales), _ptr(w_head), n_q, H,
                             _ptr(pool), pool_len, _ptr(prev_idx), k, _ptr(idx_out), _ptr(ws),
                             ws.numel() if ws is not None else 0, _stream(stream))
    _check(st, "csa2_reindex")
    return idx_out


def csa2_reindex_f32(cache, k, iq, w_head, pool, idx_out=None, ws=None, stream=None):
    """Reindex from fp32 indexer queries iq [B, n_q, H, d_idx]: the query
    quantisation runs inside the Reindex kernels (same results as
    csa2_quantize_fp4 followed by csa2_reindex)."""
    B, n_q, H = iq.shape[0], iq.shape[1], iq.shape[2]
    if idx_out is None:
        idx_out = torch.empty((B, n_q, k), dtype=torch.int32, device=iq.device)
    pool_len = pool.shape[-1]
    if ws is None:
        ws = workspace(OP_REINDEX, cache.batch, n_q, H, k, pool_len, iq.device)
    c = cache.struct()
    st = load().csa2_reindex_f32(ctypes.byref(c), _ptr(iq), _ptr(w_head), n_q, H, _ptr(pool), pool_len, k,
                                 _ptr(idx_out), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "csa2_reindex_f32")
    return idx_out


def csa2_reindex_noalloc(cache, k, iq_codes, iq_scales, w_head, pool, idx_out=None, stream=None):
    """Reindex with the library's built-in scratch instead of a workspace (for
    callers that cannot allocate device memory; see include/csa2.h)."""
    B, n_q, H = iq_codes.shape[0], iq_codes.shape[1], iq_codes.shape[2]
    if idx_out is None:
        idx_out = torch.empty((B, n_q, k), dtype=torch.int32, device=iq_codes.device)
    c = cache.struct()
    st = load().csa2_reindex_noalloc(ctypes.byref(c), _ptr(iq_codes), _ptr(iq_scales), _ptr(w_head), n_q, H,
                                     _ptr(pool), pool.shape[-1], k, _ptr(idx_out), _stream(stream))
    _check(st, "csa2_reindex_noalloc")
    return idx_out


def csa2_sparse_attn(cache, q, q_pos, idx, swa, swa_pos0, scale=D_LAT ** -0.5, out=None, lse=None,
                     want_lse=False, ws=None, stream=None):
    """q bf16 [B, n_q, H, 512]; idx int32 [B, n_q, k]; swa bf16 [B, swa_len, 512].
    Returns (out fp32 [B, n_q, H, 512], lse fp32 [B, n_q, H] or None)."""
    B, n_q, H = q.shape[0], q.shape[1], q.shape[2]
    k = idx.shape[-1] if idx is not None else 0
    if out is None:
        out = torch.empty((B, n_q, H, D_LAT), dtype=torch.float32, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, n_q, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(OP_SPARSE_ATTN, cache.batch, n_q, H, k, cache.capacity, q.device)
    c = cache.struct()
    st = load().csa2_sparse_attn(ctypes.byref(c), _ptr(q), n_q, H, _ptr(q_pos), _ptr(idx), k, _ptr(swa),
                                 int(swa_pos0), int(swa.shape[1]) if swa is not None else 0, float(scale), _ptr(out),
                                 _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "csa2_sparse_attn")
    return out, lse

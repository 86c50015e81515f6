"""A CSA2 decode step over the layers that share one global KV.

Layer modes follow "DeepSeek-v4.1 Flash: KVキャッシュ圧縮の限界を押し広げる" §2.3.2
and §2.3.4: a Full layer scores every eligible entry, keeps its top-k and (with
HSI) a block-max candidate pool; a Reindex layer re-scores only the pool with
its own indexer queries; a Reuse layer takes the latest indices unchanged.
Every layer computes its own attention over its indices plus its window.  A
window-only ("swa") layer, like the first two encoder layers of §2.3.3,
attends to its window alone.

``DecodeStep`` owns the device buffers of one workload (one global-KV copy
and the layers that read it) and enqueues a whole step on a stream
(optionally captured as one CUDA graph); ``ScheduleStep`` chains several of
them, one per copy, into one step of a whole model.  Each call they make is a
C-ABI entry point of libcsa2; this module only sequences them.
"""
import torch

from . import (FULL, REINDEX, REUSE, OP_INDEXER_TOPK, OP_REINDEX, OP_SPARSE_ATTN, Cache, csa2_cache_write,
               csa2_cache_write_projected, csa2_indexer_topk, csa2_quantize_fp4, csa2_reindex_f32, csa2_sparse_attn, workspace)

_MODES = {"full": FULL, "reindex": REINDEX, "reuse": REUSE}


class _Graphed:
    """capture()/run() over the subclass's enqueue()"""
    graph = None

    def capture(self):
        """record one step as a CUDA graph (replayed by run())"""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.enqueue(s)          # warm-up outside the graph
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.enqueue()
        self.graph = g
        return g

    def run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.enqueue()


class DecodeStep(_Graphed):
    """Buffers and launch sequence for one step of a layer schedule.

    layers: tuple of "full" / "reindex" / "reuse"; B sequences, n_q queries
    each at raw positions q_pos; the cache holds `capacity` entries per
    sequence.  Per layer l the step reads iq[l] (fp32, quantised on device),
    w_head[l], q[l] and win[l] and writes out[l] (+ lse[l]); a Full or Reindex
    layer writes idx[l], a Reuse layer reads layer_idx(l) in place."""

    def __init__(self, B, capacity, n_q, layers, H=64, H_I=8, d_I=128, k=512, pool_blocks=0, pool_block_size=8,
                 swa_len=128, chunk_pos=0, device="cuda", want_lse=False, ratio=2):
        self.B, self.capacity, self.n_q, self.layers = B, capacity, n_q, tuple(layers)
        self.H, self.H_I, self.d_I, self.k = H, H_I, d_I, k
        self.pool_blocks, self.bs = pool_blocks, pool_block_size
        self.swa_len, self.chunk_pos = swa_len, chunk_pos
        self.dev = device
        L = len(self.layers)
        f32, bf16, i32 = torch.float32, torch.bfloat16, torch.int32
        self.cache = Cache(B, capacity, d_I, device, ratio=ratio)
        # step inputs
        n_idx = sum(m in ("full", "reindex") for m in self.layers)
        self.iq = torch.zeros((max(n_idx, 1), B, n_q, H_I, d_I), dtype=f32, device=device)
        self.w_head = torch.zeros((max(n_idx, 1), B, n_q, H_I), dtype=f32, device=device)
        self.q = torch.zeros((L, B, n_q, H, 512), dtype=bf16, device=device)
        self.win = torch.zeros((L, B, swa_len, 512), dtype=bf16, device=device)
        self.q_pos = torch.zeros((B, n_q), dtype=torch.int64, device=device)
        self.swa_pos0 = 0
        # chunked prefill: hidden states (and raw indexer keys) written in the step
        self.chunk_len = 0
        self.h_chunk = None
        self.kraw_chunk = None
        self.w0 = torch.zeros(512, dtype=f32, device=device)
        self.w1 = torch.zeros(512, dtype=f32, device=device)
        # FP4 indexer-key projection W (codes, scales): when set, the cache
        # writes project the indexer keys from the entries
        self.wik_codes = self.wik_scales = None
        # outputs / intermediates
        self.iq_codes = torch.zeros((B, n_q, H_I, d_I // 2), dtype=torch.uint8, device=device)
        self.iq_scales = torch.zeros((B, n_q, H_I, d_I // 16), dtype=torch.uint8, device=device)
        self.idx = torch.full((L, B, n_q, k), -1, dtype=i32, device=device)
        # pool_block_size 0: the pool is the pool_blocks best entries
        self.pool_len = (pool_blocks * pool_block_size if pool_block_size else pool_blocks) if pool_blocks else 0
        self.pool = torch.full((B, n_q, self.pool_len), -1, dtype=i32, device=device) if pool_blocks else None
        self.out = torch.zeros((L, B, n_q, H, 512), dtype=f32, device=device)
        self.lse = torch.zeros((L, B, n_q, H), dtype=f32, device=device) if want_lse else None
        self.ws_full = workspace(OP_INDEXER_TOPK, B, n_q, H_I, k, capacity, device)
        self.ws_re = (workspace(OP_REINDEX, B, n_q, H_I, k, self.pool_len, device)
                      if "reindex" in self.layers else None)
        self.ws_attn = workspace(OP_SPARSE_ATTN, B, n_q, H, k, capacity, device)
        self.graph = None

    def set_chunk(self, chunk_len, w0, w1):
        """chunked prefill: the step first writes `chunk_len` raw positions
        starting at chunk_pos into the cache"""
        self.chunk_len = chunk_len
        self.h_chunk = torch.zeros((self.B, chunk_len, 512), dtype=torch.bfloat16, device=self.dev)
        self.kraw_chunk = torch.zeros((self.B, chunk_len // self.cache.ratio, self.d_I), dtype=torch.bfloat16,
                                      device=self.dev)
        self.w0.copy_(w0)
        self.w1.copy_(w1)

    def enqueue(self, stream=None):
        """all layers of one step, in order, on `stream` (default: current)"""
        if self.chunk_len and self.wik_codes is not None:
            csa2_cache_write_projected(self.cache, self.h_chunk, self.chunk_pos, self.w0, self.w1, self.wik_codes,
                                       self.wik_scales, stream=stream)
        elif self.chunk_len:
            csa2_cache_write(self.cache, self.h_chunk, self.chunk_pos, self.w0, self.w1, self.kraw_chunk,
                             stream=stream)
        t = 0
        for l, mode in enumerate(self.layers):
            idx_l = self.layer_idx(l)
            if mode in ("reuse", "swa"):
                pass                 # Reuse: the latest indices, read in place; SWA: no indices
            elif mode == "full":
                csa2_quantize_fp4(self.iq[t], self.iq_codes, self.iq_scales, stream=stream)
                csa2_indexer_topk(self.cache, self.iq_codes, self.iq_scales, self.w_head[t], self.q_pos, self.k,
                                  self.pool_blocks, self.bs, idx_out=idx_l, pool_out=self.pool, ws=self.ws_full,
                                  stream=stream)
                t += 1
            else:
                # the Reindex kernels quantise this layer's queries themselves
                csa2_reindex_f32(self.cache, self.k, self.iq[t], self.w_head[t], self.pool, idx_out=idx_l,
                                 ws=self.ws_re, stream=stream)
                t += 1
            csa2_sparse_attn(self.cache, self.q[l], self.q_pos, idx_l, self.win[l], self.swa_pos0, out=self.out[l],
                             lse=None if self.lse is None else self.lse[l], ws=self.ws_attn, stream=stream)

    def layer_idx(self, l):
        """the index list layer l attends with: its own for a Full or Reindex
        layer; for a Reuse layer the latest one before it, read in place
        ("DeepSeek-v4.1 Flash" §2.3.2: Reuse takes the latest indices unchanged);
        none (k = 0) for a window-only layer.  Only the layers that compute
        indices write their slot of self.idx."""
        if self.layers[l] == "swa":
            return self.idx[l][..., :0]
        src = l
        while src > 0 and self.layers[src] in ("reuse", "swa"):
            src -= 1
        return self.idx[src]

    def twin(self):
        """a second step over the same cache, intermediates and workspaces with
        its own inputs (iq, w_head, q, win, q_pos) and outputs (idx, out, lse),
        so that one step's copies can overlap the other's compute; the two must
        not run concurrently on the device"""
        t = object.__new__(DecodeStep)
        t.__dict__.update(self.__dict__)
        for name in ("iq", "w_head", "q", "win", "q_pos", "idx", "out", "lse", "h_chunk", "kraw_chunk"):
            if getattr(self, name) is not None:
                setattr(t, name, getattr(self, name).clone())
        t.graph = None
        return t


class ScheduleStep(_Graphed):
    """one step of a model whose layers are split over several global-KV copies:
    the segments (DecodeSteps, one per copy) run in order on one stream"""

    def __init__(self, segments):
        self.segments = list(segments)
        self.graph = None

    @property
    def layers(self):
        return tuple(m for s in self.segments for m in s.layers)

    def enqueue(self, stream=None):
        for s in self.segments:
            s.enqueue(stream)

    def twin(self):
        """as DecodeStep.twin, segment by segment"""
        return ScheduleStep([s.twin() for s in self.segments])

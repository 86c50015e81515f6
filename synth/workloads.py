"""The five synthetic CSA2 workloads and the recipe that draws their inputs.

Sizes follow the statement of the problem for CSA2 decode in "DeepSeek-V4.1
Flash: KVキャッシュ圧縮の限界を押し広げる" (section 2.3, CSA2; window 128, top-k 512,
512-dim shared latent, 2:1 encoder merge) and the spec table of the
ai.freelance-job.com summary (KV latent 512, window 128).

Distributions (all seeded by the workload's index, one stream per tensor):
  h        encoder hidden states   bf16  N(0,1)      [B, T, 512]
  w0, w1   channel-wise merge      f32   U(0.3,0.7)  [512]
  kraw     indexer-key rows        bf16  N(0,1)      [B, T/2, d_I]
  iq[l]    indexer queries         f32   N(0,1)      [B, n_q, H_I, d_I]
  w[l]     indexer head weights    f32   U(0,1)      [B, n_q, H_I]
  q[l]     attention queries       bf16  N(0,1)      [B, n_q, H, 512]
  win[l]   window rows of layer l  bf16  N(0,1)      [B, 128, 512]  (l >= 1; layer 0 reads h)
  w_ik     indexer-key projection  f32   N(0,1/512)  [d_I, 512]  (workloads whose keys are projected)
Layer modes: "full", "reindex", "reuse" (CSA2) and "swa" (window-only attention).
Element i of a tensor is sample i of its stream, so one sequence's slice is
drawn on its own.  Nothing in here merges, quantises or scores.
"""
from dataclasses import dataclass, field

import numpy as np

from . import normal_bf16, normal_f32, uniform_f32

D_LAT = 512
WINDOW = 128

# stream ids
S_H, S_W0, S_W1, S_KRAW, S_WIK = 1, 2, 3, 4, 5
S_IQ, S_WH, S_Q, S_WIN = 1000, 2000, 3000, 4000


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int                 # sequences
    T: int                 # raw positions held in the cache (prefix + chunk)
    H_I: int               # indexer heads
    d_I: int               # indexer head dim
    k: int                 # top-k
    H: int                 # attention heads
    layers: tuple          # per layer: "full" | "reindex" | "reuse"
    pool_blocks: int = 0   # HSI blocks kept by the Full layer (0 = no pool)
    pool_block_size: int = 8   # 0: the pool is the pool_blocks best entries (no blocks)
    chunk: int = 0         # >0: chunked prefill, the last `chunk` positions are queries and are written in the step
    ratio: int = 2         # raw positions per global entry: 2 (encoder merge) or 1 (the decoder's per-position cache)
    ikey_proj: bool = False  # indexer keys projected from the entries (w_ik) instead of drawn rows
    new_entry: bool = False  # decode: the step itself writes the newest entry (its last `ratio` raw positions)

    @property
    def seed(self):
        return self.index

    @property
    def n_entries(self):
        return self.T // self.ratio

    @property
    def pool_len(self):
        """slots of the Full layer's candidate pool"""
        if not self.pool_blocks:
            return 0
        return self.pool_blocks * self.pool_block_size if self.pool_block_size else self.pool_blocks

    @property
    def prefix(self):
        return self.T - self.chunk

    @property
    def n_q(self):
        return self.chunk if self.chunk else 1

    def q_positions(self):
        """raw positions of the queries of one sequence"""
        if self.chunk:
            return np.arange(self.prefix, self.T, dtype=np.int64)
        return np.array([self.T - 1], dtype=np.int64)

    def swa_range(self):
        """(first raw position, count) of the window rows the queries read"""
        first = max(0, int(self.q_positions()[0]) - (WINDOW - 1))
        return first, self.T - first

    # ---- input tensors (numpy, host) ----
    def merge_weights(self):
        return (uniform_f32(self.seed, S_W0, (D_LAT,), 0.3, 0.7),
                uniform_f32(self.seed, S_W1, (D_LAT,), 0.3, 0.7))

    def h(self, b, pos0, n_pos):
        """bf16 hidden states of sequence b, raw positions [pos0, pos0+n_pos)"""
        return normal_bf16(self.seed, S_H, (n_pos, D_LAT), offset=(b * self.T + pos0) * D_LAT)

    def kraw(self, b, e0, n):
        """bf16 raw indexer-key rows of sequence b, entries [e0, e0+n)"""
        return normal_bf16(self.seed, S_KRAW, (n, self.d_I), offset=(b * self.n_entries + e0) * self.d_I)

    def w_ik(self):
        """f32 [d_I, 512] N(0, 1/512): the projection of an entry to its indexer key"""
        return (normal_f32(self.seed, S_WIK, (self.d_I, D_LAT)) * np.float32(1.0 / np.sqrt(D_LAT))).astype(np.float32)

    def iq(self, layer, b):
        n = self.n_q * self.H_I * self.d_I
        return normal_f32(self.seed, S_IQ + layer, (self.n_q, self.H_I, self.d_I), offset=b * n)

    def w_head(self, layer, b):
        n = self.n_q * self.H_I
        return uniform_f32(self.seed, S_WH + layer, (self.n_q, self.H_I), 0.0, 1.0, offset=b * n)

    def q(self, layer, b, q0=0, nq=None):
        nq = self.n_q if nq is None else nq
        per_q = self.H * D_LAT
        return normal_bf16(self.seed, S_Q + layer, (nq, self.H, D_LAT), offset=(b * self.n_q + q0) * per_q)

    def window(self, layer, b):
        """bf16 window rows [swa_count, 512] of sequence b for this layer"""
        first, count = self.swa_range()
        if layer == 0:
            return self.h(b, first, count)
        return normal_bf16(self.seed, S_WIN + layer, (count, D_LAT), offset=b * count * D_LAT)


WORKLOADS = [
    Workload(0, "tiny-2k-b1", B=1, T=2048, H_I=4, d_I=64, k=64, H=16, layers=("full",)),
    Workload(1, "decode-32k-b16", B=16, T=32768, H_I=8, d_I=128, k=512, H=64, layers=("full",)),
    Workload(2, "decode-128k-b64-20L", B=64, T=131072, H_I=8, d_I=128, k=512, H=64,
             layers=("full",) + ("reindex",) * 9 + ("reuse",) * 10, pool_blocks=256, pool_block_size=8),
    Workload(3, "decode-1m-b4", B=4, T=1048576, H_I=8, d_I=128, k=512, H=64, layers=("full",)),
    Workload(4, "prefill-chunk-8k-after-120k", B=1, T=131072, H_I=8, d_I=128, k=512, H=64,
             layers=("full",), chunk=8192),
]

# per-entry bytes of one cache copy: 256 B latent codes + 32 B scales + 64 B indexer-key codes + 8 B scales
ENTRY_BYTES = 256 + 32 + 64 + 8


@dataclass(frozen=True)
class Schedule:
    """The 40 layers of the CED model ("DeepSeek-v4.1 Flash" §2.3.3) as segments
    of consecutive layers, each over its own global-KV copy:

      encoder copy 0: SWA, SWA, Full, Reuse x5   (the two SWA layers read no global entry)
      encoder copy 1: Full, Reuse x5
      encoder copy 2: Full, Reuse x5
      decoder copy:   Full (+HSI pool), Reuse x3, then 4 x [Reindex, Reuse x3]

    The encoder copies merge 2:1; the decoder copy keeps one entry per raw
    position and projects its indexer keys from the entries.  In a decode
    step every copy first receives its newest entry.  Each segment draws from
    its own seed, so the four copies hold different data."""
    name: str
    segments: tuple

    @property
    def B(self):
        return self.segments[0].B

    @property
    def T(self):
        return self.segments[0].T

    @property
    def layers(self):
        return tuple(m for s in self.segments for m in s.layers)

    def cache_bytes_per_token(self):
        """stored global-KV bytes per raw position, over every copy"""
        return sum(ENTRY_BYTES / s.ratio for s in self.segments)


def ced_schedule(name, B, T, index0=10, pool_blocks=256, pool_block_size=8):
    common = dict(B=B, T=T, H_I=8, d_I=128, k=512, H=64, new_entry=True)
    enc_block = ("full",) + ("reuse",) * 5
    dec = ("full",) + ("reuse",) * 3 + (("reindex",) + ("reuse",) * 3) * 4
    return Schedule(name, (
        Workload(index0, name + "/enc0", layers=("swa", "swa") + enc_block, **common),
        Workload(index0 + 1, name + "/enc1", layers=enc_block, **common),
        Workload(index0 + 2, name + "/enc2", layers=enc_block, **common),
        Workload(index0 + 3, name + "/dec", layers=dec, ratio=1, ikey_proj=True, pool_blocks=pool_blocks,
                 pool_block_size=pool_block_size, **common),
    ))


CED_40L = ced_schedule("decode-128k-b64-40L-ced", B=64, T=131072)


def scaled(w, **kw):
    """a copy of workload w with some sizes replaced (small parity cases)"""
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)


def scaled_schedule(sched, name=None, **kw):
    """a copy of a schedule with the same sizes replaced in every segment"""
    name = name or sched.name
    segs = []
    for s in sched.segments:
        d = dict(kw)
        d["name"] = name + "/" + s.name.split("/")[-1]
        segs.append(scaled(s, **d))
    return Schedule(name, tuple(segs))

"""Fill a DecodeStep with one of the seeded synthetic workloads.

Inputs are drawn on the host by the ``synth`` generator (the same bytes the
oracle draws), copied to the device, and the context is written into the cache
by the library's own cache-write kernel, one sequence at a time so that the
host staging buffer stays small.
"""
import numpy as np
import torch

from synth.workloads import D_LAT

from . import Cache, csa2_cache_write, csa2_cache_write_projected, csa2_quantize_fp4
from .decode import DecodeStep, ScheduleStep


def _bf16(a):
    """uint16 bit patterns (numpy) -> torch bfloat16 tensor (host)"""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def seq_view(cache, b):
    """a batch-1 Cache aliasing sequence b of `cache`"""
    v = Cache.__new__(Cache)
    v.batch, v.capacity, v.d_idx, v.ratio = 1, cache.capacity, cache.d_idx, cache.ratio
    v.lat_codes = cache.lat_codes[b:b + 1]
    v.lat_scales = cache.lat_scales[b:b + 1]
    v.ikey_codes = cache.ikey_codes[b:b + 1]
    v.ikey_scales = cache.ikey_scales[b:b + 1]
    return v


class HostInputs:
    """pinned host copies of one step's inputs (for the end-to-end timing).

    The per-step inputs are the queries of every layer (q, iq, w_head), the
    query positions and, for the sliding window, only the newest row of every
    (layer, sequence): the window is device-resident KV state to which a
    decode step appends one row, like the compressed cache itself."""

    def __init__(self, step):
        """pinned host buffers holding the step's own inputs: the values the
        device buffers of `step` hold now are copied out once, here, so every
        timed step moves and computes the real workload"""
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        self.names = ["iq", "w_head", "q", "q_pos"] + (["h_chunk"] if step.chunk_len else []) + \
            (["kraw_chunk"] if step.chunk_len and step.wik_codes is None else [])
        self.host = {n: pin(getattr(step, n)) for n in self.names}
        for n in self.names:
            self.host[n].copy_(getattr(step, n))
        self.win_new = pin(step.win[:, :, -1])
        self.win_new.copy_(step.win[:, :, -1])
        self.win_dev = {}
        self.out = pin(step.out)

    def copy_in(self, step):
        """enqueue this step's host -> device copies on the current stream (the
        newest window rows land in a contiguous device buffer, then in place)"""
        for n in self.names:
            getattr(step, n).copy_(self.host[n], non_blocking=True)
        key = id(step)
        if key not in self.win_dev:
            self.win_dev[key] = torch.empty(self.win_new.shape, dtype=self.win_new.dtype, device=step.win.device)
        self.win_dev[key].copy_(self.win_new, non_blocking=True)
        step.win[:, :, -1].copy_(self.win_dev[key])

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host.values()) + \
            self.win_new.numel() * self.win_new.element_size()

    def d2h_bytes(self):
        return self.out.numel() * self.out.element_size()


def build_step(wl, device="cuda", want_lse=False, seqs=None):
    """DecodeStep for workload wl with context, inputs and window rows loaded.
    seqs: restrict to these sequence ids (default all wl.B)."""
    seqs = list(range(wl.B)) if seqs is None else list(seqs)
    B = len(seqs)
    first, count = wl.swa_range()
    step = DecodeStep(B, wl.n_entries, wl.n_q, wl.layers, H=wl.H, H_I=wl.H_I, d_I=wl.d_I, k=wl.k,
                      pool_blocks=wl.pool_blocks, pool_block_size=wl.pool_block_size, swa_len=count,
                      chunk_pos=wl.prefix, device=device, want_lse=want_lse, ratio=wl.ratio)
    step.swa_pos0 = first
    w0, w1 = wl.merge_weights()
    w0_d = torch.from_numpy(w0).to(device)
    w1_d = torch.from_numpy(w1).to(device)
    if wl.chunk:
        step.set_chunk(wl.chunk, w0_d, w1_d)
    elif wl.new_entry:
        # a decode step writes its own newest entry: the last `ratio` raw positions
        step.chunk_pos = wl.T - wl.ratio
        step.set_chunk(wl.ratio, w0_d, w1_d)
    qpos = torch.from_numpy(wl.q_positions())
    step.q_pos.copy_(qpos[None, :].expand(B, -1))
    if wl.ikey_proj:
        # the indexer-key projection W, quantised to FP4 by the library's own quantiser
        wik = torch.from_numpy(wl.w_ik()).to(device)
        step.wik_codes, step.wik_scales = csa2_quantize_fp4(wik)
    for bi, b in enumerate(seqs):
        # context written once, outside the step
        n_ctx = step.chunk_pos if step.chunk_len else wl.T
        if n_ctx:
            h = _bf16(wl.h(b, 0, n_ctx))[None].to(device)
            if wl.ikey_proj:
                csa2_cache_write_projected(seq_view(step.cache, bi), h, 0, w0_d, w1_d, step.wik_codes,
                                           step.wik_scales)
            else:
                kr = wl.kraw(b, 0, n_ctx // wl.ratio)
                csa2_cache_write(seq_view(step.cache, bi), h, 0, w0_d, w1_d, _bf16(kr)[None].to(device))
        if step.chunk_len:
            p0, n = step.chunk_pos, step.chunk_len
            step.h_chunk[bi].copy_(_bf16(wl.h(b, p0, n)))
            if not wl.ikey_proj:
                step.kraw_chunk[bi].copy_(_bf16(wl.kraw(b, p0 // wl.ratio, n // wl.ratio)))
        t = 0
        for l, mode in enumerate(wl.layers):
            step.win[l, bi].copy_(_bf16(wl.window(l, b)))
            step.q[l, bi].copy_(_bf16(wl.q(l, b)))
            if mode in ("full", "reindex"):
                step.iq[t, bi].copy_(torch.from_numpy(wl.iq(l, b)))
                step.w_head[t, bi].copy_(torch.from_numpy(wl.w_head(l, b)))
                t += 1
    torch.cuda.synchronize()
    return step


def build_schedule(sched, device="cuda", want_lse=False, seqs=None):
    """ScheduleStep for a Schedule: one DecodeStep per global-KV copy, each
    with its context, inputs and window rows loaded"""
    return ScheduleStep([build_step(w, device, want_lse, seqs) for w in sched.segments])

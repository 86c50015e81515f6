"""The CED model's 40-layer decode step ("DeepSeek-v4.1 Flash" §2.3.3): four
global-KV copies, each written its newest entry inside the step, then the
layers that read it.  CUDA path vs the fp64 oracle, through the C ABI; the
same bar as the single-copy walks (cache bytes, indices and pools bit-exact,
attention rows within 2e-3 max relative error)."""
import numpy as np
import pytest
import torch

import oracle
from synth.workloads import CED_40L, scaled_schedule

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3


@pytest.fixture(scope="module")
def csa():
    import __graft_entry__
    __graft_entry__.build()
    import compressed_sparse_attention_decode_gb300 as m
    return m


def rel_err_rows(out, ref):
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return float((np.abs(out - ref).max(axis=-1) / den).max())


def check_segment(seg, wl, bi, b, layers=None, check_cache=True):
    ref_cache = oracle.sequence_cache(wl, b)
    if check_cache:
        got = (seg.cache.lat_codes, seg.cache.lat_scales, seg.cache.ikey_codes, seg.cache.ikey_scales)
        for name, g, w in zip(("lat_codes", "lat_scales", "ikey_codes", "ikey_scales"), got, ref_cache):
            assert np.array_equal(g[bi].cpu().numpy(), w), (wl.name, b, name)
    ref = oracle.run_sequence(wl, b, cache=ref_cache, layers=layers)
    for l in ref["idx"]:
        assert np.array_equal(seg.layer_idx(l)[bi].cpu().numpy(), ref["idx"][l]), (wl.name, b, l)
    for l in ref["pool"]:
        assert np.array_equal(seg.pool[bi].cpu().numpy(), ref["pool"][l]), (wl.name, b, l)
    for l in ref["out"]:
        err = rel_err_rows(seg.out[l, bi].cpu().numpy(), ref["out"][l])
        assert err <= ATTN_TOL, (wl.name, b, l, err)


def test_ced_40_layers_small(csa):
    """every layer of every copy on a 9,296-position context, two sequences,
    from one captured graph; the newest entry of each copy written in the step"""
    from compressed_sparse_attention_decode_gb300.synthetic import build_schedule
    sched = scaled_schedule(CED_40L, B=2, T=9296)
    step = build_schedule(sched)
    step.capture()
    step.run()
    torch.cuda.synchronize()
    assert len(step.layers) == 40
    for seg, wl in zip(step.segments, sched.segments):
        for bi in range(2):
            check_segment(seg, wl, bi, bi)


def test_ced_storage_is_900_bytes_per_token(csa):
    """the device bytes the four copies hold: three 2:1 copies plus the
    per-position decoder copy at 360 B an entry come to 900 B per raw position"""
    from compressed_sparse_attention_decode_gb300.synthetic import build_schedule
    sched = scaled_schedule(CED_40L, B=2, T=4096)
    step = build_schedule(sched)
    held = sum(t.numel() * t.element_size() for s in step.segments
               for t in (s.cache.lat_codes, s.cache.lat_scales, s.cache.ikey_codes, s.cache.ikey_scales))
    assert held == 900 * sched.B * sched.T


def test_ced_40_layers_full_size_sampled(csa):
    """the benchmark's 40-layer workload (64 sequences, 128K context) and launch
    configuration (one graph per step), run twice; the last sequence checked
    across every layer of every copy, the first on the decoder copy"""
    from compressed_sparse_attention_decode_gb300.synthetic import build_schedule
    step = build_schedule(CED_40L)
    step.capture()
    step.run()
    step.run()
    torch.cuda.synchronize()
    for seg, wl in zip(step.segments, CED_40L.segments):
        check_segment(seg, wl, 63, 63, check_cache=False)
    seg, wl = step.segments[-1], CED_40L.segments[-1]
    check_segment(seg, wl, 0, 0, layers=[0, 4, 19], check_cache=False)

"""Host-side facts of the CED model's 40-layer schedule ("DeepSeek-v4.1 Flash"
§2.3.3) and the window-only layer of the oracle."""
import numpy as np

import oracle
from synth.workloads import CED_40L, ENTRY_BYTES, WORKLOADS, scaled


def test_layer_counts_follow_the_pages():
    """2 SWA layers, 3 encoder blocks of Full + 5 Reuse, 5 decoder blocks of 4
    layers (the first led by Full, the other four by Reindex): 40 layers"""
    L = CED_40L.layers
    assert len(L) == 40
    assert L[:2] == ("swa", "swa")
    assert L[2:20] == (("full",) + ("reuse",) * 5) * 3
    dec = L[20:]
    assert [dec[4 * i] for i in range(5)] == ["full"] + ["reindex"] * 4
    assert all(dec[4 * i + j] == "reuse" for i in range(5) for j in (1, 2, 3))
    enc, d = CED_40L.segments[:3], CED_40L.segments[3]
    assert all(s.ratio == 2 and not s.ikey_proj and not s.pool_blocks for s in enc)
    assert d.ratio == 1 and d.ikey_proj and d.pool_blocks
    assert len({s.seed for s in CED_40L.segments}) == 4


def test_storage_accounting():
    """FP4 latent (256 B codes + 32 B scales) and FP4 indexer key (64 B + 8 B)
    per entry; three encoder copies at one entry per two positions and the
    decoder copy at one per position: 3 x 360 / 2 + 360 = 900 B per token,
    within 1.2 % of the pages' figure of about 890 B per token"""
    assert ENTRY_BYTES == 360
    assert CED_40L.cache_bytes_per_token() == 900
    assert abs(CED_40L.cache_bytes_per_token() / 890 - 1) < 0.012
    # a million-token context: 900 MB against the pages' about 890 MB
    assert sum(s.n_entries * ENTRY_BYTES for s in
               (scaled(x, T=1_000_000) for x in CED_40L.segments)) == 900_000_000


def _softmax_attention(q, rows):
    """textbook single-query attention of every head over the given rows (fp64)"""
    s = q @ rows.T / np.sqrt(512.0)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    return (p @ rows) / p.sum(axis=1, keepdims=True), (m[:, 0] + np.log(p.sum(axis=1)))


def test_window_only_layer_is_plain_softmax_attention():
    """an SWA layer attends to its 128 window rows alone: the textbook softmax
    attention; a Reuse layer after it takes the indices of the last layer that
    made some (the SWA layer makes none)"""
    wl = scaled(WORKLOADS[0], T=2048, layers=("full", "swa", "reuse", "swa"))
    res = oracle.run_sequence(wl, 0)
    first, count = wl.swa_range()
    f = lambda a: oracle.synth_bf16_to_f32(a).astype(np.float64)
    for l in (1, 3):
        assert res["idx"][l].shape == (1, 0)
        o, lse = _softmax_attention(f(wl.q(l, 0)[0]), f(wl.window(l, 0)))
        assert np.abs(res["out"][l][0] - o).max() <= 1e-12 * np.abs(o).max()
        assert np.abs(res["lse"][l][0] - lse).max() <= 1e-12 * np.abs(lse).max()
    assert np.array_equal(res["idx"][2], res["idx"][0])

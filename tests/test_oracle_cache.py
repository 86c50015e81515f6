"""Pins for the cache write: 2:1 channel-wise merge, FP4 quantisation, storage."""
from fractions import Fraction

import numpy as np

import oracle
import synth
from conftest import read_golden
from exact import rn_f32


def test_merge_is_one_rounded_product_then_one_fma():
    rng = np.random.default_rng(0)
    h = synth.normal_bf16(11, 1, (64, 512))
    w0 = rng.uniform(0.3, 0.7, 512).astype(np.float32)
    w1 = rng.uniform(0.3, 0.7, 512).astype(np.float32)
    e = oracle.merge_pairs(h, w0, w1)
    hf = synth.bf16_to_f32(h)
    for i in range(0, 32, 5):
        for c in range(0, 512, 37):
            p0 = rn_f32(Fraction(float(w0[c])) * Fraction(float(hf[2 * i, c])))
            want = rn_f32(Fraction(float(w1[c])) * Fraction(float(hf[2 * i + 1, c])) + Fraction(p0))
            assert float(e[i, c]) == want


def test_merge_special_weights():
    h = synth.normal_bf16(12, 1, (200, 512))
    hf = synth.bf16_to_f32(h)
    one, zero, half = (np.full(512, v, np.float32) for v in (1.0, 0.0, 0.5))
    assert np.array_equal(oracle.merge_pairs(h, one, zero), hf[0::2])
    assert np.array_equal(oracle.merge_pairs(h, zero, one), hf[1::2])
    # (h0 + h1) / 2 of two bf16 values is exact in float64; one rounding to float32
    avg = ((hf[0::2].astype(np.float64) + hf[1::2]) / 2).astype(np.float32)
    assert np.array_equal(oracle.merge_pairs(h, half, half), avg)


def test_cache_write_equals_merge_then_quantise():
    wl_h = synth.normal_bf16(13, 1, (256, 512))
    kraw = synth.normal_bf16(13, 2, (128, 128))
    w0 = synth.uniform_f32(13, 3, (512,), 0.3, 0.7)
    w1 = synth.uniform_f32(13, 4, (512,), 0.3, 0.7)
    lc, ls, kc, ks = oracle.cache_write(wl_h, w0, w1, kraw)
    c2, s2 = oracle.quantize_rows(oracle.merge_pairs(wl_h, w0, w1))
    assert np.array_equal(lc, c2) and np.array_equal(ls, s2)
    c3, s3 = oracle.quantize_rows(synth.bf16_to_f32(kraw))
    assert np.array_equal(kc, c3) and np.array_equal(ks, s3)
    # dequantised latent stays within the codec's error of the merged values
    e = oracle.merge_pairs(wl_h, w0, w1).astype(np.float64)
    dq = oracle.dequant_rows(lc, ls)
    sv = np.array([[oracle.e4m3_value(b) for b in row] for row in ls]).repeat(16, axis=1)
    assert np.all(np.abs(dq - e) <= sv + np.maximum(np.abs(e) - 6 * sv, 0))


def test_storage_per_token_matches_the_pages():
    g = read_golden("storage.txt")
    h = synth.normal_bf16(14, 1, (32, 512))
    kraw = synth.normal_bf16(14, 2, (16, 128))
    w = np.full(512, 0.5, np.float32)
    lc, ls, kc, ks = oracle.cache_write(h, w, w, kraw)
    per_entry = (lc.nbytes + ls.nbytes + kc.nbytes + ks.nbytes) / lc.shape[0]
    assert per_entry == 360  # 256 + 32 latent, 64 + 8 indexer key
    enc, dec = int(g["encoder_copies"]), int(g["decoder_copies"])
    per_token = enc * per_entry / int(g["encoder_ratio"]) + dec * per_entry / int(g["decoder_ratio"])
    tol = float(g["rel_tol"])
    assert abs(per_token - int(g["bytes_per_token"])) / int(g["bytes_per_token"]) < tol
    assert abs(per_token * 1e6 / 1e6 - int(g["mb_at_1m"])) / int(g["mb_at_1m"]) < tol
    assert abs(per_token * 1e5 / 1e6 - int(g["mb_at_100k"])) / int(g["mb_at_100k"]) < tol


def test_projected_indexer_keys_are_the_exact_sum_rounded_once():
    """k = FP4(fp32(W . L)) over the stored entries: the oracle's fp64 sum is checked against
    exact rational arithmetic (every dequantised FP4 value is a small binary fraction), the
    single rounding against an independent round-to-nearest-even, and the codes against the
    codec; the W scale from 2^-9 up to 448 exercises the range the fp64 sum must hold"""
    lat = oracle.quantize_rows(synth.normal_f32(21, 1, (6, 512)) * np.float32(40.0))
    wf = synth.normal_f32(21, 2, (128, 512)) * np.float32(1.0 / np.sqrt(512.0))
    wf[:8] *= np.float32(2.0 ** 12)                 # large rows
    wf[8:16] *= np.float32(2.0 ** -14)              # tiny rows
    wc, ws = oracle.quantize_rows(wf)
    kc, ks = oracle.project_ikeys(lat[0], lat[1], wc, ws)
    Wd = oracle.dequant_rows(wc, ws)
    Ld = oracle.dequant_rows(lat[0], lat[1])
    for i in range(6):
        k = np.empty(128, np.float32)
        for d in range(128):
            exact = sum(Fraction(float(Wd[d, c])) * Fraction(float(Ld[i, c])) for c in range(512))
            assert float(exact) == float(sum(Fraction(float(x)) for x in Wd[d] * Ld[i]))   # products exact in fp64
            k[d] = rn_f32(exact) if exact != 0 else 0.0
        ck, cs = oracle.quantize_rows(k[None])
        assert np.array_equal(kc[i], ck[0]) and np.array_equal(ks[i], cs[0])


def test_decoder_cache_has_one_entry_per_position():
    """ratio 1: entry i is raw position i, quantised as it is; its window and eligibility
    leave no gap and no overlap with the entries before the window"""
    h = synth.normal_bf16(22, 1, (300, 512))
    lc, ls = oracle.cache_write_r1(h)
    wc, ws = oracle.quantize_rows(synth.bf16_to_f32(h))
    assert np.array_equal(lc, wc) and np.array_equal(ls, ws)
    for p in (127, 128, 200, 299):
        n = oracle.n_elig(p, ratio=1)
        assert n == max(0, p - 127)
        assert set(range(n)) | set(range(max(0, p - 127), p + 1)) == set(range(p + 1))

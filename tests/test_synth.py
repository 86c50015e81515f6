"""The seeded generator: deterministic, sliceable, the stated distributions."""
import math

import numpy as np

import synth
from synth.workloads import WORKLOADS, scaled


def test_slices_are_independent_draws():
    full = synth.normal_f32(3, 7, (4096,))
    part = synth.normal_f32(3, 7, (100,), offset=1234)
    assert np.array_equal(full[1234:1334], part)
    u = synth.uniform_f32(3, 8, (1000,), 0.3, 0.7)
    assert np.array_equal(u[500:], synth.uniform_f32(3, 8, (500,), 0.3, 0.7, offset=500))


def test_streams_and_seeds_differ():
    a = synth.raw_bits(0, 1, 64)
    assert not np.array_equal(a, synth.raw_bits(0, 2, 64))
    assert not np.array_equal(a, synth.raw_bits(1, 1, 64))
    assert len(set(a.tolist())) == 64


def test_moments():
    x = synth.normal_f32(0, 1, (1 << 20,)).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    # fourth moment of N(0,1) is 3
    assert abs((x ** 4).mean() - 3.0) < 0.05
    u = synth.uniform_f32(0, 2, (1 << 20,), 0.3, 0.7).astype(np.float64)
    assert u.min() >= 0.3 and u.max() <= 0.7 and abs(u.mean() - 0.5) < 1e-3


def test_own_log_and_sincos_match_libm():
    for v in np.concatenate([np.linspace(1e-300, 1, 2001)[1:], [2.0 ** -53, 0.5, 0.75]]):
        assert abs(synth.gen_log(v) - math.log(v)) <= 4e-16 * max(1.0, abs(math.log(v)))
    for v in np.linspace(0, 1, 4001)[1:-1]:
        c, s = synth.gen_sincos_turns(v)
        assert abs(c - math.cos(2 * math.pi * v)) < 2e-15 and abs(s - math.sin(2 * math.pi * v)) < 2e-15


def test_bf16_is_rne_of_f32():
    x = synth.normal_f32(5, 9, (10000,))
    b = synth.normal_bf16(5, 9, (10000,))
    # reference rounding via numpy integer arithmetic on the float32 bits
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(b, r)
    assert np.all(np.abs(synth.bf16_to_f32(b) - x) <= np.abs(x) * 2.0 ** -8)


def test_workload_shapes():
    w0 = WORKLOADS[0]
    assert (w0.T, WORKLOADS[2].T, WORKLOADS[3].T) == (2048, 131072, 1048576)
    w4 = WORKLOADS[4]
    assert w4.n_q == 8192 and w4.swa_range() == (122880 - 127, 8192 + 127)
    small = scaled(w0, T=512)
    assert small.T == 512 and small.h(0, 0, 4).shape == (4, 512)
    # one sequence's slice equals the matching rows of the whole tensor
    w = scaled(w0, B=2, T=256)
    both = synth.normal_bf16(w.seed, 1, (2, 256, 512))
    assert np.array_equal(w.h(1, 10, 5), both[1, 10:15])

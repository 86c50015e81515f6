"""Seeded synthetic inputs shared by the oracle and the CUDA path.

The module draws numbers and nothing else: no merging, quantisation, scoring
or attention happens here.  Every tensor of a workload is a pure function of
(seed, stream, flat element index), so a test can draw the slice that belongs
to one sequence without drawing the others.  The C source is compiled on first
use (or by ``__graft_entry__.build()``) with gcc.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force=False):
    """Compile libsynth.so (gcc, OpenMP, no contraction of a*b+c)."""
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
        u64, i64 = ctypes.c_uint64, ctypes.c_int64
        vp = ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, vp]
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, i64, vp]
        lib.synth_uniform_f32.argtypes = [u64, u64, u64, i64, ctypes.c_double, ctypes.c_double, vp]
        lib.synth_bits.argtypes = [u64, u64, u64, i64, vp]
        lib.synth_log.argtypes = [ctypes.c_double]
        lib.synth_log.restype = ctypes.c_double
        lib.synth_sincos_turns.argtypes = [ctypes.c_double, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_double)]
        _lib = lib
    return _lib


def _count(shape):
    n = 1
    for s in shape:
        n *= int(s)
    return n


def normal_f32(seed, stream, shape, offset=0, out=None):
    """N(0,1) samples rounded to float32; element i is sample offset+i of the stream."""
    n = _count(shape)
    out = np.empty(shape, np.float32) if out is None else out
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    _load().synth_normal_f32(seed, stream, offset, n, out.ctypes.data)
    return out


def normal_bf16(seed, stream, shape, offset=0, out=None):
    """N(0,1) samples rounded (float32, then RNE) to bfloat16; returned as uint16 bit patterns."""
    n = _count(shape)
    out = np.empty(shape, np.uint16) if out is None else out
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    _load().synth_normal_bf16(seed, stream, offset, n, out.ctypes.data)
    return out


def uniform_f32(seed, stream, shape, lo, hi, offset=0, out=None):
    """U(lo, hi) samples rounded to float32."""
    n = _count(shape)
    out = np.empty(shape, np.float32) if out is None else out
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    _load().synth_uniform_f32(seed, stream, offset, n, float(lo), float(hi), out.ctypes.data)
    return out


def raw_bits(seed, stream, n, offset=0):
    out = np.empty(n, np.uint64)
    _load().synth_bits(seed, stream, offset, n, out.ctypes.data)
    return out


def gen_log(u):
    return _load().synth_log(u)


def gen_sincos_turns(v):
    c, s = ctypes.c_double(), ctypes.c_double()
    _load().synth_sincos_turns(v, ctypes.byref(c), ctypes.byref(s))
    return c.value, s.value


def bf16_to_f32(a):
    """uint16 bfloat16 bit patterns -> float32 (exact widening)."""
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)

"""Seeded synthetic inputs for the paged-attention workloads.

This module is the input generator shared by the checker and the GPU path.
It holds none of the attention arithmetic and no paged address map: it
draws integers (context lengths, block orders), builds value banks of
normal deviates, and fills flat fp16 arrays by plain linear element index.

Every draw comes from SplitMix64 streams (Steele, Lea, Flood, OOPSLA 2014;
finaliser constants from Vigna's `splitmix64.c`), so the same seed gives the
same inputs on every machine, independent of the numpy version.

Element values: element ``i`` of stream ``(seed, stream_id)`` is
``bank[splitmix_at(base, i) >> (64 - BANK_BITS)]`` with ``base =
stream_base(seed, stream_id)``; the bank holds ``2**BANK_BITS`` fp16 values,
``fp16(sigma * z)`` for Box-Muller normals ``z``.
"""
from __future__ import annotations

import ctypes
import math
import os
from functools import lru_cache

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1
BANK_BITS = 24

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libsynth.so")

# Tensor ids inside one layer; stream_id = layer * 16 + tensor id.
KEY_POOL, VALUE_POOL, QUERY, KEY_NEW, VALUE_NEW = 0, 1, 2, 3, 4


def stream_id(layer: int, tensor: int) -> int:
    return int(layer) * 16 + int(tensor)


def mix64(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def splitmix_at(x0: int, i: int) -> int:
    """i-th (0-based) output of the SplitMix64 stream whose state starts at x0."""
    return mix64(x0 + (i + 1) * GAMMA)


def stream_base(seed: int, stream: int) -> int:
    return splitmix_at(((int(seed) << 32) + int(stream)) & MASK64, 0)


class Draws:
    """Sequential SplitMix64 draws for the discrete structure of a workload."""

    def __init__(self, seed: int):
        self.state = int(seed) & MASK64

    def u64(self) -> int:
        self.state = (self.state + GAMMA) & MASK64
        return mix64(self.state)

    def uniform01(self) -> float:
        return (self.u64() >> 11) * 2.0 ** -53

    def integer(self, lo: int, hi: int) -> int:
        """Uniform integer in [lo, hi] by 32-bit multiply-shift (bias < 2^-32 * range)."""
        n = hi - lo + 1
        return lo + (((self.u64() >> 32) * n) >> 32)

    def normal(self) -> float:
        """One Box-Muller deviate (the cosine branch)."""
        u1 = self.uniform01()
        u2 = self.uniform01()
        return math.sqrt(-2.0 * math.log(1.0 - u1)) * math.cos(2.0 * math.pi * u2)

    def permutation(self, n: int) -> np.ndarray:
        """Fisher-Yates shuffle of 0..n-1 (Durstenfeld's in-place form)."""
        a = list(range(n))
        for i in range(n - 1, 0, -1):
            j = self.integer(0, i)
            a[i], a[j] = a[j], a[i]
        return np.asarray(a, dtype=np.int64)


_LIB_HANDLE = None


def _lib() -> ctypes.CDLL:
    global _LIB_HANDLE
    if _LIB_HANDLE is not None:
        return _LIB_HANDLE
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    u64, vp = ctypes.c_uint64, ctypes.c_void_p
    lib.synth_splitmix64_at.argtypes = [u64, u64]
    lib.synth_splitmix64_at.restype = u64
    lib.synth_stream_base.argtypes = [u64, u64]
    lib.synth_stream_base.restype = u64
    lib.synth_bank_normal.argtypes = [vp, u64, u64]
    lib.synth_bank_normal.restype = None
    lib.synth_raw.argtypes = [vp, u64, u64, u64]
    lib.synth_raw.restype = None
    lib.synth_fill_host.argtypes = [vp, vp, ctypes.c_int, u64, u64, u64]
    lib.synth_fill_host.restype = None
    lib.synth_fill_device.argtypes = [vp, vp, ctypes.c_int, u64, u64, u64, vp]
    lib.synth_fill_device.restype = ctypes.c_int
    _LIB_HANDLE = lib
    return lib


@lru_cache(maxsize=4)
def normal_bank(seed: int) -> np.ndarray:
    """2**BANK_BITS standard normal deviates (float64), read-only."""
    out = np.empty(1 << BANK_BITS, dtype=np.float64)
    _lib().synth_bank_normal(out.ctypes.data, out.size, int(seed) & MASK64)
    out.setflags(write=False)
    return out


@lru_cache(maxsize=8)
def fp16_bank(seed: int, sigma: float) -> np.ndarray:
    """The bank scaled by sigma and rounded to fp16 (numpy's IEEE round-to-nearest-even),
    returned as raw uint16 bit patterns."""
    b = (float(sigma) * normal_bank(seed)).astype(np.float16).view(np.uint16)
    b.setflags(write=False)
    return b


def host_values(seed: int, stream: int, start: int, n: int, bank16: np.ndarray) -> np.ndarray:
    """Elements start .. start+n-1 of a stream, as uint16 fp16 bit patterns."""
    out = np.empty(int(n), dtype=np.uint16)
    if n:
        b = np.ascontiguousarray(bank16, dtype=np.uint16)
        _lib().synth_fill_host(out.ctypes.data, b.ctypes.data, BANK_BITS,
                               stream_base(seed, stream), int(start), int(n))
    return out


def host_tensor(seed: int, stream: int, shape, bank16: np.ndarray) -> np.ndarray:
    """A whole tensor of the given shape (elements 0 .. prod(shape)-1), uint16."""
    n = int(np.prod(shape))
    return host_values(seed, stream, 0, n, bank16).reshape(shape)


def device_fill(ptr: int, seed: int, stream: int, start: int, n: int, bank16_dev_ptr: int,
                cuda_stream: int = 0) -> None:
    """Write elements start .. start+n-1 of a stream to device memory at ptr."""
    rc = _lib().synth_fill_device(ctypes.c_void_p(ptr), ctypes.c_void_p(bank16_dev_ptr), BANK_BITS,
                                  stream_base(seed, stream), int(start), int(n),
                                  ctypes.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_device failed with cudaError {rc}")

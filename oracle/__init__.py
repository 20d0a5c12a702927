"""Oracle for the paged-attention decode path.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline / reference leg.  The product library
never imports it and has no CPU fallback.

``oracle.c`` is a plain fp64 statement of the pages' definitions (see its
header for the sources); this module marshals numpy arrays into it.
``block_model`` is a plain model of the pages' block manager.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(closed forms, special cases reducing to library routines, worked examples,
brute force on tiny inputs); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_build.OUT):
        _build.build()
    L = ctypes.CDLL(_build.OUT)
    vp, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_half_to_double.restype = f64
    L.oracle_double_to_half.argtypes = [f64]
    L.oracle_double_to_half.restype = ctypes.c_uint16
    L.oracle_half_to_double_array.argtypes = [vp, vp, ctypes.c_size_t]
    L.oracle_double_to_half_array.argtypes = [vp, vp, ctypes.c_size_t]
    L.oracle_slot_mapping.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32]
    L.oracle_slot_mapping.restype = i32
    L.oracle_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32]
    L.oracle_reshape_and_cache.restype = i32
    L.oracle_copy_blocks.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, i32]
    L.oracle_copy_blocks.restype = i32
    L.oracle_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f64]
    L.oracle_decode.restype = i32
    f32 = ctypes.c_float
    L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_double.restype = f64
    L.oracle_double_to_e4m3.argtypes = [f64]
    L.oracle_double_to_e4m3.restype = ctypes.c_uint8
    L.oracle_e4m3_to_double_array.argtypes = [vp, vp, ctypes.c_size_t]
    L.oracle_double_to_e4m3_array.argtypes = [vp, vp, ctypes.c_size_t]
    L.oracle_quantize_e4m3_array.argtypes = [vp, vp, ctypes.c_size_t, f32]
    L.oracle_reshape_and_cache_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, f32]
    L.oracle_reshape_and_cache_fp8.restype = i32
    L.oracle_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f64,
                                    f64, f64]
    L.oracle_decode_fp8.restype = i32
    L.oracle_swap_blocks.argtypes = [vp, vp, i32, vp, i32, ctypes.c_size_t, ctypes.c_int64,
                                     ctypes.c_int64]
    L.oracle_swap_blocks.restype = i32
    L.oracle_prefill.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, f64]
    L.oracle_prefill.restype = i32
    L.oracle_prefill_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                     f64, f64, f64]
    L.oracle_prefill_fp8.restype = i32
    L.oracle_num_threads.argtypes = []
    L.oracle_num_threads.restype = i32
    L.oracle_set_num_threads.argtypes = [i32]
    L.oracle_set_num_threads.restype = None
    _LIB = L
    return L


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _u16(a: np.ndarray) -> np.ndarray:
    """fp16 data as uint16 bit patterns (accepts float16 or uint16 arrays)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    return _c(a, np.uint16)


def half_to_double(h: np.ndarray) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, dtype=np.float64)
    lib().oracle_half_to_double_array(out.ctypes.data, h.ctypes.data, h.size)
    return out


def double_to_half(x: np.ndarray) -> np.ndarray:
    """Round to fp16 (nearest, ties to even); returns uint16 bit patterns."""
    x = _c(np.asarray(x, dtype=np.float64), np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_double_to_half_array(out.ctypes.data, x.ctypes.data, x.size)
    return out


def slot_mapping(block_tables, token_seq, token_pos, block_size: int, num_blocks: int):
    bt = _c(block_tables, np.int32)
    ts = _c(token_seq, np.int32)
    tp = _c(token_pos, np.int32)
    out = np.empty(ts.shape[0], dtype=np.int64)
    rc = lib().oracle_slot_mapping(out.ctypes.data, bt.ctypes.data, bt.shape[1], ts.ctypes.data,
                                   tp.ctypes.data, ts.shape[0], bt.shape[0], block_size, num_blocks)
    return out, rc


def _inplace_u16(a: np.ndarray) -> np.ndarray:
    """A uint16 view of a C-contiguous fp16/uint16 array that is written in place."""
    if not (isinstance(a, np.ndarray) and a.flags.c_contiguous and a.dtype in (np.uint16, np.float16)):
        raise ValueError("in-place cache arguments must be C-contiguous uint16/float16 arrays")
    return a.view(np.uint16)


def reshape_and_cache(key_cache, value_cache, key, value, slot_mapping_arr, block_size: int) -> int:
    """In place on the (uint16) host caches [NB, H, B, D]."""
    kc, vc = _inplace_u16(key_cache), _inplace_u16(value_cache)
    k, v = _u16(key), _u16(value)
    sm = _c(slot_mapping_arr, np.int64)
    T, H, D = k.shape
    NB = kc.shape[0]
    return lib().oracle_reshape_and_cache(kc.ctypes.data, vc.ctypes.data, k.ctypes.data, v.ctypes.data,
                                          sm.ctypes.data, T, H, D, block_size, NB)


def copy_blocks(key_caches, value_caches, block_mapping) -> int:
    """In place on lists of (uint16) host caches, one per layer."""
    kcs = [_inplace_u16(x) for x in key_caches]
    vcs = [_inplace_u16(x) for x in value_caches]
    bm = _c(np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2), np.int64)
    NB, H, B, D = kcs[0].shape
    kp = (ctypes.c_void_p * len(kcs))(*[x.ctypes.data for x in kcs])
    vp_ = (ctypes.c_void_p * len(vcs))(*[x.ctypes.data for x in vcs])
    return lib().oracle_copy_blocks(kp, vp_, len(kcs), bm.ctypes.data, bm.shape[0], H, D, B, NB)


def decode(query, key_cache, value_cache, block_tables, context_lens, scale: float,
           want64: bool = True):
    """Returns (out16 uint16 [S,H,D], out64 float64 [S,H,D] or None, status)."""
    q = _u16(query)
    kc, vc = _u16(key_cache), _u16(value_cache)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    S, H, D = q.shape
    NB, H2, B, D2 = kc.shape
    assert H2 == H and D2 == D and bt.shape[0] == S and cl.shape[0] == S
    out16 = np.empty((S, H, D), dtype=np.uint16)
    out64 = np.empty((S, H, D), dtype=np.float64) if want64 else None
    rc = lib().oracle_decode(out16.ctypes.data, out64.ctypes.data if want64 else None, q.ctypes.data,
                             kc.ctypes.data, vc.ctypes.data, bt.ctypes.data, bt.shape[1],
                             cl.ctypes.data, S, H, D, B, NB, float(scale))
    return out16, out64, rc


def e4m3_to_double(codes: np.ndarray) -> np.ndarray:
    c = _c(np.asarray(codes, dtype=np.uint8), np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_to_double_array(out.ctypes.data, c.ctypes.data, c.size)
    return out


def double_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code (ties to even), saturating at +-448; uint8."""
    x = _c(np.asarray(x, dtype=np.float64), np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_double_to_e4m3_array(out.ctypes.data, x.ctypes.data, x.size)
    return out


def quantize_e4m3(x16, scale: float) -> np.ndarray:
    """E4M3 codes of fp16 values (uint16 bits or float16): E4M3(fl32(x / scale))."""
    x = _u16(x16)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_quantize_e4m3_array(out.ctypes.data, x.ctypes.data, x.size, float(scale))
    return out


def _inplace_u8(a: np.ndarray) -> np.ndarray:
    if not (isinstance(a, np.ndarray) and a.flags.c_contiguous and a.dtype == np.uint8):
        raise ValueError("FP8 caches must be C-contiguous uint8 arrays")
    return a


def reshape_and_cache_fp8(key_cache, value_cache, key, value, slot_mapping_arr, block_size: int,
                          k_scale: float, v_scale: float) -> int:
    """In place on the uint8 (E4M3) host caches [NB, H, B, D]."""
    kc, vc = _inplace_u8(key_cache), _inplace_u8(value_cache)
    k, v = _u16(key), _u16(value)
    sm = _c(slot_mapping_arr, np.int64)
    T, H, D = k.shape
    return lib().oracle_reshape_and_cache_fp8(kc.ctypes.data, vc.ctypes.data, k.ctypes.data,
                                              v.ctypes.data, sm.ctypes.data, T, H, D, block_size,
                                              kc.shape[0], float(k_scale), float(v_scale))


def decode_fp8(query, key_cache, value_cache, block_tables, context_lens, scale: float,
               k_scale: float, v_scale: float, want64: bool = True):
    """Decode over uint8 (E4M3) caches; returns (out16, out64 or None, status)."""
    q = _u16(query)
    kc = _c(key_cache, np.uint8)
    vc = _c(value_cache, np.uint8)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    S, H, D = q.shape
    NB, H2, B, D2 = kc.shape
    assert H2 == H and D2 == D
    out16 = np.empty((S, H, D), dtype=np.uint16)
    out64 = np.empty((S, H, D), dtype=np.float64) if want64 else None
    rc = lib().oracle_decode_fp8(out16.ctypes.data, out64.ctypes.data if want64 else None,
                                 q.ctypes.data, kc.ctypes.data, vc.ctypes.data, bt.ctypes.data,
                                 bt.shape[1], cl.ctypes.data, S, H, D, B, NB, float(scale),
                                 float(k_scale), float(v_scale))
    return out16, out64, rc


def swap_blocks(dst_pools, src_pools, block_mapping) -> int:
    """In place: block dst of every dst_pools[c] := block src of src_pools[c] for each
    (src, dst) row of block_mapping.  Pools are C-contiguous arrays whose first axis is
    the block id (any element type; the copy is bytewise)."""
    if len(dst_pools) != len(src_pools):
        raise ValueError("one destination pool per source pool")
    n = len(src_pools)
    for a in list(dst_pools) + list(src_pools):
        if not (isinstance(a, np.ndarray) and a.flags.c_contiguous):
            raise ValueError("pools must be C-contiguous numpy arrays")
    bb = src_pools[0].nbytes // src_pools[0].shape[0]
    if any(a.nbytes // a.shape[0] != bb for a in list(dst_pools) + list(src_pools)):
        raise ValueError("all pools must have the same block size in bytes")
    m = _c(block_mapping, np.int64)
    dp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in dst_pools])
    sp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in src_pools])
    return lib().oracle_swap_blocks(dp, sp, n, m.ctypes.data, m.shape[0], bb,
                                    src_pools[0].shape[0], dst_pools[0].shape[0])


def prefill(query, key_cache, value_cache, block_tables, context_lens, query_start, scale: float,
            want64: bool = True):
    """Multi-query paged attention: query / out [total_q, H, D]; query_start int32 [S+1].
    Returns (out16, out64 or None, status)."""
    q = _u16(query)
    kc, vc = _u16(key_cache), _u16(value_cache)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    qs = _c(query_start, np.int32)
    TQ, H, D = q.shape
    NB, H2, B, D2 = kc.shape
    assert H2 == H and D2 == D and qs.shape[0] == cl.shape[0] + 1 and qs[-1] == TQ
    out16 = np.zeros((TQ, H, D), dtype=np.uint16)
    out64 = np.zeros((TQ, H, D), dtype=np.float64) if want64 else None
    rc = lib().oracle_prefill(out16.ctypes.data, out64.ctypes.data if want64 else None,
                              q.ctypes.data, kc.ctypes.data, vc.ctypes.data, bt.ctypes.data,
                              bt.shape[1], cl.ctypes.data, qs.ctypes.data, cl.shape[0], H, D, B,
                              NB, float(scale))
    return out16, out64, rc


def prefill_fp8(query, key_cache, value_cache, block_tables, context_lens, query_start,
                scale: float, k_scale: float, v_scale: float, want64: bool = True):
    """Multi-query paged attention over uint8 (E4M3) caches; returns (out16, out64 or None,
    status)."""
    q = _u16(query)
    kc = _c(key_cache, np.uint8)
    vc = _c(value_cache, np.uint8)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    qs = _c(query_start, np.int32)
    TQ, H, D = q.shape
    NB, H2, B, D2 = kc.shape
    assert H2 == H and D2 == D and qs.shape[0] == cl.shape[0] + 1 and qs[-1] == TQ
    out16 = np.zeros((TQ, H, D), dtype=np.uint16)
    out64 = np.zeros((TQ, H, D), dtype=np.float64) if want64 else None
    rc = lib().oracle_prefill_fp8(out16.ctypes.data, out64.ctypes.data if want64 else None,
                                  q.ctypes.data, kc.ctypes.data, vc.ctypes.data, bt.ctypes.data,
                                  bt.shape[1], cl.ctypes.data, qs.ctypes.data, cl.shape[0], H, D,
                                  B, NB, float(scale), float(k_scale), float(v_scale))
    return out16, out64, rc


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (timing only)."""
    lib().oracle_set_num_threads(int(n))

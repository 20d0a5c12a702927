"""GB300 paged-attention decode library: Python binding of libpa.so.

The functions below carry the C ABI's names (see include/pa.h) and only
marshal arguments: torch tensors supply device pointers and shapes, the
current torch CUDA stream is passed unless one is given.  Every computation
runs in the library's CUDA kernels; there is no CPU fallback, and importing
this package fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

LIB_PATH = _build.OUT

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing; build it first "
                      "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)
_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

_lib.pa_decode_workspace_size.argtypes = [_i32, _i32, _i32, _i32]
_lib.pa_decode_workspace_size.restype = _sz
_lib.pa_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                           ctypes.c_float, _i32, _vp, _sz, _vp]
_lib.pa_decode.restype = _i32
_lib.pa_decode_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                              ctypes.c_float, _i32, _vp, _sz, ctypes.c_uint, _vp]
_lib.pa_decode_ex.restype = _i32
_lib.pa_decode_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                  _i32, ctypes.c_float, _i32, _vp, _sz, ctypes.c_uint, _vp]
_lib.pa_decode_append.restype = _i32
_lib.pa_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                   ctypes.c_float, _i32, _vp]
_lib.pa_decode_noalloc.restype = _i32
_lib.pa_reshape_and_cache.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp]
_lib.pa_reshape_and_cache.restype = _i32
_lib.pa_copy_blocks.argtypes = [_vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _vp]
_lib.pa_copy_blocks.restype = _i32
_lib.pa_slot_mapping.argtypes = [_vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _vp]
_lib.pa_slot_mapping.restype = _i32
_lib.pa_selftest_wait_timeout.argtypes = [_vp]
_lib.pa_selftest_wait_timeout.restype = _i32
_lib.pa_check_errors.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint32)]
_lib.pa_check_errors.restype = _i32
_lib.pa_status_string.argtypes = [_i32]
_lib.pa_status_string.restype = ctypes.c_char_p
_lib.pa_decode_partition_tokens.argtypes = [_i32, _i32, _i32]
_lib.pa_decode_partition_tokens.restype = _i32
_lib.pa_decode_set_partition_tokens.argtypes = [_i32]
_lib.pa_decode_set_partition_tokens.restype = None
_f32 = ctypes.c_float
_lib.pa_decode_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                               _f32, _f32, _f32, _i32, _vp, _sz, _vp]
_lib.pa_decode_fp8.restype = _i32
_lib.pa_decode_fp8_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                  _f32, _f32, _f32, _i32, _vp, _sz, ctypes.c_uint, _vp]
_lib.pa_decode_fp8_ex.restype = _i32
_lib.pa_decode_append_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                      _i32, _i32, _f32, _f32, _f32, _i32, _vp, _sz, ctypes.c_uint, _vp]
_lib.pa_decode_append_fp8.restype = _i32
_lib.pa_reshape_and_cache_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                          _f32, _f32, _vp]
_lib.pa_reshape_and_cache_fp8.restype = _i32
_lib.pa_convert_cache_fp8.argtypes = [_vp, _vp, _sz, _f32, _vp]
_lib.pa_convert_cache_fp8.restype = _i32
_lib.pa_prefill.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                            _i32, _f32, _i32, _vp]
_lib.pa_prefill.restype = _i32
_lib.pa_prefill_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                                _i32, _i32, _f32, _f32, _f32, _i32, _vp]
_lib.pa_prefill_fp8.restype = _i32
_lib.pa_prefill_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                               _i32, _f32, _i32, _i32, ctypes.c_uint32, _vp]
_lib.pa_prefill_ex.restype = _i32
_lib.pa_prefill_fp8_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                                   _i32, _i32, _f32, _f32, _f32, _i32, _i32, ctypes.c_uint32, _vp]
_lib.pa_prefill_fp8_ex.restype = _i32
_lib.pa_swap_blocks.argtypes = [_vp, _vp, _i32, _vp, _i32, _sz, ctypes.c_int64, ctypes.c_int64, _vp]
_lib.pa_swap_blocks.restype = _i32
_lib.pa_copy_blocks_fp8.argtypes = [_vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _vp]
_lib.pa_copy_blocks_fp8.restype = _i32

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_OUT_OF_RANGE, PA_ERR_TIMEOUT = range(6)
PA_ERRBIT_BLOCK_ID, PA_ERRBIT_CONTEXT, PA_ERRBIT_SLOT = 0x1, 0x2, 0x4
PA_ERRBIT_COPY, PA_ERRBIT_TOKEN, PA_ERRBIT_TIMEOUT = 0x8, 0x10, 0x20
PA_DECODE_ZEROED_WORKSPACE = 0x1
PA_DECODE_INPUTS_READY = 0x2
PA_PREFILL_INPUTS_READY = 0x2


class PAError(RuntimeError):
    def __init__(self, status: int, what: str, bits: int = 0):
        self.status = status
        self.bits = bits
        super().__init__(f"{what}: {pa_status_string(status)}" + (f" (bits 0x{bits:x})" if bits else ""))


def pa_status_string(status: int) -> str:
    return _lib.pa_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PAError(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor, name: str, dtype: torch.dtype) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _cache_ptr(t: torch.Tensor, name: str, fp8: bool) -> int:
    """fp16 caches are torch.float16; FP8 (E4M3) caches are torch.uint8 holding
    the codes (a torch.float8_e4m3fn tensor is accepted as the same bytes)."""
    if not fp8:
        return _ptr(t, name, torch.float16)
    if isinstance(t, torch.Tensor) and t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    return _ptr(t, name, torch.uint8)


def pa_decode_workspace_size(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int) -> int:
    return int(_lib.pa_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len))


def pa_decode_partition_tokens(num_seqs: int, num_heads: int, max_context_len: int) -> int:
    return int(_lib.pa_decode_partition_tokens(num_seqs, num_heads, max_context_len))


def pa_decode_set_partition_tokens(tokens: int) -> None:
    _lib.pa_decode_set_partition_tokens(int(tokens))


def decode_workspace(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                     device=None) -> torch.Tensor:
    """A zero-filled device byte buffer of pa_decode_workspace_size(...) bytes (allocated by
    torch), so it may be passed with PA_DECODE_ZEROED_WORKSPACE (see pa_decode_ex)."""
    n = pa_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens):
    S, H, D = query.shape
    NB, H2, B, D2 = key_cache.shape
    if (H2, D2) != (H, D) or tuple(value_cache.shape) != tuple(key_cache.shape):
        raise ValueError("cache shape does not match query")
    if tuple(out.shape) != (S, H, D) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("out / block_tables shape")
    if context_lens.shape != (S,):
        raise ValueError("context_lens shape")
    return S, H, D, B, NB


def pa_decode(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
              value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
              scale: float, max_context_len: int, workspace: torch.Tensor, stream=None) -> None:
    """out[S,H,D] = paged decode attention (see pa_decode in include/pa.h)."""
    S, H, D, B, NB = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    st = _lib.pa_decode(_ptr(out, "out", torch.float16), _ptr(query, "query", torch.float16),
                        _ptr(key_cache, "key_cache", torch.float16),
                        _ptr(value_cache, "value_cache", torch.float16),
                        _ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                        _ptr(context_lens, "context_lens", torch.int32), S, H, D, B, NB,
                        float(scale), int(max_context_len), _ptr(workspace, "workspace", torch.uint8),
                        workspace.numel(), _stream(stream))
    _check(st, "pa_decode")


def pa_decode_ex(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                 value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                 scale: float, max_context_len: int, workspace: torch.Tensor, flags: int = 0,
                 stream=None) -> None:
    """pa_decode with flags (PA_DECODE_ZEROED_WORKSPACE, PA_DECODE_INPUTS_READY; see pa_decode_ex
    in include/pa.h)."""
    S, H, D, B, NB = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    st = _lib.pa_decode_ex(_ptr(out, "out", torch.float16), _ptr(query, "query", torch.float16),
                           _ptr(key_cache, "key_cache", torch.float16),
                           _ptr(value_cache, "value_cache", torch.float16),
                           _ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                           _ptr(context_lens, "context_lens", torch.int32), S, H, D, B, NB,
                           float(scale), int(max_context_len),
                           _ptr(workspace, "workspace", torch.uint8), workspace.numel(), int(flags),
                           _stream(stream))
    _check(st, "pa_decode_ex")


def pa_decode_append(out: torch.Tensor, query: torch.Tensor, key_new: torch.Tensor,
                     value_new: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                     block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                     max_context_len: int, workspace: torch.Tensor, flags: int = 0,
                     stream=None) -> None:
    """The cache write of each sequence's new token (key_new / value_new [S,H,D], written at
    position context_lens[s] - 1) fused into pa_decode_ex (see pa_decode_append in include/pa.h)."""
    S, H, D, B, NB = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    if tuple(key_new.shape) != (S, H, D) or tuple(value_new.shape) != (S, H, D):
        raise ValueError("key_new / value_new must be [S, H, D]")
    st = _lib.pa_decode_append(_ptr(out, "out", torch.float16), _ptr(query, "query", torch.float16),
                               _ptr(key_new, "key_new", torch.float16),
                               _ptr(value_new, "value_new", torch.float16),
                               _ptr(key_cache, "key_cache", torch.float16),
                               _ptr(value_cache, "value_cache", torch.float16),
                               _ptr(block_tables, "block_tables", torch.int32),
                               block_tables.shape[1],
                               _ptr(context_lens, "context_lens", torch.int32), S, H, D, B, NB,
                               float(scale), int(max_context_len),
                               _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                               int(flags), _stream(stream))
    _check(st, "pa_decode_append")


def pa_decode_noalloc(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                      value_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, max_context_len: int,
                      stream=None) -> None:
    """pa_decode with the library's fixed scratch instead of a workspace (see
    pa_decode_noalloc in include/pa.h: calls on one device must be serialised)."""
    S, H, D, B, NB = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    st = _lib.pa_decode_noalloc(_ptr(out, "out", torch.float16), _ptr(query, "query", torch.float16),
                                _ptr(key_cache, "key_cache", torch.float16),
                                _ptr(value_cache, "value_cache", torch.float16),
                                _ptr(block_tables, "block_tables", torch.int32),
                                block_tables.shape[1], _ptr(context_lens, "context_lens", torch.int32),
                                S, H, D, B, NB, float(scale), int(max_context_len), _stream(stream))
    _check(st, "pa_decode_noalloc")


def pa_decode_fp8(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                  value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                  scale: float, k_scale: float, v_scale: float, max_context_len: int,
                  workspace: torch.Tensor, stream=None) -> None:
    """pa_decode over FP8 (E4M3, uint8) caches with per-tensor scales."""
    S, H, D, B, NB = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    st = _lib.pa_decode_fp8(_ptr(out, "out", torch.float16), _ptr(query, "query", torch.float16),
                            _cache_ptr(key_cache, "key_cache", True),
                            _cache_ptr(value_cache, "value_cache", True),
                            _ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                            _ptr(context_lens, "context_lens", torch.int32), S, H, D, B, NB,
                            float(scale), float(k_scale), float(v_scale), int(max_context_len),
                            _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                            _stream(stream))
    _check(st, "pa_decode_fp8")


def pa_decode_fp8_ex(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                     value_cache: torch.Tensor, block_tables: torch.Tensor,
                     context_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float,
                     max_context_len: int, workspace: torch.Tensor, flags: int = 0,
                     stream=None) -> None:
    """pa_decode_fp8 with flags (see pa_decode_ex)."""
    S, H, D, B, NB = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    st = _lib.pa_decode_fp8_ex(_ptr(out, "out", torch.float16), _ptr(query, "query", torch.float16),
                               _cache_ptr(key_cache, "key_cache", True),
                               _cache_ptr(value_cache, "value_cache", True),
                               _ptr(block_tables, "block_tables", torch.int32),
                               block_tables.shape[1],
                               _ptr(context_lens, "context_lens", torch.int32), S, H, D, B, NB,
                               float(scale), float(k_scale), float(v_scale), int(max_context_len),
                               _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
                               int(flags), _stream(stream))
    _check(st, "pa_decode_fp8_ex")


def pa_decode_append_fp8(out: torch.Tensor, query: torch.Tensor, key_new: torch.Tensor,
                         value_new: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, block_tables: torch.Tensor,
                         context_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float,
                         max_context_len: int, workspace: torch.Tensor, flags: int = 0,
                         stream=None) -> None:
    """pa_decode_append over FP8 (E4M3, uint8) caches (the new rows are quantised)."""
    S, H, D, B, NB = _decode_shapes(out, query, key_cache, value_cache, block_tables, context_lens)
    if tuple(key_new.shape) != (S, H, D) or tuple(value_new.shape) != (S, H, D):
        raise ValueError("key_new / value_new must be [S, H, D]")
    st = _lib.pa_decode_append_fp8(_ptr(out, "out", torch.float16),
                                   _ptr(query, "query", torch.float16),
                                   _ptr(key_new, "key_new", torch.float16),
                                   _ptr(value_new, "value_new", torch.float16),
                                   _cache_ptr(key_cache, "key_cache", True),
                                   _cache_ptr(value_cache, "value_cache", True),
                                   _ptr(block_tables, "block_tables", torch.int32),
                                   block_tables.shape[1],
                                   _ptr(context_lens, "context_lens", torch.int32), S, H, D, B, NB,
                                   float(scale), float(k_scale), float(v_scale),
                                   int(max_context_len), _ptr(workspace, "workspace", torch.uint8),
                                   workspace.numel(), int(flags), _stream(stream))
    _check(st, "pa_decode_append_fp8")


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """Scatter key/value [T,H,D] into their slots of the paged caches."""
    T, H, D = key.shape
    NB, H2, B, D2 = key_cache.shape
    if (H2, D2) != (H, D) or tuple(value.shape) != (T, H, D) or slot_mapping.shape != (T,):
        raise ValueError("shape mismatch")
    st = _lib.pa_reshape_and_cache(_ptr(key, "key", torch.float16), _ptr(value, "value", torch.float16),
                                   _ptr(key_cache, "key_cache", torch.float16),
                                   _ptr(value_cache, "value_cache", torch.float16),
                                   _ptr(slot_mapping, "slot_mapping", torch.int64), T, H, D, B, NB,
                                   _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                             value_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                             v_scale: float, stream=None) -> None:
    """Quantise key/value [T,H,D] (fp16) to E4M3 codes into their slots of uint8 caches."""
    T, H, D = key.shape
    NB, H2, B, D2 = key_cache.shape
    if (H2, D2) != (H, D) or tuple(value.shape) != (T, H, D) or slot_mapping.shape != (T,):
        raise ValueError("shape mismatch")
    st = _lib.pa_reshape_and_cache_fp8(_ptr(key, "key", torch.float16),
                                       _ptr(value, "value", torch.float16),
                                       _cache_ptr(key_cache, "key_cache", True),
                                       _cache_ptr(value_cache, "value_cache", True),
                                       _ptr(slot_mapping, "slot_mapping", torch.int64), T, H, D, B,
                                       NB, float(k_scale), float(v_scale), _stream(stream))
    _check(st, "pa_reshape_and_cache_fp8")


def pa_convert_cache_fp8(src: torch.Tensor, dst: torch.Tensor, scale: float, stream=None) -> None:
    """dst (uint8, same shape) := E4M3 codes of src (fp16) under `scale`, element by element."""
    if tuple(src.shape) != tuple(dst.shape):
        raise ValueError("src and dst must have the same shape")
    st = _lib.pa_convert_cache_fp8(_ptr(src, "src", torch.float16), _cache_ptr(dst, "dst", True),
                                   src.numel(), float(scale), _stream(stream))
    _check(st, "pa_convert_cache_fp8")


def pa_copy_blocks(key_caches, value_caches, block_mapping: torch.Tensor, stream=None) -> None:
    """Copy-on-write block copy across all layers; block_mapping is int64 [P, 2] (src, dst),
    a CUDA tensor or pinned host memory (a pinned mapping is also checked on the host)."""
    _copy_blocks(key_caches, value_caches, block_mapping, stream, False)


def pa_copy_blocks_fp8(key_caches, value_caches, block_mapping: torch.Tensor, stream=None) -> None:
    """pa_copy_blocks for FP8 (uint8) caches."""
    _copy_blocks(key_caches, value_caches, block_mapping, stream, True)


def _copy_blocks(key_caches, value_caches, block_mapping, stream, fp8: bool) -> None:
    L = len(key_caches)
    if len(value_caches) != L or L == 0:
        raise ValueError("need one value cache per key cache")
    NB, H, B, D = key_caches[0].shape
    for t in list(key_caches) + list(value_caches):
        if tuple(t.shape) != (NB, H, B, D):
            raise ValueError("all caches must share one shape")
    kp = (ctypes.c_void_p * L)(*[_cache_ptr(t, "key_caches[i]", fp8) for t in key_caches])
    vp = (ctypes.c_void_p * L)(*[_cache_ptr(t, "value_caches[i]", fp8) for t in value_caches])
    if block_mapping.dtype != torch.int64 or block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be int64 [P, 2]")
    fn = _lib.pa_copy_blocks_fp8 if fp8 else _lib.pa_copy_blocks
    st = fn(kp, vp, L, _swap_ptr(block_mapping, "block_mapping"), block_mapping.shape[0],
            H, D, B, NB, _stream(stream))
    _check(st, "pa_copy_blocks_fp8" if fp8 else "pa_copy_blocks")


def pa_prefill(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
               value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
               query_start: torch.Tensor, scale: float, max_query_len: int, stream=None) -> None:
    """Multi-query paged attention (chunked prefill / mixed batches): out[TQ,H,D] for the new
    tokens query[TQ,H,D]; query_start int32 [S+1] (see pa_prefill in include/pa.h)."""
    _prefill(out, query, key_cache, value_cache, block_tables, context_lens, query_start, scale,
             max_query_len, stream, None)


def pa_prefill_ex(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                  value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                  query_start: torch.Tensor, scale: float, max_query_len: int,
                  num_decode_rows: int = -1, flags: int = 0, stream=None) -> None:
    """pa_prefill with the batch's count of one-token sequences (-1: not known) and flags
    (PA_PREFILL_INPUTS_READY); see pa_prefill_ex in include/pa.h."""
    _prefill(out, query, key_cache, value_cache, block_tables, context_lens, query_start, scale,
             max_query_len, stream, None, (int(num_decode_rows), int(flags)))


def pa_prefill_fp8_ex(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                      value_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, query_start: torch.Tensor, scale: float,
                      k_scale: float, v_scale: float, max_query_len: int,
                      num_decode_rows: int = -1, flags: int = 0, stream=None) -> None:
    """pa_prefill_fp8 with the count of one-token sequences and flags (see pa_prefill_ex in
    include/pa.h)."""
    _prefill(out, query, key_cache, value_cache, block_tables, context_lens, query_start, scale,
             max_query_len, stream, (float(k_scale), float(v_scale)), (int(num_decode_rows), int(flags)))


def pa_prefill_fp8(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                   value_cache: torch.Tensor, block_tables: torch.Tensor,
                   context_lens: torch.Tensor, query_start: torch.Tensor, scale: float,
                   k_scale: float, v_scale: float, max_query_len: int, stream=None) -> None:
    """pa_prefill over E4M3 caches (uint8 or float8_e4m3fn tensors) with per-tensor scales."""
    _prefill(out, query, key_cache, value_cache, block_tables, context_lens, query_start, scale,
             max_query_len, stream, (float(k_scale), float(v_scale)))


def _prefill(out, query, key_cache, value_cache, block_tables, context_lens, query_start, scale,
             max_query_len, stream, fp8, ex=None) -> None:
    TQ, H, D = query.shape
    NB, H2, B, D2 = key_cache.shape
    S = context_lens.shape[0]
    if (H2, D2) != (H, D) or tuple(value_cache.shape) != tuple(key_cache.shape):
        raise ValueError("cache shape does not match query")
    if tuple(out.shape) != (TQ, H, D) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("out / block_tables shape")
    if query_start.shape != (S + 1,):
        raise ValueError("query_start must be [num_seqs + 1]")
    common = (_ptr(out, "out", torch.float16), _ptr(query, "query", torch.float16),
              _cache_ptr(key_cache, "key_cache", fp8 is not None),
              _cache_ptr(value_cache, "value_cache", fp8 is not None),
              _ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
              _ptr(context_lens, "context_lens", torch.int32),
              _ptr(query_start, "query_start", torch.int32), S, TQ, H, D, B, NB, float(scale))
    name = "pa_prefill" + ("_fp8" if fp8 is not None else "") + ("_ex" if ex is not None else "")
    args = common + ((fp8[0], fp8[1]) if fp8 is not None else ()) + (int(max_query_len),)
    if ex is not None:  # (num_decode_rows, flags)
        args += ex
    st = getattr(_lib, name)(*args, _stream(stream))
    _check(st, name)


def _swap_ptr(t: torch.Tensor, name: str) -> int:
    """A CUDA tensor or a pinned CPU tensor (the kernel reaches pinned host memory directly)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def pa_swap_blocks(dst_caches, src_caches, block_mapping: torch.Tensor, stream=None) -> None:
    """Block dst of every dst_caches[c] := block src of src_caches[c] for each (src, dst) row of
    block_mapping (int64 [P, 2], CUDA or pinned).  One side is the device pool, the other a
    pinned host pool; dim 0 of every cache is the block id.  Pass all layers' K and V caches."""
    n = len(src_caches)
    if len(dst_caches) != n or n == 0:
        raise ValueError("one destination cache per source cache")
    bb = src_caches[0].numel() // src_caches[0].shape[0] * src_caches[0].element_size()
    for t in list(src_caches) + list(dst_caches):
        if t.numel() // t.shape[0] * t.element_size() != bb:
            raise ValueError("all caches must have the same block size in bytes")
        if tuple(t.shape[1:]) != tuple(src_caches[0].shape[1:]) or t.dtype != src_caches[0].dtype:
            raise ValueError("all caches must share block shape and dtype")
    if block_mapping.dtype != torch.int64 or block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be int64 [P, 2]")
    dp = (ctypes.c_void_p * n)(*[_swap_ptr(t, "dst_caches[i]") for t in dst_caches])
    sp = (ctypes.c_void_p * n)(*[_swap_ptr(t, "src_caches[i]") for t in src_caches])
    st = _lib.pa_swap_blocks(dp, sp, n, _swap_ptr(block_mapping, "block_mapping"),
                             block_mapping.shape[0], bb, src_caches[0].shape[0],
                             dst_caches[0].shape[0], _stream(stream))
    _check(st, "pa_swap_blocks")


def pa_slot_mapping(slot_mapping: torch.Tensor, block_tables: torch.Tensor, token_seq: torch.Tensor,
                    token_pos: torch.Tensor, block_size: int, num_blocks: int, stream=None) -> None:
    """slot_mapping[t] = block_tables[seq][pos // B] * B + pos % B for each new token."""
    T = token_seq.shape[0]
    if token_pos.shape != (T,) or slot_mapping.shape != (T,) or block_tables.dim() != 2:
        raise ValueError("shape mismatch")
    st = _lib.pa_slot_mapping(_ptr(slot_mapping, "slot_mapping", torch.int64),
                              _ptr(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                              _ptr(token_seq, "token_seq", torch.int32),
                              _ptr(token_pos, "token_pos", torch.int32), T, block_tables.shape[0],
                              int(block_size), int(num_blocks), _stream(stream))
    _check(st, "pa_slot_mapping")


def pa_selftest_wait_timeout(stream=None) -> None:
    """Launches a kernel whose bounded wait never completes (see pa_selftest_wait_timeout in
    include/pa.h): about a second later the device error word holds PA_ERRBIT_TIMEOUT."""
    _check(_lib.pa_selftest_wait_timeout(_stream(stream)), "pa_selftest_wait_timeout")


def pa_check_errors(stream=None) -> tuple[int, int]:
    """Synchronise the stream and read + clear the device error word: (status, bits)."""
    bits = ctypes.c_uint32(0)
    st = _lib.pa_check_errors(_stream(stream), ctypes.byref(bits))
    return int(st), int(bits.value)


def raise_on_device_errors(stream=None) -> None:
    st, bits = pa_check_errors(stream)
    if st != PA_OK:
        raise PAError(st, "device error word", bits)


__all__ = [
    "pa_decode", "pa_reshape_and_cache", "pa_copy_blocks", "pa_slot_mapping", "pa_check_errors",
    "pa_selftest_wait_timeout",
    "pa_decode_fp8", "pa_reshape_and_cache_fp8", "pa_copy_blocks_fp8", "pa_convert_cache_fp8",
    "pa_swap_blocks", "pa_prefill", "pa_prefill_fp8", "pa_decode_noalloc", "pa_decode_ex",
    "pa_decode_fp8_ex", "pa_decode_append", "pa_decode_append_fp8", "pa_prefill_ex",
    "pa_prefill_fp8_ex",
    "pa_status_string", "pa_decode_workspace_size", "pa_decode_partition_tokens",
    "pa_decode_set_partition_tokens", "decode_workspace", "raise_on_device_errors", "PAError",
]

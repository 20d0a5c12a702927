"""Device-side inputs for a workload: caches filled in HBM by the generator's
fill kernel, small per-layer tensors generated on the host and uploaded.

Allocation goes through torch (plumbing); nothing here computes attention or
maps addresses.  Values are bit-identical to ``synth.host_values`` for the
same (seed, stream, element index).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import synth
from .configs import Workload

_BANKS: dict = {}


def device_bank(seed: int, sigma: float, device) -> torch.Tensor:
    key = (int(seed), float(sigma), str(device))
    if key not in _BANKS:
        host = synth.fp16_bank(seed, sigma)
        _BANKS[key] = torch.from_numpy(host.view(np.int16).copy()).to(device)
    return _BANKS[key]


def fill(t: torch.Tensor, seed: int, stream_id: int, bank: torch.Tensor, start: int = 0) -> None:
    """t (contiguous fp16/int16 CUDA tensor) := elements start.. of the stream."""
    assert t.is_cuda and t.is_contiguous() and t.element_size() == 2
    synth.device_fill(t.data_ptr(), seed, stream_id, start, t.numel(), bank.data_ptr(),
                      torch.cuda.current_stream(t.device).cuda_stream)


def upload_u16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.float16)


@dataclass
class DeviceWorkload:
    w: Workload
    key_caches: list
    value_caches: list
    queries: list
    keys_new: list
    values_new: list
    block_tables: torch.Tensor | None
    context_lens: torch.Tensor
    token_seq: torch.Tensor
    token_pos: torch.Tensor
    layers: list = field(default_factory=list)


def materialize(w: Workload, layers=None, device="cuda", fill_caches: bool = True,
                fp8_convert=None, fp8_scales=None) -> DeviceWorkload:
    """Allocate and fill the caches of the given layers (default: all) and upload the
    per-layer query and new-token tensors.

    With fp8_convert (a callable (src_fp16, dst_uint8, scale) supplied by the
    caller) the caches are uint8 FP8 caches: each layer's fp16 pool is
    generated into a scratch buffer and handed to fp8_convert with
    fp8_scales = (k_scale, v_scale)."""
    layers = list(range(w.num_layers)) if layers is None else list(layers)
    kv_bank = device_bank(w.seed, w.kv_sigma, device)
    shape = (w.num_blocks, w.num_heads, w.block_size, w.head_dim)
    kcs, vcs, qs, kn, vn = [], [], [], [], []
    tok_seq, tok_pos = w.new_tokens()
    T = len(tok_seq)
    scratch = None
    if fp8_convert is not None and fill_caches:
        scratch = torch.empty(shape, dtype=torch.float16, device=device)
    for l in layers:
        if fp8_convert is not None:
            kc = torch.empty(shape, dtype=torch.uint8, device=device)
            vc = torch.empty(shape, dtype=torch.uint8, device=device)
            if fill_caches:
                for dst, stream, sc in ((kc, w.key_pool_stream(l), fp8_scales[0]),
                                        (vc, w.value_pool_stream(l), fp8_scales[1])):
                    fill(scratch, w.seed, stream, kv_bank)
                    fp8_convert(scratch, dst, sc)
        else:
            kc = torch.empty(shape, dtype=torch.float16, device=device)
            vc = torch.empty(shape, dtype=torch.float16, device=device)
            if fill_caches:
                fill(kc, w.seed, w.key_pool_stream(l), kv_bank)
                fill(vc, w.seed, w.value_pool_stream(l), kv_bank)
        kcs.append(kc)
        vcs.append(vc)
        qs.append(upload_u16(synth.host_tensor(w.seed, w.query_stream(l),
                                               (w.num_seqs, w.num_heads, w.head_dim), w.q_bank()), device))
        kn.append(upload_u16(synth.host_tensor(w.seed, w.key_new_stream(l), (T, w.num_heads, w.head_dim),
                                               w.kv_bank()), device))
        vn.append(upload_u16(synth.host_tensor(w.seed, w.value_new_stream(l), (T, w.num_heads, w.head_dim),
                                               w.kv_bank()), device))
    del scratch
    # Each kind's per-layer tensors are views of one [L, ...] allocation, so consecutive
    # layers' rows lie back to back (the decode step can then upload several layers in one copy).
    qs, kn, vn = _stacked(qs), _stacked(kn), _stacked(vn)
    # The step's small int32 inputs (block tables, context lengths, new tokens' sequences and
    # positions) as views of one allocation, back to back (one upload in the decode step).
    small = [np.ascontiguousarray(a, dtype=np.int32) for a in
             (w.block_tables if w.block_tables is not None else np.zeros((0,), np.int32),
              w.context_lens, tok_seq, tok_pos)]
    flat = torch.from_numpy(np.concatenate([a.reshape(-1) for a in small])).to(device)
    views, off = [], 0
    for a in small:
        views.append(flat[off:off + a.size].view(a.shape))
        off += a.size
    bt = None if w.block_tables is None else views[0]
    return DeviceWorkload(w, kcs, vcs, qs, kn, vn, bt, views[1], views[2], views[3], layers)


def _stacked(ts: list) -> list:
    """The tensors copied into one [len(ts), ...] allocation, returned as its per-row views."""
    if not ts:
        return ts
    big = torch.empty((len(ts),) + tuple(ts[0].shape), dtype=ts[0].dtype, device=ts[0].device)
    for i, t in enumerate(ts):
        big[i].copy_(t)
    return list(big.unbind(0))


def host_pool(w: Workload, layer: int) -> tuple[np.ndarray, np.ndarray]:
    """The same layer's caches generated on the host (uint16 [NB, H, B, D])."""
    shape = (w.num_blocks, w.num_heads, w.block_size, w.head_dim)
    bank = w.kv_bank()
    return (synth.host_tensor(w.seed, w.key_pool_stream(layer), shape, bank),
            synth.host_tensor(w.seed, w.value_pool_stream(layer), shape, bank))


def host_blocks(w: Workload, layer: int, blocks) -> tuple[np.ndarray, np.ndarray]:
    """Selected physical blocks of a layer's caches, generated on the host:
    uint16 [len(blocks), H, B, D] for keys and values."""
    blocks = np.asarray(blocks, dtype=np.int64)
    n = w.tile_elems
    bank = w.kv_bank()
    k = np.empty((len(blocks), n), dtype=np.uint16)
    v = np.empty((len(blocks), n), dtype=np.uint16)
    for i, b in enumerate(blocks):
        k[i] = synth.host_values(w.seed, w.key_pool_stream(layer), int(b) * n, n, bank)
        v[i] = synth.host_values(w.seed, w.value_pool_stream(layer), int(b) * n, n, bank)
    shape = (len(blocks), w.num_heads, w.block_size, w.head_dim)
    return k.reshape(shape), v.reshape(shape)


def host_small(w: Workload, layer: int):
    """(query [S,H,D], key_new [T,H,D], value_new [T,H,D]) as uint16, as uploaded."""
    tok_seq, _ = w.new_tokens()
    T = len(tok_seq)
    q = synth.host_tensor(w.seed, w.query_stream(layer), (w.num_seqs, w.num_heads, w.head_dim), w.q_bank())
    k = synth.host_tensor(w.seed, w.key_new_stream(layer), (T, w.num_heads, w.head_dim), w.kv_bank())
    v = synth.host_tensor(w.seed, w.value_new_stream(layer), (T, w.num_heads, w.head_dim), w.kv_bank())
    return q, k, v


def host_queries(w: Workload) -> np.ndarray:
    """A prefill workload's new-token queries [sum(q_lens), H, D] (uint16)."""
    tq = int(np.sum(w.extra["q_lens"]))
    return synth.host_tensor(w.seed, w.query_stream(0), (tq, w.num_heads, w.head_dim), w.q_bank())


def materialize_prefill(w: Workload, device="cuda") -> dict:
    """Device tensors of a prefill workload: layer-0 caches (generator fill), the
    queries, block tables, context lengths and query_start."""
    from .configs import query_start
    kv_bank = device_bank(w.seed, w.kv_sigma, device)
    shape = (w.num_blocks, w.num_heads, w.block_size, w.head_dim)
    kc = torch.empty(shape, dtype=torch.float16, device=device)
    vc = torch.empty(shape, dtype=torch.float16, device=device)
    fill(kc, w.seed, w.key_pool_stream(0), kv_bank)
    fill(vc, w.seed, w.value_pool_stream(0), kv_bank)
    return {
        "key_cache": kc, "value_cache": vc,
        "query": upload_u16(host_queries(w), device),
        "block_tables": torch.from_numpy(w.block_tables).to(device),
        "context_lens": torch.from_numpy(w.context_lens).to(device),
        "query_start": torch.from_numpy(query_start(w)).to(device),
    }

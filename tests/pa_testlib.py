"""Helpers shared by the GPU parity tests (test plumbing only)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import gpu

# Decode tolerance: elementwise |gpu - ref| <= ATOL + RTOL * |ref|, ref = the
# oracle's unrounded binary64 result (max abs 2e-3 / rel 1e-2 read in the
# allclose form, since a pure relative bound cannot hold where ref ~ 0).
ATOL, RTOL = 2e-3, 1e-2
NAN16 = 0x7E00


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def decode_gate(got: torch.Tensor, ref64: np.ndarray, what: str = "") -> tuple[float, float]:
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref64.shape
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref64)
    bad = err > ATOL + RTOL * np.abs(ref64)
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance, "
                           f"max abs err {err.max():.3e}")
    big = np.abs(ref64) >= 0.1
    max_rel = float((err[big] / np.abs(ref64[big])).max()) if big.any() else 0.0
    return float(err.max()), max_rel


def live_slot_mask(bt: np.ndarray, ctx: np.ndarray, num_blocks: int, block_size: int) -> np.ndarray:
    """bool [NB, B]: True where some sequence's live token lives."""
    mask = np.zeros((num_blocks, block_size), dtype=bool)
    for s, c in enumerate(ctx):
        for i in range(int(c)):
            mask[bt[s, i // block_size], i % block_size] = True
    return mask


def poison_dead_slots_host(kc: np.ndarray, vc: np.ndarray, mask: np.ndarray) -> None:
    dead = ~mask
    kc.transpose(0, 2, 1, 3)[dead] = NAN16
    vc.transpose(0, 2, 1, 3)[dead] = NAN16


def poison_dead_slots_device(kc: torch.Tensor, vc: torch.Tensor, mask: np.ndarray) -> None:
    dead = torch.from_numpy(~mask).to(kc.device)             # [NB, B]
    nan = torch.tensor(float("nan"), dtype=torch.float16, device=kc.device)
    for t in (kc, vc):
        t.permute(0, 2, 1, 3)[dead] = nan


def sampled_oracle(w, layer: int, seqs, new_tokens: bool = True, fp8_scales=None):
    """Oracle outputs for a subset of sequences of a full-size workload, on a
    mini-pool holding only their blocks (relabelled 0..n-1; relabelling does
    not change the result).  Applies the decode step's cache write of each
    sampled sequence's new token.  With fp8_scales = (k_scale, v_scale) the
    pool is the FP8 cache (the oracle quantises the generated fp16 pool, the
    cache write quantises, the decode dequantises).  Returns ref64 [len(seqs), H, D]."""
    seqs = np.asarray(seqs)
    B = w.block_size
    nbs = [-(-int(w.context_lens[s]) // B) for s in seqs]
    used = np.unique(np.concatenate([w.block_tables[s, :n] for s, n in zip(seqs, nbs)]))
    remap = {int(b): i for i, b in enumerate(used)}
    kc, vc = gpu.host_blocks(w, layer, used)
    bt = np.full((len(seqs), w.max_blocks_per_seq), -1, dtype=np.int32)
    for i, (s, n) in enumerate(zip(seqs, nbs)):
        bt[i, :n] = [remap[int(b)] for b in w.block_tables[s, :n]]
    q, kn, vn = gpu.host_small(w, layer)
    ctx = w.context_lens[seqs].astype(np.int32)
    if new_tokens:
        tok_seq, tok_pos = w.new_tokens()
        idx = [int(np.nonzero(tok_seq == s)[0][0]) for s in seqs]
        slots, rc = oracle.slot_mapping(bt, np.arange(len(seqs), dtype=np.int32),
                                        tok_pos[idx].astype(np.int32), B, len(used))
        assert rc == 0
    if fp8_scales is not None:
        ks, vs = fp8_scales
        kc, vc = oracle.quantize_e4m3(kc, ks), oracle.quantize_e4m3(vc, vs)
        if new_tokens:
            assert oracle.reshape_and_cache_fp8(kc, vc, kn[idx], vn[idx], slots, B, ks, vs) == 0
        _, ref64, rc = oracle.decode_fp8(q[seqs], kc, vc, bt, ctx, w.scale, ks, vs)
        assert rc == 0
        return ref64
    if new_tokens:
        assert oracle.reshape_and_cache(kc, vc, kn[idx], vn[idx], slots, B) == 0
    _, ref64, rc = oracle.decode(q[seqs], kc, vc, bt, ctx, w.scale)
    assert rc == 0
    return ref64


# ---- FP8 caches

NAN8 = 0x7F   # an E4M3 NaN code


def materialize_fp8(w, layers=None, device="cuda"):
    """Device workload with uint8 FP8 caches: each layer's generated fp16 pool
    converted by the library's pa_convert_cache_fp8 under configs.fp8_scales."""
    import paged_kv_cache_158_gb300 as pa
    from workloads import configs
    return gpu.materialize(w, layers=layers, device=device, fp8_convert=pa.pa_convert_cache_fp8,
                           fp8_scales=configs.fp8_scales(w))


def poison_dead_slots_host_fp8(kc: np.ndarray, vc: np.ndarray, mask: np.ndarray) -> None:
    dead = ~mask
    kc.transpose(0, 2, 1, 3)[dead] = NAN8
    vc.transpose(0, 2, 1, 3)[dead] = NAN8


def poison_dead_slots_device_fp8(kc: torch.Tensor, vc: torch.Tensor, mask: np.ndarray) -> None:
    dead = torch.from_numpy(~mask).to(kc.device)
    for t in (kc, vc):
        t.permute(0, 2, 1, 3)[dead] = NAN8


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint8)

"""Helpers shared by the GPU parity tests (test plumbing only)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import gpu

# Decode tolerance, as stated for fp16 outputs: max abs error <= 2e-3 and max
# relative error <= 1e-2.  Each bound is applied where it can hold:
#   * abs: |gpu - ref| <= 2e-3 wherever |ref| < 4; from |ref| = 4 on, one
#     step of fp16 at the rounded reference (2^-8 = 3.9e-3 in [4, 8)) is
#     allowed instead, since a correctly rounded fp16 output is already up to
#     half a step away there;
#   * rel: |gpu - ref| / |ref| <= 1e-2 wherever |ref| >= 0.1 (a relative bound
#     cannot hold where ref ~ 0);
# plus the elementwise allclose form |gpu - ref| <= 2e-3 + 1e-2 |ref| as a
# guard.  ref is the oracle's unrounded binary64 result.  Every check records
# its maxima in GATE_LOG; the session prints them (conftest).
# Multi-query attention is held to the same tolerance; its checks are
# tagged "prefill" in the log.
ATOL, RTOL = 2e-3, 1e-2
REL_FLOOR = 0.1
ABS_STEP_FROM = 4.0
NAN16 = 0x7E00
GATE_LOG: list[tuple[str, int, float, float, str]] = []


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def gate_errors(g: np.ndarray, ref64: np.ndarray) -> tuple[float, float, np.ndarray, np.ndarray]:
    """(max abs err, max rel err over |ref| >= 0.1, abs-bound violations,
    rel-bound violations) of float64 arrays g and ref64."""
    err = np.abs(g - ref64)
    mag = np.abs(ref64)
    step = np.spacing(np.minimum(mag, 65504.0).astype(np.float16)).astype(np.float64)
    abs_bound = np.where(mag < ABS_STEP_FROM, ATOL, np.maximum(ATOL, step))
    big = mag >= REL_FLOOR
    rel = np.zeros_like(err)
    rel[big] = err[big] / mag[big]
    bad_abs = err > abs_bound
    bad_rel = big & (rel > RTOL)
    max_abs = float(err.max()) if err.size else 0.0
    max_rel = float(rel.max()) if rel.size else 0.0
    return max_abs, max_rel, bad_abs, bad_rel


def decode_gate(got: torch.Tensor, ref64: np.ndarray, what: str = "",
                record: bool = True, kind: str = "decode") -> tuple[float, float]:
    """Asserts the decode tolerance on every element; returns (max abs err,
    max rel err over |ref| >= 0.1) and, if record, logs them in GATE_LOG
    under `kind` ("decode" or "prefill")."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref64.shape
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    max_abs, max_rel, bad_abs, bad_rel = gate_errors(g, ref64)
    err = np.abs(g - ref64)
    guard = err > ATOL + RTOL * np.abs(ref64)
    assert not guard.any(), f"{what}: {int(guard.sum())} elements outside 2e-3 + 1e-2|ref|"
    assert not bad_abs.any(), (f"{what}: {int(bad_abs.sum())} elements above the abs bound, "
                               f"max abs err {max_abs:.3e}")
    assert not bad_rel.any(), (f"{what}: {int(bad_rel.sum())} elements above the rel bound, "
                               f"max rel err {max_rel:.3e}")
    if record:
        GATE_LOG.append((what, int(g.size), max_abs, max_rel, kind))
    return max_abs, max_rel


def prefill_gate(got: torch.Tensor, ref64: np.ndarray, what: str = "",
                 record: bool = True) -> tuple[float, float]:
    """decode_gate for multi-query attention outputs (logged as "prefill")."""
    return decode_gate(got, ref64, what, record, kind="prefill")


def live_slot_mask(bt: np.ndarray, ctx: np.ndarray, num_blocks: int, block_size: int) -> np.ndarray:
    """bool [NB, B]: True where some sequence's live token lives."""
    mask = np.zeros((num_blocks, block_size), dtype=bool)
    for s, c in enumerate(ctx):
        i = np.arange(int(c))
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


def whole_layer_oracle(w, layer: int, fp8_scales=None, poison: bool = True) -> np.ndarray:
    """Oracle output of one whole layer of a workload after its decode step's
    cache write: the layer's full pool generated on the host, the new tokens'
    slots from the oracle's slot map, the oracle's cache write, every dead
    slot poisoned with NaN (so a read of one shows), then the oracle's decode
    of every (sequence, head).  With fp8_scales = (k_scale, v_scale) the pool
    is the FP8 cache (quantised by the oracle).  Returns ref64 [S, H, D]."""
    B = w.block_size
    kc, vc = gpu.host_pool(w, layer)
    q, kn, vn = gpu.host_small(w, layer)
    seqs, pos = w.new_tokens()
    slots, rc = oracle.slot_mapping(w.block_tables, seqs, pos, B, w.num_blocks)
    assert rc == 0
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, B) if poison else None
    if fp8_scales is not None:
        ks, vs = fp8_scales
        kc, vc = oracle.quantize_e4m3(kc, ks), oracle.quantize_e4m3(vc, vs)
        assert oracle.reshape_and_cache_fp8(kc, vc, kn, vn, slots, B, ks, vs) == 0
        if poison:
            poison_dead_slots_host_fp8(kc, vc, mask)
        _, ref64, rc = oracle.decode_fp8(q, kc, vc, w.block_tables, w.context_lens, w.scale, ks, vs)
    else:
        assert oracle.reshape_and_cache(kc, vc, kn, vn, slots, B) == 0
        if poison:
            poison_dead_slots_host(kc, vc, mask)
        _, ref64, rc = oracle.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
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

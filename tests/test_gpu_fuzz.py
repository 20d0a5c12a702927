"""Seeded random parity against the oracle: decode over fp16 and FP8 caches, the decode with
the cache write fused in, and multi-query attention, on random shapes (head size, block size,
batch size, heads), ragged contexts with empty, one-token and block-boundary lengths, and
forced partition sizes; every output element by element, every dead cache slot NaN-poisoned
so that a read of one shows."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa
from pa_testlib import (decode_gate, live_slot_mask, materialize_fp8, poison_dead_slots_device,
                        poison_dead_slots_device_fp8, prefill_gate, whole_layer_oracle)
from workloads import configs, gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _reset():
    pa.pa_decode_set_partition_tokens(0)
    pa.pa_check_errors()
    yield
    pa.pa_decode_set_partition_tokens(0)
    torch.cuda.synchronize()


def random_decode_workload(i):
    """Case i: shapes and contexts drawn from a seeded generator.  Contexts are drawn first,
    the tables built for them, then some are shortened to 0, 1, B - 1, B or B + 1 (a shorter
    context leaves the rest of its table unread)."""
    rng = np.random.default_rng(9000 + i)
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([4, 8, 16, 32]))
    S = int(rng.integers(1, 41))
    H = int(rng.integers(1, 9))
    cmax = int(rng.choice([B + 2, 3 * B, 200, 700, 2100]))
    w = configs.small_random(9000 + i, S, H, D, B, cmax, min_context=min(cmax, B + 2))
    for s in rng.choice(S, size=min(S, 4), replace=False):
        w.context_lens[s] = min(int(w.context_lens[s]), int(rng.choice([0, 1, B - 1, B, B + 1])))
    part = int(rng.choice([0, 32, 64, 160]))
    return w, part


def _new_rows(w, dw):
    """The new tokens' rows as [S, H, D] (zeros for empty contexts)."""
    seqs, _ = w.new_tokens()
    kn = torch.zeros((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float16, device=DEV)
    vn = torch.zeros_like(kn)
    idx = torch.from_numpy(seqs.astype(np.int64)).to(DEV)
    kn[idx] = dw.keys_new[0]
    vn[idx] = dw.values_new[0]
    return kn, vn


@pytest.mark.parametrize("i", range(12))
@pytest.mark.parametrize("mode", ["fp16", "fp16_fused", "fp8", "fp8_fused"])
def test_random_decode_step_against_oracle(i, mode):
    w, part = random_decode_workload(i)
    pa.pa_decode_set_partition_tokens(part)
    fp8 = mode.startswith("fp8")
    ks, vs = configs.fp8_scales(w)
    dw = materialize_fp8(w) if fp8 else gpu.materialize(w, device=DEV)
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, w.block_size)
    (poison_dead_slots_device_fp8 if fp8 else poison_dead_slots_device)(dw.key_caches[0],
                                                                        dw.value_caches[0], mask)
    out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=torch.float16,
                     device=DEV)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    args = (dw.key_caches[0], dw.value_caches[0], dw.block_tables, dw.context_lens, w.scale)
    if mode.endswith("fused"):
        kn, vn = _new_rows(w, dw)
        if fp8:
            pa.pa_decode_append_fp8(out, dw.queries[0], kn, vn, *args, ks, vs, w.max_context_len, ws)
        else:
            pa.pa_decode_append(out, dw.queries[0], kn, vn, *args, w.max_context_len, ws)
    else:
        T = dw.token_seq.numel()
        if T:
            slots = torch.empty(T, dtype=torch.int64, device=DEV)
            pa.pa_slot_mapping(slots, dw.block_tables, dw.token_seq, dw.token_pos, w.block_size,
                               w.num_blocks)
            if fp8:
                pa.pa_reshape_and_cache_fp8(dw.keys_new[0], dw.values_new[0], dw.key_caches[0],
                                            dw.value_caches[0], slots, ks, vs)
            else:
                pa.pa_reshape_and_cache(dw.keys_new[0], dw.values_new[0], dw.key_caches[0],
                                        dw.value_caches[0], slots)
        if fp8:
            pa.pa_decode_fp8(out, dw.queries[0], *args, ks, vs, w.max_context_len, ws)
        else:
            pa.pa_decode(out, dw.queries[0], *args, w.max_context_len, ws)
    torch.cuda.synchronize()
    ref64 = whole_layer_oracle(w, 0, fp8_scales=(ks, vs) if fp8 else None)
    decode_gate(out, ref64, f"random decode {i} {mode} D{w.head_dim} B{w.block_size} "
                            f"S{w.num_seqs} H{w.num_heads} part{part}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("i", range(10))
@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("count", [False, True])
def test_random_prefill_against_oracle(i, fp8, count):
    """Random mixes of empty, one-token and longer chunks (some crossing several 128-row
    tiles) over random contexts; count: the call is told how many one-token sequences the
    batch holds (up to four heads of a row per CTA)."""
    rng = np.random.default_rng(9100 + i)
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([8, 16, 32]))
    H = int(rng.integers(1, 7))
    S = int(rng.integers(1, 13))
    q_lens = [int(rng.choice([0, 1, 1, int(rng.integers(2, 130)), int(rng.integers(130, 600))]))
              for _ in range(S)]
    if max(q_lens) == 0:
        q_lens[0] = 5
    ctx = [q + int(rng.integers(0 if q else 1, 900)) for q in q_lens]
    w = configs.prefill_workload("random", 9100 + i, q_lens, ctx, H, D, B)
    dv = gpu.materialize_prefill(w, DEV)
    ks, vs = configs.fp8_scales(w)
    if fp8:
        for name, sc in (("key_cache", ks), ("value_cache", vs)):
            codes = torch.empty(dv[name].shape, dtype=torch.uint8, device=DEV)
            pa.pa_convert_cache_fp8(dv[name], codes, sc)
            dv[name] = codes
    tq = int(np.sum(q_lens))
    out = torch.full((tq, H, D), float("nan"), dtype=torch.float16, device=DEV)
    args = (out, dv["query"], dv["key_cache"], dv["value_cache"], dv["block_tables"],
            dv["context_lens"], dv["query_start"], w.scale)
    n_rows = sum(1 for q in q_lens if q == 1) if count else -1
    if fp8:
        pa.pa_prefill_fp8_ex(*args, ks, vs, max(q_lens), n_rows)
    else:
        pa.pa_prefill_ex(*args, max(q_lens), n_rows)
    torch.cuda.synchronize()
    kc, vc = gpu.host_pool(w, 0)
    q = gpu.host_queries(w)
    if fp8:
        kc8, vc8 = oracle.quantize_e4m3(kc, ks), oracle.quantize_e4m3(vc, vs)
        _, ref64, rc = oracle.prefill_fp8(q, kc8, vc8, w.block_tables, w.context_lens,
                                          configs.query_start(w), w.scale, ks, vs)
    else:
        _, ref64, rc = oracle.prefill(q, kc, vc, w.block_tables, w.context_lens,
                                      configs.query_start(w), w.scale)
    assert rc == 0
    prefill_gate(out, ref64, f"random prefill {i} {'fp8' if fp8 else 'fp16'} D{D} B{B} S{S} H{H} "
                             f"count {n_rows}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)

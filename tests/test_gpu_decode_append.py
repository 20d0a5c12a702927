"""The decode with the new token's cache write fused in (pa_decode_append,
pa_decode_append_fp8): outputs and caches bit-identical to the slot map +
cache write + decode it replaces, for every head size and block size, fp16
and FP8 caches, several partitions per sequence, empty and one-token
contexts, and more sequences than one launch; whole layers against the
oracle; clipped contexts and bad block ids write nothing and are reported."""
import numpy as np
import pytest
import torch

import paged_kv_cache_158_gb300 as pa
from pa_testlib import (decode_gate, live_slot_mask, materialize_fp8, poison_dead_slots_device,
                        poison_dead_slots_device_fp8, whole_layer_oracle)
from workloads import configs, gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"
ZW = pa.PA_DECODE_ZEROED_WORKSPACE


@pytest.fixture(autouse=True)
def _reset():
    pa.pa_decode_set_partition_tokens(0)
    pa.pa_check_errors()
    yield
    pa.pa_decode_set_partition_tokens(0)
    torch.cuda.synchronize()


def new_rows(w, dw):
    """[S, H, D] new key/value rows: row s is sequence s's new token (zeros where c = 0)."""
    seqs, _ = w.new_tokens()
    kn = torch.zeros((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float16, device=DEV)
    vn = torch.zeros_like(kn)
    idx = torch.from_numpy(seqs.astype(np.int64)).to(DEV)
    kn[idx] = dw.keys_new[0]
    vn[idx] = dw.values_new[0]
    return kn, vn


def separate(w, dw, fp8, ws):
    ks, vs = configs.fp8_scales(w)
    slots = torch.empty(dw.token_seq.numel(), dtype=torch.int64, device=DEV)
    pa.pa_slot_mapping(slots, dw.block_tables, dw.token_seq, dw.token_pos, w.block_size, w.num_blocks)
    out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=torch.float16,
                     device=DEV)
    if fp8:
        pa.pa_reshape_and_cache_fp8(dw.keys_new[0], dw.values_new[0], dw.key_caches[0],
                                    dw.value_caches[0], slots, ks, vs)
        pa.pa_decode_fp8_ex(out, dw.queries[0], dw.key_caches[0], dw.value_caches[0],
                            dw.block_tables, dw.context_lens, w.scale, ks, vs, w.max_context_len,
                            ws, ZW)
    else:
        pa.pa_reshape_and_cache(dw.keys_new[0], dw.values_new[0], dw.key_caches[0],
                                dw.value_caches[0], slots)
        pa.pa_decode_ex(out, dw.queries[0], dw.key_caches[0], dw.value_caches[0], dw.block_tables,
                        dw.context_lens, w.scale, w.max_context_len, ws, ZW)
    return out


def fused(w, dw, fp8, ws, kn, vn, max_ctx=None):
    ks, vs = configs.fp8_scales(w)
    out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=torch.float16,
                     device=DEV)
    mc = w.max_context_len if max_ctx is None else max_ctx
    if fp8:
        pa.pa_decode_append_fp8(out, dw.queries[0], kn, vn, dw.key_caches[0], dw.value_caches[0],
                                dw.block_tables, dw.context_lens, w.scale, ks, vs, mc, ws, ZW)
    else:
        pa.pa_decode_append(out, dw.queries[0], kn, vn, dw.key_caches[0], dw.value_caches[0],
                            dw.block_tables, dw.context_lens, w.scale, mc, ws, ZW)
    return out


def two_copies(w, fp8):
    """The same device workload twice (caches poisoned with NaN in every dead slot)."""
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, w.block_size)
    res = []
    for _ in range(2):
        dw = materialize_fp8(w) if fp8 else gpu.materialize(w, device=DEV)
        if fp8:
            poison_dead_slots_device_fp8(dw.key_caches[0], dw.value_caches[0], mask)
        else:
            poison_dead_slots_device(dw.key_caches[0], dw.value_caches[0], mask)
        res.append(dw)
    return res


def same_bits(a, b):
    return torch.equal(a.view(torch.int8), b.view(torch.int8))


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("part", [0, 32])
@pytest.mark.parametrize("D,B", [(d, b) for d in (64, 128) for b in (4, 8, 16, 32)])
def test_fused_write_matches_write_then_decode(D, B, part, fp8):
    pa.pa_decode_set_partition_tokens(part)
    # Tables drawn for at least B + 1 tokens, then three sequences shortened:
    # empty, one token, exactly one block.
    w = configs.small_random(6000 + D + B + part + fp8, 9, 3, D, B, 150, min_context=B + 1)
    w.context_lens[0], w.context_lens[1], w.context_lens[2] = 0, 1, B
    w.block_tables[0, :] = -1
    a, b = two_copies(w, fp8)
    ws_a = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    ws_b = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    ref = separate(w, a, fp8, ws_a)
    kn, vn = new_rows(w, b)
    got = fused(w, b, fp8, ws_b, kn, vn)
    torch.cuda.synchronize()
    assert same_bits(got, ref)
    assert same_bits(b.key_caches[0], a.key_caches[0]) and same_bits(b.value_caches[0], a.value_caches[0])
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("fp8", [False, True])
def test_fused_write_more_sequences_than_one_launch(fp8):
    pa.pa_decode_set_partition_tokens(32)
    w = configs.small_random(6100 + fp8, 1100, 2, 128, 16, 90, min_context=1)
    a, b = two_copies(w, fp8)
    ws_a = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    ws_b = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    ref = separate(w, a, fp8, ws_a)
    kn, vn = new_rows(w, b)
    got = fused(w, b, fp8, ws_b, kn, vn)
    torch.cuda.synchronize()
    assert same_bits(got, ref)
    assert same_bits(b.key_caches[0], a.key_caches[0]) and same_bits(b.value_caches[0], a.value_caches[0])


@pytest.mark.parametrize("cfg,fp8", [(2, False), (2, True), (5, False), (5, True)])
def test_fused_write_whole_layer_against_oracle(cfg, fp8):
    """The 7B-shaped layer and one long-context layer at full size, every
    output against the oracle's own slot map, cache write and decode."""
    w = configs.ALL[cfg]() if cfg != 5 else configs.config5(num_layers=1)
    dw = materialize_fp8(w, layers=[0]) if fp8 else gpu.materialize(w, layers=[0], device=DEV)
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, w.block_size)
    if fp8:
        poison_dead_slots_device_fp8(dw.key_caches[0], dw.value_caches[0], mask)
    else:
        poison_dead_slots_device(dw.key_caches[0], dw.value_caches[0], mask)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    kn, vn = new_rows(w, dw)
    out = fused(w, dw, fp8, ws, kn, vn)
    ref64 = whole_layer_oracle(w, 0, fp8_scales=configs.fp8_scales(w) if fp8 else None)
    decode_gate(out, ref64, f"append {'fp8 ' if fp8 else ''}{w.name}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_fused_write_skips_clipped_contexts_and_bad_blocks():
    """A context clipped by max_context_len, and a block id out of range at the
    new token's position: both are reported and write nothing; the other
    sequences are written as usual."""
    w = configs.small_random(6200, 4, 2, 64, 16, 60, min_context=20)
    ctx = w.context_lens
    top = int(ctx.max())
    clipped = int(np.argmax(ctx))
    for s in range(4):                        # only `clipped` goes past max_context_len
        if s != clipped:
            ctx[s] = min(int(ctx[s]), top - 1)
    bad = (clipped + 1) % 4
    _, b = two_copies(w, False)
    bad_blk = (int(ctx[bad]) - 1) // 16
    b.block_tables[bad, bad_blk] = w.num_blocks + 5    # after the poisoning, which reads the table
    before_k = b.key_caches[0].clone()
    kn, vn = new_rows(w, b)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, top - 1)
    fused(w, b, False, ws, kn, vn, max_ctx=top - 1)
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE
    assert bits & pa.PA_ERRBIT_CONTEXT and bits & pa.PA_ERRBIT_BLOCK_ID
    kc = b.key_caches[0]
    for s in range(4):
        c = int(ctx[s])
        blk = int(w.block_tables[s, (c - 1) // 16])
        row = kc[blk, :, (c - 1) % 16].view(torch.int16)
        if s in (clipped, bad):               # nothing written at the new token's slot
            assert torch.equal(row, before_k[blk, :, (c - 1) % 16].view(torch.int16))
        else:
            assert torch.equal(row, kn[s].view(torch.int16))


def test_append_rejects_missing_rows():
    w = configs.small_random(6300, 2, 2, 64, 16, 30, min_context=1)
    dw = gpu.materialize(w, device=DEV)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    out = torch.empty((2, 2, 64), dtype=torch.float16, device=DEV)
    with pytest.raises(ValueError):
        pa.pa_decode_append(out, dw.queries[0], dw.keys_new[0][:1], dw.values_new[0][:1],
                            dw.key_caches[0], dw.value_caches[0], dw.block_tables, dw.context_lens,
                            w.scale, w.max_context_len, ws)

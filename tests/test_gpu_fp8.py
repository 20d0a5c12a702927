"""GPU parity of the FP8 (E4M3) KV-cache path against the oracle: cache
conversion and cache write bit-exact (every fp16 pattern, saturation,
padding), block copy bit-exact, decode within the decode tolerance on small
ragged batches (several partitions, NaN codes in every dead slot), on whole
workload steps and on whole layers of the full-size workloads; plus permutation
invariance and determinism."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa
from pa_testlib import (NAN8, decode_gate, live_slot_mask, materialize_fp8, poison_dead_slots_device_fp8,
                        poison_dead_slots_host_fp8, sampled_oracle, u8, whole_layer_oracle)
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


def run_decode_fp8(dw, layer_idx=0):
    w = dw.w
    ks, vs = configs.fp8_scales(w)
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float16, device=DEV)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    pa.pa_decode_fp8(out, dw.queries[layer_idx], dw.key_caches[layer_idx], dw.value_caches[layer_idx],
                     dw.block_tables, dw.context_lens, w.scale, ks, vs, w.max_context_len, ws)
    return out


def cache_write_fp8(dw, layer_idx=0):
    w = dw.w
    ks, vs = configs.fp8_scales(w)
    slots = torch.empty(dw.token_seq.numel(), dtype=torch.int64, device=DEV)
    pa.pa_slot_mapping(slots, dw.block_tables, dw.token_seq, dw.token_pos, w.block_size, w.num_blocks)
    pa.pa_reshape_and_cache_fp8(dw.keys_new[layer_idx], dw.values_new[layer_idx],
                                dw.key_caches[layer_idx], dw.value_caches[layer_idx], slots, ks, vs)


def oracle_fp8_pool(w, layer=0):
    ks, vs = configs.fp8_scales(w)
    kc16, vc16 = gpu.host_pool(w, layer)
    return oracle.quantize_e4m3(kc16, ks), oracle.quantize_e4m3(vc16, vs)


# ------------------------------------------------------------ conversion / write

@pytest.mark.parametrize("scale", [1.0, 0.37, 0.0625, 3.0, 0.0137])
def test_convert_every_fp16_pattern_bit_exact(scale):
    """Every finite fp16 pattern and +-inf (values past 448 saturate)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    keep = np.isfinite(bits.view(np.float16)) | np.isin(bits, [0x7C00, 0xFC00])
    x = bits[keep]
    x = np.concatenate([x, np.zeros((-len(x)) % 16, dtype=np.uint16)])
    src = torch.from_numpy(x.view(np.int16).copy()).to(DEV).view(torch.float16)
    dst = torch.empty(src.shape, dtype=torch.uint8, device=DEV)
    pa.pa_convert_cache_fp8(src, dst, scale)
    assert np.array_equal(u8(dst), oracle.quantize_e4m3(x, scale))


@pytest.mark.parametrize("D,B", [(64, 4), (64, 16), (128, 8), (128, 32)])
def test_reshape_and_cache_fp8_bit_exact(D, B):
    w = configs.small_random(2000 + D + B, 9, 3, D, B, 200, min_context=1)
    dw = materialize_fp8(w)
    kc8, vc8 = oracle_fp8_pool(w)
    assert np.array_equal(u8(dw.key_caches[0]), kc8) and np.array_equal(u8(dw.value_caches[0]), vc8)
    # new tokens, with one padding token and a saturating key
    seqs, pos = w.new_tokens()
    slots, rc = oracle.slot_mapping(w.block_tables, seqs, pos, B, w.num_blocks)
    assert rc == 0
    slots[2] = -1
    _, kn, vn = gpu.host_small(w, 0)
    kn = kn.copy()
    kn[0, 0, :4] = np.array([60000.0, -60000.0, 7.0, -0.0], dtype=np.float16).view(np.uint16)
    ks, vs = configs.fp8_scales(w)
    assert oracle.reshape_and_cache_fp8(kc8, vc8, kn, vn, slots, B, ks, vs) == 0
    pa.pa_reshape_and_cache_fp8(gpu.upload_u16(kn, DEV), dw.values_new[0], dw.key_caches[0],
                                dw.value_caches[0], torch.from_numpy(slots).to(DEV), ks, vs)
    assert np.array_equal(u8(dw.key_caches[0]), kc8) and np.array_equal(u8(dw.value_caches[0]), vc8)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_reshape_and_cache_fp8_bad_slot_flagged():
    w = configs.small_random(2100, 3, 2, 128, 16, 40, min_context=1)
    dw = materialize_fp8(w)
    before = u8(dw.key_caches[0]).copy()
    slots = torch.tensor([0, w.num_blocks * 16, -1], dtype=torch.int64, device=DEV)
    ks, vs = configs.fp8_scales(w)
    pa.pa_reshape_and_cache_fp8(dw.keys_new[0][:3], dw.values_new[0][:3], dw.key_caches[0],
                                dw.value_caches[0], slots, ks, vs)
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_SLOT
    after = u8(dw.key_caches[0])
    # slot 0 written, nothing else changed
    diff = np.argwhere((after != before).transpose(0, 2, 1, 3).any(axis=(2, 3)))
    assert all(tuple(d) == (0, 0) for d in diff)


def test_copy_blocks_fp8_bit_exact():
    w = configs.small_random(2200, 4, 4, 64, 16, 100, min_context=10, spare_blocks=6)
    dw = materialize_fp8(w, layers=[0])
    k2 = dw.key_caches + [dw.key_caches[0].flip(0).contiguous()]
    v2 = dw.value_caches + [dw.value_caches[0].flip(0).contiguous()]
    hk = [u8(t).copy() for t in k2]
    hv = [u8(t).copy() for t in v2]
    pairs = np.array([[0, w.num_blocks - 1], [3, w.num_blocks - 2], [5, 1]], dtype=np.int64)
    pa.pa_copy_blocks_fp8(k2, v2, torch.from_numpy(pairs).to(DEV))
    for l in range(2):
        for src, dst in pairs:
            hk[l][dst] = hk[l][src]
            hv[l][dst] = hv[l][src]
        assert np.array_equal(u8(k2[l]), hk[l]) and np.array_equal(u8(v2[l]), hv[l])
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


# ------------------------------------------------------------ decode

SMALL = [(d, b) for d in (64, 128) for b in (4, 8, 16, 32)]


@pytest.mark.parametrize("part", [0, 32, 96])
@pytest.mark.parametrize("D,B", SMALL)
def test_decode_fp8_small_random(D, B, part):
    """Ragged contexts (including 0 and 1), NaN codes in every dead slot,
    forced small partitions so several partitions and the merge kernel run."""
    pa.pa_decode_set_partition_tokens(part)
    w = configs.small_random(3000 + D + B + part, 7, 3, D, B, 300, min_context=0)
    w.context_lens[0], w.context_lens[1] = 0, 1
    w.block_tables[0, :] = -1
    dw = materialize_fp8(w)
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, B)
    poison_dead_slots_device_fp8(dw.key_caches[0], dw.value_caches[0], mask)
    out = run_decode_fp8(dw)
    kc8, vc8 = oracle_fp8_pool(w)
    poison_dead_slots_host_fp8(kc8, vc8, mask)
    q = gpu.host_small(w, 0)[0]
    ks, vs = configs.fp8_scales(w)
    _, ref64, rc = oracle.decode_fp8(q, kc8, vc8, w.block_tables, w.context_lens, w.scale, ks, vs)
    assert rc == 0
    decode_gate(out, ref64, f"fp8 D{D} B{B} part{part}")
    assert (out[0].view(torch.int16) == 0).all()        # empty context: zero row
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("cfg", [1, 2])
def test_decode_fp8_step_workload_all_outputs(cfg):
    """Slot map + FP8 cache write + FP8 decode of workloads 1 and 2, every output."""
    w = configs.ALL[cfg]()
    dw = materialize_fp8(w, layers=[0])
    cache_write_fp8(dw)
    out = run_decode_fp8(dw)
    ref64 = sampled_oracle(w, 0, np.arange(w.num_seqs), fp8_scales=configs.fp8_scales(w))
    decode_gate(out, ref64, f"fp8 {w.name}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("layers", [(0, 21), (30, 39)])
def test_decode_fp8_workload3_whole_layers(layers):
    """13B shape with all 40 layers' FP8 caches resident: the FP8 decode step of
    whole layers, every output against the oracle."""
    w = configs.config3()
    dw = materialize_fp8(w)
    for li in layers:
        cache_write_fp8(dw, li)
        out = run_decode_fp8(dw, li)
        decode_gate(out, whole_layer_oracle(w, li, fp8_scales=configs.fp8_scales(w)),
                    f"fp8 {w.name} layer {li}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    del dw
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layer", [0, 31])
def test_decode_fp8_workload5_whole_layer(layer):
    """Long-context skewed batch, FP8 caches: one whole layer's decode step,
    every output against the oracle, NaN codes in every dead slot."""
    w = configs.config5()
    dw = materialize_fp8(w, layers=[layer])
    poison_dead_slots_device_fp8(dw.key_caches[0], dw.value_caches[0],
                                 live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, w.block_size))
    cache_write_fp8(dw, 0)
    out = run_decode_fp8(dw, 0)
    decode_gate(out, whole_layer_oracle(w, layer, fp8_scales=configs.fp8_scales(w)),
                f"fp8 {w.name} layer {layer}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    del dw
    torch.cuda.empty_cache()


def test_decode_fp8_permutation_invariance_and_determinism():
    w = configs.config2()
    dw = materialize_fp8(w, layers=[0])
    a = run_decode_fp8(dw).clone()
    assert torch.equal(a.view(torch.int16), run_decode_fp8(dw).view(torch.int16))
    perm = torch.from_numpy(np.random.default_rng(2).permutation(w.num_blocks)).to(DEV)
    kc2 = torch.empty_like(dw.key_caches[0])
    vc2 = torch.empty_like(dw.value_caches[0])
    kc2[perm] = dw.key_caches[0]
    vc2[perm] = dw.value_caches[0]
    bt = dw.block_tables.long()
    dw.block_tables = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).int().contiguous()
    dw.key_caches[0], dw.value_caches[0] = kc2, vc2
    assert torch.equal(a.view(torch.int16), run_decode_fp8(dw).view(torch.int16))


def test_decode_fp8_single_token_is_scaled_code():
    """One token: the output is its value row, E4M3(code) * v_scale, rounded to fp16."""
    w = configs.small_random(2300, 5, 4, 128, 16, 1, min_context=1)
    dw = materialize_fp8(w)
    out = run_decode_fp8(dw)
    _, vs = configs.fp8_scales(w)
    vc = u8(dw.value_caches[0])
    for s in range(w.num_seqs):
        row = oracle.e4m3_to_double(vc[w.block_tables[s, 0], :, 0, :]) * np.float32(vs)
        expect = row.astype(np.float32).astype(np.float16)
        assert np.array_equal(out[s].cpu().numpy(), expect)


def test_decode_fp8_out_of_range_block_id_is_flagged():
    w = configs.small_random(2400, 3, 2, 64, 16, 80, min_context=40)
    w.block_tables[2, 0] = -7
    dw = materialize_fp8(w)
    run_decode_fp8(dw)
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits & pa.PA_ERRBIT_BLOCK_ID
    assert NAN8 == 0x7F


def test_decode_fp8_more_sequences_than_one_launch():
    """1100 sequences over two launches, forced 32-token partitions, every output."""
    pa.pa_decode_set_partition_tokens(32)
    w = configs.small_random(5300, 1100, 2, 128, 16, 100, min_context=0)
    dw = materialize_fp8(w)
    out = run_decode_fp8(dw)
    kc8, vc8 = oracle_fp8_pool(w)
    q = gpu.host_small(w, 0)[0]
    ks, vs = configs.fp8_scales(w)
    _, ref64, rc = oracle.decode_fp8(q, kc8, vc8, w.block_tables, w.context_lens, w.scale, ks, vs)
    assert rc == 0
    decode_gate(out, ref64, "fp8 S1100")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)

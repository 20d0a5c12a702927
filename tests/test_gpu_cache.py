"""GPU parity of the integer / byte paths, bit-exact against the oracle:
slot map, cache write, copy-on-write block copy; plus the generator's
device fill and the device error word."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa
from pa_testlib import u16
from workloads import configs, gpu, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_error_word():
    pa.pa_check_errors()
    yield
    torch.cuda.synchronize()


def test_generator_device_fill_matches_host():
    w = configs.small_random(3, 5, 4, 128, 16, 90)
    for layer in (0, 3):
        dw = gpu.materialize(w, layers=[layer], device=DEV)
        kc, vc = gpu.host_pool(w, layer)
        assert np.array_equal(u16(dw.key_caches[0]), kc)
        assert np.array_equal(u16(dw.value_caches[0]), vc)
    odd = torch.empty(1001, dtype=torch.float16, device=DEV)          # scalar (unvectorised) path
    gpu.fill(odd, 9, 5, gpu.device_bank(9, 1.0, DEV), start=77)
    assert np.array_equal(u16(odd), synth.host_values(9, 5, 77, 1001, synth.fp16_bank(9, 1.0)))


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_slot_mapping_bit_exact(cfg):
    w = configs.ALL[cfg]()
    seqs, pos = w.new_tokens()
    rng = np.random.default_rng(cfg)
    # plus random earlier positions of random sequences
    extra_s = rng.integers(0, w.num_seqs, 500).astype(np.int32)
    extra_p = np.array([rng.integers(0, max(1, w.context_lens[s])) for s in extra_s], dtype=np.int32)
    seqs = np.concatenate([seqs, extra_s]).astype(np.int32)
    pos = np.concatenate([pos, extra_p]).astype(np.int32)
    ref, rc = oracle.slot_mapping(w.block_tables, seqs, pos, w.block_size, w.num_blocks)
    assert rc == 0
    out = torch.empty(len(seqs), dtype=torch.int64, device=DEV)
    pa.pa_slot_mapping(out, torch.from_numpy(w.block_tables).to(DEV), torch.from_numpy(seqs).to(DEV),
                       torch.from_numpy(pos).to(DEV), w.block_size, w.num_blocks)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_slot_mapping_padding_and_range_errors():
    bt = torch.tensor([[3, 1, -1], [0, 7, 2]], dtype=torch.int32, device=DEV)
    seq = torch.tensor([-1, 0, 1, 5, 0, 1], dtype=torch.int32, device=DEV)
    pos = torch.tensor([0, 5, 9, 0, 13, 4], dtype=torch.int32, device=DEV)
    out = torch.empty(6, dtype=torch.int64, device=DEV)
    pa.pa_slot_mapping(out, bt, seq, pos, 4, 6)
    # padding; (0,5)->blk 1 off 1; (1,9)->blk 2 off 1; bad seq; pos past table; blk 7 >= NB
    assert out.cpu().tolist() == [-1, 5, 9, -1, -1, -1]
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_TOKEN
    assert pa.pa_check_errors() == (pa.PA_OK, 0)       # read clears the word


CACHE_SHAPES = [(d, b) for d in (64, 128) for b in (4, 8, 16, 32)]


@pytest.mark.parametrize("D,B", CACHE_SHAPES)
def test_reshape_and_cache_bit_exact_random(D, B):
    rng = np.random.default_rng(D * 100 + B)
    NB, H, T = 64, 3, 150
    kc = rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint64).astype(np.uint16)
    vc = rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint64).astype(np.uint16)
    k = rng.integers(0, 1 << 16, (T, H, D), dtype=np.uint64).astype(np.uint16)
    v = rng.integers(0, 1 << 16, (T, H, D), dtype=np.uint64).astype(np.uint16)
    slots = rng.permutation(NB * B)[:T].astype(np.int64)
    slots[rng.random(T) < 0.1] = -1
    dk, dv = (torch.from_numpy(x.view(np.int16)).to(DEV).view(torch.float16) for x in (kc, vc))
    tk, tv = (torch.from_numpy(x.view(np.int16)).to(DEV).view(torch.float16) for x in (k, v))
    pa.pa_reshape_and_cache(tk, tv, dk, dv, torch.from_numpy(slots).to(DEV))
    assert oracle.reshape_and_cache(kc, vc, k, v, slots, B) == 0
    assert np.array_equal(u16(dk), kc) and np.array_equal(u16(dv), vc)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_reshape_and_cache_workload_bit_exact(cfg):
    """The decode step's cache write at full size (workload 3: one layer)."""
    w = configs.ALL[cfg]()
    dw = gpu.materialize(w, layers=[0], device=DEV)
    T = dw.token_seq.numel()
    slots = torch.empty(T, dtype=torch.int64, device=DEV)
    pa.pa_slot_mapping(slots, dw.block_tables, dw.token_seq, dw.token_pos, w.block_size, w.num_blocks)
    pa.pa_reshape_and_cache(dw.keys_new[0], dw.values_new[0], dw.key_caches[0], dw.value_caches[0], slots)
    kc, vc = gpu.host_pool(w, 0)
    _, kn, vn = gpu.host_small(w, 0)
    seqs, pos = w.new_tokens()
    ref_slots, _ = oracle.slot_mapping(w.block_tables, seqs, pos, w.block_size, w.num_blocks)
    assert oracle.reshape_and_cache(kc, vc, kn, vn, ref_slots, w.block_size) == 0
    assert np.array_equal(u16(dw.key_caches[0]), kc)
    assert np.array_equal(u16(dw.value_caches[0]), vc)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_reshape_and_cache_empty_and_bad_slot():
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.ones((2, 2, 64), dtype=torch.float16, device=DEV)
    pa.pa_reshape_and_cache(k[:0], k[:0], kc, vc, torch.empty(0, dtype=torch.int64, device=DEV))
    pa.pa_reshape_and_cache(k, k, kc, vc, torch.tensor([5, 64], dtype=torch.int64, device=DEV))
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_SLOT
    assert kc[0, :, 5].eq(1).all() and kc.sum().item() == 2 * 64     # the good token landed alone


@pytest.mark.parametrize("layers", [1, 3, 33])
@pytest.mark.parametrize("D,B", [(128, 16), (64, 4), (128, 32)])
def test_copy_blocks_bit_exact(layers, D, B):
    rng = np.random.default_rng(layers * 7 + B)
    NB, H = 24, 3
    kcs = [rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint64).astype(np.uint16) for _ in range(layers)]
    vcs = [rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint64).astype(np.uint16) for _ in range(layers)]
    ids = rng.permutation(NB)
    pairs = np.stack([ids[:7], ids[7:14]], axis=1).astype(np.int64)
    dk = [torch.from_numpy(x.view(np.int16)).to(DEV).view(torch.float16) for x in kcs]
    dv = [torch.from_numpy(x.view(np.int16)).to(DEV).view(torch.float16) for x in vcs]
    pa.pa_copy_blocks(dk, dv, torch.from_numpy(pairs).to(DEV))
    assert oracle.copy_blocks(kcs, vcs, pairs) == 0
    for l in range(layers):
        assert np.array_equal(u16(dk[l]), kcs[l]) and np.array_equal(u16(dv[l]), vcs[l])
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_copy_blocks_bad_pair_is_skipped():
    kc = torch.arange(4 * 2 * 4 * 64, device=DEV).to(torch.float16).view(4, 2, 4, 64)
    vc = kc.clone()
    before = kc.clone()
    pairs = torch.tensor([[0, 9], [1, 2]], dtype=torch.int64, device=DEV)
    pa.pa_copy_blocks([kc], [vc], pairs)
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_COPY
    expect = before.clone()
    expect[2] = before[1]
    assert torch.equal(kc, expect) and torch.equal(vc, expect)

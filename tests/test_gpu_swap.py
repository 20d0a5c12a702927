"""GPU parity of the block swap between the device pool and a pinned host
pool: swap-out and swap-in bit-exact against the oracle, for fp16 and FP8
caches, with the block mapping in device or pinned host memory; bad ids are
flagged and skipped; host memory the device cannot reach is refused."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean():
    pa.pa_check_errors()
    yield
    torch.cuda.synchronize()


def host_view(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu().contiguous()
    return a.view(torch.uint8).numpy().reshape(a.shape[0], -1).copy()


def pools(rng, layers, nb_dev, nb_host, shape, dtype):
    dev = []
    for _ in range(2 * layers):
        raw = rng.integers(0, 1 << 16, (nb_dev,) + shape, dtype=np.uint16)
        t = torch.from_numpy(raw.view(np.int16)).to(DEV)
        dev.append(t.view(torch.float16) if dtype == torch.float16 else t.view(torch.uint8)
                   .view((nb_dev,) + shape[:-1] + (2 * shape[-1],)))
    host = [torch.zeros((nb_host,) + tuple(dev[0].shape[1:]), dtype=dev[0].dtype).pin_memory()
            for _ in range(2 * layers)]
    return dev, host


@pytest.mark.parametrize("dtype,map_on_device", [(torch.float16, True), (torch.uint8, False)])
def test_swap_out_and_in_bit_exact(dtype, map_on_device):
    rng = np.random.default_rng(7 if map_on_device else 8)
    layers, nb_dev, nb_host = 3, 40, 25
    shape = (4, 16, 64)                      # H, B, D (uint8 caches: D doubles)
    dev, host = pools(rng, layers, nb_dev, nb_host, shape, dtype)
    ref_dev = [host_view(t) for t in dev]
    ref_host = [host_view(t) for t in host]

    out_map = np.stack([rng.choice(nb_dev, 12, replace=False), rng.choice(nb_host, 12, replace=False)],
                       axis=1).astype(np.int64)
    m = torch.from_numpy(out_map)
    m = m.to(DEV) if map_on_device else m.pin_memory()
    pa.pa_swap_blocks(host, dev, m)
    torch.cuda.synchronize()
    assert oracle.swap_blocks(ref_host, ref_dev, out_map) == 0
    for t, r in zip(host, ref_host):
        assert np.array_equal(host_view(t), r)

    # swap in to other device blocks (the ones not swapped out)
    free = np.setdiff1d(np.arange(nb_dev), out_map[:, 0])
    in_map = np.stack([out_map[:, 1], rng.choice(free, 12, replace=False)], axis=1).astype(np.int64)
    m = torch.from_numpy(in_map)
    m = m.to(DEV) if map_on_device else m.pin_memory()
    pa.pa_swap_blocks(dev, host, m)
    torch.cuda.synchronize()
    assert oracle.swap_blocks(ref_dev, ref_host, in_map) == 0
    for t, r in zip(dev, ref_dev):
        assert np.array_equal(host_view(t), r)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_swap_bad_id_is_flagged_and_skipped():
    rng = np.random.default_rng(9)
    dev, host = pools(rng, 1, 10, 6, (2, 8, 64), torch.float16)
    ref_dev = [host_view(t) for t in dev]
    ref_host = [host_view(t) for t in host]
    mapping = np.array([[1, 0], [10, 1], [2, 6], [3, 5]], dtype=np.int64)
    pa.pa_swap_blocks(host, dev, torch.from_numpy(mapping).to(DEV))
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_COPY
    assert oracle.swap_blocks(ref_host, ref_dev, mapping) == -1
    for t, r in zip(host, ref_host):
        assert np.array_equal(host_view(t), r)


def test_swap_refuses_pageable_host_memory():
    dev = torch.zeros((4, 2, 8, 64), dtype=torch.float16, device=DEV)
    pageable = np.zeros((4, 2, 8, 64), dtype=np.float16)
    mapping = torch.tensor([[0, 1]], dtype=torch.int64, device=DEV)
    lib = ctypes.CDLL(pa.LIB_PATH)
    vp = ctypes.c_void_p
    lib.pa_swap_blocks.argtypes = [vp, vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_size_t,
                                   ctypes.c_int64, ctypes.c_int64, vp]
    dst = (ctypes.c_void_p * 1)(pageable.ctypes.data)
    src = (ctypes.c_void_p * 1)(dev.data_ptr())
    assert lib.pa_swap_blocks(dst, src, 1, mapping.data_ptr(), 1, 2 * 8 * 64 * 2, 4, 4, None) == \
        pa.PA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        pa.pa_swap_blocks([torch.zeros_like(dev).cpu()], [dev], mapping)


def test_swap_duplicate_destinations_are_skipped_and_flagged():
    rng = np.random.default_rng(10)
    dev, host = pools(rng, 1, 10, 6, (2, 8, 64), torch.float16)
    ref_host = [host_view(t) for t in host]
    ref_dev = [host_view(t) for t in dev]
    mapping = np.array([[1, 2], [4, 2], [5, 0]], dtype=np.int64)   # pairs 0 and 1 share destination 2
    pa.pa_swap_blocks(host, dev, torch.from_numpy(mapping).to(DEV))
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_COPY
    for t, r, d in zip(host, ref_host, ref_dev):
        expect = r.copy()
        expect[0] = d[5]
        assert np.array_equal(host_view(t), expect)


def test_block_manager_swap_round_trip_keeps_decode_bits():
    """Decode, swap a sequence out with the block manager's pairs, let another
    sequence overwrite the freed GPU blocks, swap it back into different
    blocks, decode again: every output is bit-identical (decode depends only
    on logical positions)."""
    from paged_kv_cache_158_gb300.pool import BlockManager
    from workloads import configs as cfgs, gpu as wgpu
    rng = np.random.default_rng(21)
    S, H, D, B, NB, NH = 4, 4, 128, 16, 64, 32
    bm = BlockManager(NB, B, S + 1, 16, free_order=rng.permutation(NB), num_host_blocks=NH)
    lens = [100, 130, 37, 200]
    for s, n in enumerate(lens):
        bm.add_sequence(s)
        bm.append_tokens(s, n)
    w = cfgs.small_random(2500, S, H, D, B, 8)   # only for its value streams and bank
    bank = wgpu.device_bank(w.seed, w.kv_sigma, DEV)
    kc = torch.empty((NB, H, B, D), dtype=torch.float16, device=DEV)
    vc = torch.empty_like(kc)
    wgpu.fill(kc, w.seed, 0, bank)
    wgpu.fill(vc, w.seed, 1, bank)
    torch.manual_seed(21)
    q = torch.randn((S, H, D), device=DEV).half()
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    ws = pa.decode_workspace(S, H, D, max(lens))

    def decode():
        out = torch.empty((S, H, D), dtype=torch.float16, device=DEV)
        bt = torch.from_numpy(bm.block_tables(np.arange(S))).to(DEV)
        pa.pa_decode(out, q, kc, vc, bt, ctx, 0.088, max(lens), ws)
        return out

    before = decode().clone()
    host_k = torch.zeros((NH, H, B, D), dtype=torch.float16).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    out_pairs = bm.swap_out(1)
    pa.pa_swap_blocks([host_k, host_v], [kc, vc], torch.from_numpy(out_pairs).to(DEV))
    bm.add_sequence(S)                                  # reuses the freed blocks
    bm.append_tokens(S, B * min(bm.num_free() // 2, 16))
    reused = torch.from_numpy(bm.tables[S, :int(bm.nblocks[S])].astype(np.int64)).to(DEV)
    kc[reused] = float("nan")
    vc[reused] = float("nan")
    in_pairs = bm.swap_in(1)
    assert not np.array_equal(np.sort(in_pairs[:, 1]), np.sort(out_pairs[:, 0]))  # new blocks
    pa.pa_swap_blocks([kc, vc], [host_k, host_v], torch.from_numpy(in_pairs).to(DEV))
    after = decode()
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), after.view(torch.int16))
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_swap_more_caches_and_pairs_than_one_launch():
    """70 caches (the kernel takes 64 per launch) and, on one cache, 70 000 pairs (at most
    65 535 per launch): every block lands where the oracle puts it."""
    rng = np.random.default_rng(31)
    dev, host = pools(rng, 35, 12, 8, (1, 4, 64), torch.float16)
    ref_dev = [host_view(t) for t in dev]
    ref_host = [host_view(t) for t in host]
    mapping = np.stack([rng.choice(12, 8, replace=False), rng.permutation(8)], 1).astype(np.int64)
    pa.pa_swap_blocks(host, dev, torch.from_numpy(mapping).to(DEV))
    torch.cuda.synchronize()
    assert oracle.swap_blocks(ref_host, ref_dev, mapping) == 0
    for t, r in zip(host, ref_host):
        assert np.array_equal(host_view(t), r)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)

    n = 70_000
    d_pool = torch.from_numpy(rng.integers(0, 1 << 16, (n, 1, 4, 64), dtype=np.uint16)
                              .view(np.int16)).to(DEV).view(torch.float16)
    h_pool = torch.zeros((n, 1, 4, 64), dtype=torch.float16).pin_memory()
    big = np.stack([rng.permutation(n), rng.permutation(n)], 1).astype(np.int64)
    pa.pa_swap_blocks([h_pool], [d_pool], torch.from_numpy(big).to(DEV))
    torch.cuda.synchronize()
    ref = [host_view(h_pool)]
    expect = np.zeros_like(ref[0])
    expect[big[:, 1]] = host_view(d_pool)[big[:, 0]]
    assert np.array_equal(ref[0], expect)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_swap_large_mapping_duplicate_destination():
    """1300 pairs (above the 1024 where each CTA copies one cache): with the
    mapping on the device, the two pairs sharing a destination are skipped and
    flagged and the rest move; the same mapping in pinned host memory is
    refused on the host before anything launches."""
    rng = np.random.default_rng(11)
    P = 1300
    dev, host = pools(rng, 2, 1400, 1350, (1, 4, 64), torch.float16)
    ref_host = [host_view(t) for t in host]
    ref_dev = [host_view(t) for t in dev]
    mapping = np.stack([rng.permutation(1400)[:P], rng.permutation(1350)[:P]], 1).astype(np.int64)
    mapping[1000, 1] = mapping[77, 1]
    with pytest.raises(pa.PAError) as e:
        pa.pa_swap_blocks(host, dev, torch.from_numpy(mapping).pin_memory())
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    for t, r in zip(host, ref_host):
        assert np.array_equal(host_view(t), r)
    pa.pa_swap_blocks(host, dev, torch.from_numpy(mapping).to(DEV))
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_COPY
    for t, r, d in zip(host, ref_host, ref_dev):
        expect = r.copy()
        for p in range(P):
            if p not in (77, 1000):
                expect[mapping[p, 1]] = d[mapping[p, 0]]
        assert np.array_equal(host_view(t), expect)

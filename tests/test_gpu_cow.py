"""Shared-prefix workload with copy-on-write, end to end on the GPU: the
product block manager plans, the GPU copies blocks, maps slots, writes the
suffix tokens and decodes.  The oracle replays the pages' block manager on
its own and runs its own copy / slot map / cache write / decode on the host.
Pools must match bit for bit, outputs within tolerance; decoding with the
prefix shared must give the same bits as with private copies."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa
from oracle.block_model import shared_prefix_flow
from pa_testlib import decode_gate, u16
from paged_kv_cache_158_gb300.pool import BlockManager
from workloads import configs, gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def product_plan(w):
    bm = BlockManager(w.num_blocks, w.block_size, w.num_seqs, w.max_blocks_per_seq, w.free_order)
    bm.add_sequence(0)
    bm.append_tokens(0, w.prefix_len)
    for s in range(1, w.num_seqs):
        bm.fork(0, s)
    for s in range(w.num_seqs):
        bm.append_tokens(s, int(w.suffix_lens[s]))
    return bm.take_copies(), bm.block_tables(), bm.context_lens()


def gpu_step(w, dw, pairs, bt, ctx):
    bt_d = torch.from_numpy(bt).to(DEV)
    ctx_d = torch.from_numpy(ctx).to(DEV)
    pa.pa_copy_blocks(dw.key_caches, dw.value_caches, torch.from_numpy(pairs).to(DEV))
    slots = torch.empty(dw.token_seq.numel(), dtype=torch.int64, device=DEV)
    pa.pa_slot_mapping(slots, bt_d, dw.token_seq, dw.token_pos, w.block_size, w.num_blocks)
    pa.pa_reshape_and_cache(dw.keys_new[0], dw.values_new[0], dw.key_caches[0], dw.value_caches[0], slots)
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float16, device=DEV)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, int(ctx.max()))
    pa.pa_decode(out, dw.queries[0], dw.key_caches[0], dw.value_caches[0], bt_d, ctx_d, w.scale,
                 int(ctx.max()), ws)
    return out


def test_shared_prefix_copy_on_write_against_oracle():
    w = configs.config4()
    pairs, bt, ctx = product_plan(w)
    assert pairs.shape == (w.num_seqs - 1, 2)
    dw = gpu.materialize(w, device=DEV)
    out = gpu_step(w, dw, pairs, bt, ctx)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)

    model, appended = shared_prefix_flow(w.num_seqs, w.prefix_len, w.suffix_lens, w.num_blocks,
                                         w.block_size, w.free_order)
    mbt = model.table_array(range(w.num_seqs), w.max_blocks_per_seq)
    kc, vc = gpu.host_pool(w, 0)
    q, kn, vn = gpu.host_small(w, 0)
    assert oracle.copy_blocks([kc], [vc], np.array(model.copies, dtype=np.int64)) == 0
    seqs = np.array([s for s, _ in appended], dtype=np.int32)
    pos = np.array([p for _, p in appended], dtype=np.int32)
    slots, rc = oracle.slot_mapping(mbt, seqs, pos, w.block_size, w.num_blocks)
    assert rc == 0
    assert oracle.reshape_and_cache(kc, vc, kn, vn, slots, w.block_size) == 0
    assert np.array_equal(u16(dw.key_caches[0]), kc)
    assert np.array_equal(u16(dw.value_caches[0]), vc)
    mctx = np.array([model.lengths[s] for s in range(w.num_seqs)], dtype=np.int32)
    _, ref64, rc = oracle.decode(q, kc, vc, mbt, mctx, w.scale)
    assert rc == 0
    decode_gate(out, ref64, w.name)


def test_shared_prefix_identity_bit_exact():
    """Same bits whether the 32 full prefix blocks are shared by reference or
    every sequence holds private copies of them."""
    w = configs.config4()
    pairs, bt, ctx = product_plan(w)
    dw = gpu.materialize(w, device=DEV)
    shared = gpu_step(w, dw, pairs, bt, ctx).clone()
    full = w.prefix_len // w.block_size
    S = w.num_seqs
    NB = w.num_blocks
    kc = torch.cat([dw.key_caches[0], torch.empty((S * full,) + tuple(dw.key_caches[0].shape[1:]),
                                                  dtype=torch.float16, device=DEV)])
    vc = torch.cat([dw.value_caches[0], torch.empty_like(kc[NB:])])
    bt2 = bt.copy()
    src = torch.from_numpy(bt[0, :full].astype(np.int64)).to(DEV)
    for s in range(S):
        ids = np.arange(NB + s * full, NB + (s + 1) * full)
        kc[torch.from_numpy(ids).to(DEV)] = kc[src]
        vc[torch.from_numpy(ids).to(DEV)] = vc[src]
        bt2[s, :full] = ids
    out = torch.empty_like(shared)
    ws = pa.decode_workspace(S, w.num_heads, w.head_dim, int(ctx.max()))
    pa.pa_decode(out, dw.queries[0], kc, vc, torch.from_numpy(bt2).to(DEV), torch.from_numpy(ctx).to(DEV),
                 w.scale, int(ctx.max()), ws)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    assert torch.equal(shared.view(torch.int16), out.view(torch.int16))


def test_copy_blocks_conflicting_pairs_are_skipped_and_flagged():
    """A pair whose destination is another pair's destination or source is not
    copied (nothing races) and the copy error bit is set; other pairs copy."""
    rng = np.random.default_rng(12)
    NB, H, B, D = 12, 2, 16, 64
    kc = torch.from_numpy(rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint16).view(np.int16)).cuda()
    vc = torch.from_numpy(rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint16).view(np.int16)).cuda()
    kc, vc = kc.view(torch.float16), vc.view(torch.float16)
    before_k, before_v = u16(kc).copy(), u16(vc).copy()
    # pairs 0 and 1 share destination 5; pair 2 writes 3, which pair 3 reads; pair 4 is clean
    mapping = np.array([[0, 5], [1, 5], [2, 3], [3, 7], [8, 9]], dtype=np.int64)
    pa.pa_check_errors()
    pa.pa_copy_blocks([kc], [vc], torch.from_numpy(mapping).cuda())
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_COPY
    ek, ev = before_k.copy(), before_v.copy()
    for src, dst in ([3, 7], [8, 9]):          # the pairs without a conflict
        ek[dst], ev[dst] = before_k[src], before_v[src]
    assert np.array_equal(u16(kc), ek) and np.array_equal(u16(vc), ev)


def _random_caches(rng, layers, NB, H, B, D):
    out = []
    for _ in range(2 * layers):
        raw = rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint16)
        out.append(torch.from_numpy(raw.view(np.int16)).cuda().view(torch.float16))
    return out[:layers], out[layers:]


def test_copy_blocks_large_mapping_conflicts_are_skipped_and_flagged():
    """1500 pairs over 3 layers (above the 1024 pairs where each CTA copies one
    cache): a repeated destination skips both of its pairs, a destination that
    is another pair's source skips the writing pair, every other pair copies
    exactly once."""
    rng = np.random.default_rng(13)
    P, NB, H, B, D, L = 1500, 3200, 1, 4, 64, 3
    kcs, vcs = _random_caches(rng, L, NB, H, B, D)
    before = [u16(t).copy() for t in kcs + vcs]
    src = rng.permutation(1500).astype(np.int64)
    dst = (1500 + rng.permutation(1500)).astype(np.int64)
    mapping = np.stack([src, dst], 1)
    mapping[700, 1] = mapping[900, 1]          # pairs 700 and 900 share a destination
    mapping[1200, 1] = mapping[5, 0]           # pair 1200 writes the block pair 5 reads
    skipped = {700, 900, 1200}
    pa.pa_copy_blocks(kcs, vcs, torch.from_numpy(mapping).to(DEV))
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_COPY
    for t, b in zip(kcs + vcs, before):
        expect = b.copy()
        for p in range(P):
            if p not in skipped:
                expect[mapping[p, 1]] = b[mapping[p, 0]]
        assert np.array_equal(u16(t), expect)


def test_copy_blocks_pinned_mapping_checked_on_host():
    """A mapping in pinned host memory is checked before anything launches:
    a repeated destination (here among 2000 pairs) or a destination that is
    another pair's source is refused with PA_ERR_INVALID_ARG and the caches are
    unchanged; a clean pinned mapping copies like a device one."""
    rng = np.random.default_rng(14)
    P, NB, H, B, D = 2000, 4100, 1, 4, 64
    kcs, vcs = _random_caches(rng, 1, NB, H, B, D)
    before = [u16(t).copy() for t in kcs + vcs]
    src = rng.permutation(2000).astype(np.int64)
    dst = (2000 + rng.permutation(2000)).astype(np.int64)
    clean = np.stack([src, dst], 1)
    for bad_row, bad_col, value in ((1999, 1, clean[3, 1]), (17, 1, clean[40, 0])):
        bad = clean.copy()
        bad[bad_row, bad_col] = value
        with pytest.raises(pa.PAError) as e:
            pa.pa_copy_blocks(kcs, vcs, torch.from_numpy(bad).pin_memory())
        assert e.value.status == pa.PA_ERR_INVALID_ARG
        torch.cuda.synchronize()
        for t, b in zip(kcs + vcs, before):
            assert np.array_equal(u16(t), b)
    pa.pa_copy_blocks(kcs, vcs, torch.from_numpy(clean).pin_memory())
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    for t, b in zip(kcs + vcs, before):
        expect = b.copy()
        expect[clean[:, 1]] = b[clean[:, 0]]
        assert np.array_equal(u16(t), expect)
    with pytest.raises(ValueError):            # pageable host memory: the device cannot reach it
        pa.pa_copy_blocks(kcs, vcs, torch.from_numpy(clean))

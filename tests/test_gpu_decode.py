"""GPU parity of paged decode against the oracle, element by element on
small and mid-size inputs (several tiles, ragged tails, many partitions)
and on whole layers of the full-size workloads in the benchmark's launch
configuration; plus the invariants the pages fix (permutation of physical
blocks, run-to-run determinism) and edge cases."""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa
from pa_testlib import (decode_gate, live_slot_mask, poison_dead_slots_device, poison_dead_slots_host,
                        u16, whole_layer_oracle)
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


def run_decode(dw, layer_idx=0, out=None):
    w = dw.w
    out = out if out is not None else torch.empty((w.num_seqs, w.num_heads, w.head_dim),
                                                  dtype=torch.float16, device=DEV)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    pa.pa_decode(out, dw.queries[layer_idx], dw.key_caches[layer_idx], dw.value_caches[layer_idx],
                 dw.block_tables, dw.context_lens, w.scale, w.max_context_len, ws)
    return out


def cache_write(dw, layer_idx=0):
    w = dw.w
    slots = torch.empty(dw.token_seq.numel(), dtype=torch.int64, device=DEV)
    pa.pa_slot_mapping(slots, dw.block_tables, dw.token_seq, dw.token_pos, w.block_size, w.num_blocks)
    pa.pa_reshape_and_cache(dw.keys_new[layer_idx], dw.values_new[layer_idx], dw.key_caches[layer_idx],
                            dw.value_caches[layer_idx], slots)


def full_oracle(w, layer=0, poison=True, write_new=True):
    kc, vc = gpu.host_pool(w, layer)
    q, kn, vn = gpu.host_small(w, layer)
    if write_new:
        seqs, pos = w.new_tokens()
        slots, rc = oracle.slot_mapping(w.block_tables, seqs, pos, w.block_size, w.num_blocks)
        assert rc == 0
        assert oracle.reshape_and_cache(kc, vc, kn, vn, slots, w.block_size) == 0
    if poison:
        poison_dead_slots_host(kc, vc, live_slot_mask(w.block_tables, w.context_lens, w.num_blocks,
                                                      w.block_size))
    return oracle.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)


SMALL = [(d, b) for d in (64, 128) for b in (4, 8, 16, 32)]


@pytest.mark.parametrize("part", [0, 32, 96])
@pytest.mark.parametrize("D,B", SMALL)
def test_decode_small_random(D, B, part):
    """Ragged contexts (including 0 and 1), NaN in every dead slot, forced
    small partitions so several partitions and the merge kernel run."""
    pa.pa_decode_set_partition_tokens(part)
    w = configs.small_random(1000 + D + B + part, 7, 3, D, B, 300, min_context=0)
    w.context_lens[0], w.context_lens[1] = 0, 1
    w.block_tables[0, :] = -1
    dw = gpu.materialize(w, device=DEV)
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, B)
    poison_dead_slots_device(dw.key_caches[0], dw.value_caches[0], mask)
    out = run_decode(dw)
    _, ref64, rc = full_oracle(w, write_new=False)
    assert rc == 0
    decode_gate(out, ref64, f"D{D} B{B} part{part}")
    assert u16(out)[0].max() == 0                      # empty context: zero row
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("cfg", [1, 2])
def test_decode_step_workload_all_outputs(cfg):
    """Slot map + cache write + decode of workloads 1 and 2, every output."""
    w = configs.ALL[cfg]()
    dw = gpu.materialize(w, device=DEV)
    poison_dead_slots_device(dw.key_caches[0], dw.value_caches[0],
                             live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, w.block_size))
    cache_write(dw)
    out = run_decode(dw)
    _, ref64, rc = full_oracle(w)
    assert rc == 0
    decode_gate(out, ref64, w.name)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("layers", [(0, 13), (26, 39)])
def test_decode_workload3_whole_layers(layers):
    """LLaMA-13B shape at full size (all 40 layers resident), the bench's launch
    configuration: the decode step (slot map, cache write, decode) of whole
    layers, every output against the oracle."""
    w = configs.config3()
    dw = gpu.materialize(w, device=DEV)
    for li in layers:
        cache_write(dw, li)
        out = run_decode(dw, li)
        decode_gate(out, whole_layer_oracle(w, li), f"{w.name} layer {li}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    del dw
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layer", [0, 31])
def test_decode_workload5_whole_layer(layer):
    """Long-context skewed batch at full size per layer (3.2 GB of K/V, 256
    sequences of 16..4096 tokens), the bench's launch configuration: one whole
    layer's decode step, every output against the oracle, NaN in every dead
    slot on both sides."""
    w = configs.config5()
    dw = gpu.materialize(w, layers=[layer], device=DEV)
    poison_dead_slots_device(dw.key_caches[0], dw.value_caches[0],
                             live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, w.block_size))
    cache_write(dw, 0)
    out = run_decode(dw, 0)
    decode_gate(out, whole_layer_oracle(w, layer), f"{w.name} layer {layer}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    del dw
    torch.cuda.empty_cache()


def test_decode_permutation_invariance_bit_exact():
    w = configs.config2()
    dw = gpu.materialize(w, device=DEV)
    a = run_decode(dw).clone()
    perm = torch.from_numpy(np.random.default_rng(1).permutation(w.num_blocks)).to(DEV)
    kc2 = torch.empty_like(dw.key_caches[0])
    vc2 = torch.empty_like(dw.value_caches[0])
    kc2[perm] = dw.key_caches[0]
    vc2[perm] = dw.value_caches[0]
    bt = dw.block_tables.long()
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).int()
    dw.key_caches[0], dw.value_caches[0], dw.block_tables = kc2, vc2, bt2.contiguous()
    b = run_decode(dw)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_decode_run_to_run_deterministic():
    w = configs.config5(num_layers=1)
    dw = gpu.materialize(w, device=DEV)
    a = run_decode(dw).clone()
    for _ in range(3):
        assert torch.equal(a.view(torch.int16), run_decode(dw).view(torch.int16))


def test_decode_single_token_returns_value_bits():
    w = configs.small_random(77, 6, 4, 128, 16, 1, min_context=1)
    dw = gpu.materialize(w, device=DEV)
    out = run_decode(dw)
    vc = u16(dw.value_caches[0])
    for s in range(w.num_seqs):
        assert np.array_equal(u16(out)[s], vc[w.block_tables[s, 0], :, 0, :])


def test_decode_out_of_range_block_id_is_flagged_not_fatal():
    w = configs.small_random(78, 3, 2, 128, 16, 80, min_context=40)
    w.block_tables[1, 1] = w.num_blocks + 5
    dw = gpu.materialize(w, device=DEV)
    run_decode(dw)
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits & pa.PA_ERRBIT_BLOCK_ID
    # the other sequences are unaffected
    out = run_decode(dw)
    pa.pa_check_errors()
    clean_bt = w.block_tables.copy()
    clean_bt[1, :] = 0
    q = gpu.host_small(w, 0)[0]
    kc, vc = gpu.host_pool(w, 0)
    _, ref64, _ = oracle.decode(q, kc, vc, clean_bt, w.context_lens, w.scale)
    for s in (0, 2):
        decode_gate(out[s:s + 1], ref64[s:s + 1], "unaffected sequence")


def test_decode_context_beyond_max_is_clipped_and_flagged():
    w = configs.small_random(79, 2, 2, 64, 16, 64, min_context=64)
    dw = gpu.materialize(w, device=DEV)
    out = torch.empty((2, 2, 64), dtype=torch.float16, device=DEV)
    ws = pa.decode_workspace(2, 2, 64, 48)
    pa.pa_decode(out, dw.queries[0], dw.key_caches[0], dw.value_caches[0], dw.block_tables,
                 dw.context_lens, w.scale, 48, ws)
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits == pa.PA_ERRBIT_CONTEXT
    q = gpu.host_small(w, 0)[0]
    kc, vc = gpu.host_pool(w, 0)
    _, ref64, _ = oracle.decode(q, kc, vc, w.block_tables, np.full(2, 48, np.int32), w.scale)
    decode_gate(out, ref64, "clipped to max_context_len")


@pytest.mark.parametrize("part", [0, 32])
def test_decode_more_sequences_than_one_launch(part):
    """1100 sequences (the call splits them over two launches of at most 1024, each with its own
    item numbering and the shared workspace), ragged and empty contexts, every output."""
    pa.pa_decode_set_partition_tokens(part)
    w = configs.small_random(5100 + part, 1100, 2, 64, 16, 100, min_context=0)
    dw = gpu.materialize(w, device=DEV)
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, 16)
    poison_dead_slots_device(dw.key_caches[0], dw.value_caches[0], mask)
    out = run_decode(dw)
    _, ref64, rc = full_oracle(w, write_new=False)
    assert rc == 0
    decode_gate(out, ref64, f"S1100 part{part}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("part", [0, 32])
def test_decode_long_contexts_many_partitions(part):
    """Contexts up to 20 000 tokens: 79 partitions of 256 (the default for so small a batch),
    or 625 of 32 (the merge walks its partials in rounds of 32), every output."""
    pa.pa_decode_set_partition_tokens(part)
    w = configs.small_random(5200 + part, 3, 2, 128, 32, 20000, min_context=15000)
    dw = gpu.materialize(w, device=DEV)
    out = run_decode(dw)
    _, ref64, rc = full_oracle(w, poison=False, write_new=False)
    assert rc == 0
    decode_gate(out, ref64, f"long contexts part{part}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_bounded_wait_gives_up_and_reports_timeout():
    """A kernel whose bounded wait never completes (a barrier that gets one of its two
    arrivals) ends after about a second with the timeout bit in the device error word; the
    word clears on reading and the context stays usable: a decode afterwards matches the
    oracle."""
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pa.pa_selftest_wait_timeout()
    st, bits = pa.pa_check_errors()
    dt = time.perf_counter() - t0
    assert (st, bits) == (pa.PA_ERR_TIMEOUT, pa.PA_ERRBIT_TIMEOUT)
    assert 0.9 < dt < 10.0
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    w = configs.small_random(4242, 5, 3, 128, 16, 200, min_context=1)
    dw = gpu.materialize(w, device=DEV)
    out = run_decode(dw)
    _, ref64, rc = full_oracle(w, write_new=False)
    assert rc == 0
    decode_gate(out, ref64, "decode after a timed-out wait")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("part", [0, 32])
def test_zeroed_workspace_flag_matches_default_and_keeps_counters_zero(part, fp8):
    """PA_DECODE_ZEROED_WORKSPACE: five calls in a row on one zero-filled
    workspace (1100 sequences: two launches, two work counters) give the same
    bits as the default call, and every call leaves the counters zero."""
    from pa_testlib import materialize_fp8
    pa.pa_decode_set_partition_tokens(part)
    w = configs.small_random(5400 + part + fp8, 1100, 2, 128, 16, 200, min_context=0)
    dw = materialize_fp8(w) if fp8 else gpu.materialize(w, device=DEV)
    ks, vs = configs.fp8_scales(w)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    ws_ref = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    args = (dw.queries[0], dw.key_caches[0], dw.value_caches[0], dw.block_tables, dw.context_lens,
            w.scale)
    ref = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float16, device=DEV)
    if fp8:
        pa.pa_decode_fp8(ref, *args, ks, vs, w.max_context_len, ws_ref)
    else:
        pa.pa_decode(ref, *args, w.max_context_len, ws_ref)
    for _ in range(5):
        out = torch.full_like(ref, float("nan"))
        if fp8:
            pa.pa_decode_fp8_ex(out, *args, ks, vs, w.max_context_len, ws,
                                pa.PA_DECODE_ZEROED_WORKSPACE)
        else:
            pa.pa_decode_ex(out, *args, w.max_context_len, ws, pa.PA_DECODE_ZEROED_WORKSPACE)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert int(ws[:8].view(torch.int32).abs().sum()) == 0    # both launches' counters
    assert int(ws_ref[:8].view(torch.int32).abs().sum()) == 0
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_decode_ex_refuses_unknown_flags():
    w = configs.small_random(5500, 3, 2, 64, 16, 40)
    dw = gpu.materialize(w, device=DEV)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float16, device=DEV)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_ex(out, dw.queries[0], dw.key_caches[0], dw.value_caches[0], dw.block_tables,
                        dw.context_lens, w.scale, w.max_context_len, ws, 0x4)
    assert e.value.status == pa.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("append", [False, True])
def test_zeroed_workspace_decode_sees_the_swap_in_just_before_it(append):
    """With PA_DECODE_ZEROED_WORKSPACE the decode kernel is the call's first
    and is launched programmatically behind the previous kernel on the
    stream, which may still be running when it starts.  Here that kernel is a
    swap-in of every sequence's only block from pinned host memory (the first
    sequences' blocks last in the mapping, so they are still on their way
    when the decode could start).  Ten rounds, each putting the old blocks
    back first, give the bits of the same call made after a synchronize: the
    outputs, and with append (the decode writes position 15 itself) the
    caches too, whose new rows must not be overwritten by the swap-in."""
    S, H, D, B = 512, 8, 128, 16
    gen = torch.Generator().manual_seed(5600 + append)
    rnd = lambda *shape: torch.randn(*shape, generator=gen).to(torch.float16)  # noqa: E731
    k_old, v_old = rnd(S, H, B, D).to(DEV), rnd(S, H, B, D).to(DEV)
    hk, hv = rnd(S, H, B, D).pin_memory(), rnd(S, H, B, D).pin_memory()
    q, k_app, v_app = (rnd(S, H, D).to(DEV) for _ in range(3))
    rows = torch.arange(S - 1, -1, -1, dtype=torch.int64)
    mapping = torch.stack([rows, rows], dim=1).contiguous().to(DEV)
    kc, vc = torch.empty_like(k_old), torch.empty_like(v_old)
    bt = torch.arange(S, dtype=torch.int32, device=DEV).view(S, 1)
    ctx = torch.full((S,), B, dtype=torch.int32, device=DEV)
    ws = pa.decode_workspace(S, H, D, B)
    scale = D ** -0.5

    def step(out, flags, sync):
        kc.copy_(k_old)
        vc.copy_(v_old)
        pa.pa_swap_blocks([kc, vc], [hk, hv], mapping)
        if sync:
            torch.cuda.synchronize()
        if append:
            pa.pa_decode_append(out, q, k_app, v_app, kc, vc, bt, ctx, scale, B, ws, flags)
        else:
            pa.pa_decode_ex(out, q, kc, vc, bt, ctx, scale, B, ws, flags)
        torch.cuda.synchronize()

    ref = torch.empty((S, H, D), dtype=torch.float16, device=DEV)
    step(ref, 0, True)
    ref_k, ref_v = kc.clone(), vc.clone()
    stale = torch.empty_like(ref)
    kc.copy_(k_old)
    vc.copy_(v_old)
    pa.pa_decode_ex(stale, q, kc, vc, bt, ctx, scale, B, ws)
    torch.cuda.synchronize()
    assert not torch.equal(stale.view(torch.int16), ref.view(torch.int16))   # the blocks matter
    for _ in range(10):
        out = torch.full_like(ref, float("nan"))
        step(out, pa.PA_DECODE_ZEROED_WORKSPACE, False)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(kc.view(torch.int16), ref_k.view(torch.int16))
        assert torch.equal(vc.view(torch.int16), ref_v.view(torch.int16))
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("append", [False, True])
def test_inputs_ready_behind_another_layers_decode(append):
    """PA_DECODE_INPUTS_READY as the decode step uses it: four layers' calls in
    a row on one workspace, each but the first behind the previous layer's
    decode (which writes none of its inputs), give the bits of calls made one
    at a time after a synchronize."""
    import dataclasses
    w = dataclasses.replace(configs.small_random(5700 + append, 300, 4, 128, 16, 900, min_context=1),
                            num_layers=4)
    dw = gpu.materialize(w, device=DEV)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
    shape = (w.num_seqs, w.num_heads, w.head_dim)
    kn = [torch.randn(shape, generator=torch.Generator().manual_seed(5710 + i)).to(torch.float16)
          .to(DEV) for i in range(4)]
    vn = [torch.randn(shape, generator=torch.Generator().manual_seed(5720 + i)).to(torch.float16)
          .to(DEV) for i in range(4)]
    kc0 = [t.clone() for t in dw.key_caches]
    vc0 = [t.clone() for t in dw.value_caches]

    def layer(i, out, flags):
        args = (dw.key_caches[i], dw.value_caches[i], dw.block_tables, dw.context_lens, w.scale)
        if append:
            pa.pa_decode_append(out, dw.queries[i], kn[i], vn[i], *args, w.max_context_len, ws, flags)
        else:
            pa.pa_decode_ex(out, dw.queries[i], *args, w.max_context_len, ws, flags)

    refs = []
    for i in range(4):
        refs.append(torch.empty(shape, dtype=torch.float16, device=DEV))
        layer(i, refs[-1], 0)
        torch.cuda.synchronize()
    ref_caches = [t.clone() for t in dw.key_caches + dw.value_caches]
    for _ in range(3):
        for t, t0 in zip(dw.key_caches + dw.value_caches, kc0 + vc0):
            t.copy_(t0)
        outs = [torch.full(shape, float("nan"), dtype=torch.float16, device=DEV) for _ in range(4)]
        for i in range(4):
            layer(i, outs[i], pa.PA_DECODE_ZEROED_WORKSPACE | (pa.PA_DECODE_INPUTS_READY if i else 0))
        torch.cuda.synchronize()
        for o, r in zip(outs, refs):
            assert torch.equal(o.view(torch.int16), r.view(torch.int16))
        for t, r in zip(dw.key_caches + dw.value_caches, ref_caches):
            assert torch.equal(t.view(torch.int16), r.view(torch.int16))
    assert pa.pa_check_errors() == (pa.PA_OK, 0)

"""The decode step replayed as a CUDA graph gives the same bits as the same
step launched eagerly, including after the inputs are updated in place
between replays and with the copy-on-write block copies in the step."""
import numpy as np
import pytest
import torch

import paged_kv_cache_158_gb300 as pa
from paged_kv_cache_158_gb300.pool import BlockManager
from paged_kv_cache_158_gb300.step import DecodeStep
from pa_testlib import u16
from workloads import configs, gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make_step(w, dw, copy_pairs=None, fp8_scales=None, stacked_outs=False):
    if stacked_outs:
        outs = list(torch.empty((len(dw.layers), w.num_seqs, w.num_heads, w.head_dim),
                                dtype=torch.float16, device=DEV).unbind(0))
    else:
        outs = [torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float16,
                            device=DEV) for _ in dw.layers]
    return DecodeStep(dw.key_caches, dw.value_caches, dw.queries, dw.keys_new, dw.values_new, outs,
                      dw.block_tables, dw.context_lens, dw.token_seq, dw.token_pos, w.block_size,
                      w.num_blocks, w.scale, int(w.context_lens.max()), copy_pairs, fp8_scales)


def clone_dw(dw):
    import copy
    c = copy.copy(dw)
    c.key_caches = [t.clone() for t in dw.key_caches]
    c.value_caches = [t.clone() for t in dw.value_caches]
    c.queries = [t.clone() for t in dw.queries]
    return c


@pytest.mark.parametrize("cfg,layers", [(2, [0]), (1, [0, 1, 2]), (5, [0, 1])])
def test_graph_replay_matches_eager(cfg, layers):
    w = configs.ALL[cfg]() if cfg != 5 else configs.config5(num_layers=2)
    dw = gpu.materialize(w, layers=layers, device=DEV)
    dw_eager = clone_dw(dw)
    eager = make_step(w, dw_eager)
    graph = make_step(w, dw)
    graph.capture()                       # runs the step twice eagerly, then captures it
    for rep in range(2):
        if rep == 1:                      # new queries, in place, before the second replay
            for qe, qg in zip(dw_eager.queries, dw.queries):
                qe.mul_(-1.0)
                qg.mul_(-1.0)
        eager.run()
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager.outs, graph.outs):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(dw_eager.key_caches + dw_eager.value_caches, dw.key_caches + dw.value_caches):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_graph_replay_matches_eager_fp8():
    from pa_testlib import materialize_fp8
    w = configs.config5(num_layers=2)
    sc = configs.fp8_scales(w)
    dw = materialize_fp8(w, layers=[0, 1])
    dw_eager = clone_dw(dw)
    eager = make_step(w, dw_eager, fp8_scales=sc)
    graph = make_step(w, dw, fp8_scales=sc)
    graph.capture()
    eager.run()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager.outs, graph.outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(dw_eager.key_caches + dw_eager.value_caches, dw.key_caches + dw.value_caches):
        assert torch.equal(a, b)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_graph_step_with_copy_on_write():
    w = configs.config4()
    bm = BlockManager(w.num_blocks, w.block_size, w.num_seqs, w.max_blocks_per_seq, w.free_order)
    bm.add_sequence(0)
    bm.append_tokens(0, w.prefix_len)
    for s in range(1, w.num_seqs):
        bm.fork(0, s)
    for s in range(w.num_seqs):
        bm.append_tokens(s, int(w.suffix_lens[s]))
    pairs = torch.from_numpy(bm.take_copies()).to(DEV)
    dw = gpu.materialize(w, device=DEV)
    dw.block_tables = torch.from_numpy(bm.block_tables()).to(DEV)
    dw_eager = clone_dw(dw)
    eager = make_step(w, dw_eager, pairs)
    graph = make_step(w, dw, pairs)
    eager.run()
    graph.capture(warmup=1)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.outs[0].view(torch.int16), graph.outs[0].view(torch.int16))
    assert np.array_equal(u16(dw_eager.key_caches[0]), u16(dw.key_caches[0]))
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("cfg,layers,use_graph,stacked", [
    (2, [0], False, False), (5, [0, 1], True, False), (1, [0, 1, 2], True, False),
    (3, list(range(11)), True, True), (3, list(range(11)), False, True)])
def test_host_staged_step_matches_device_step(cfg, layers, use_graph, stacked):
    """Inputs uploaded from pinned host buffers and outputs read back, overlapped layer by
    layer (eager or as one graph): the host outputs and the caches are bit-identical to the
    device-resident step's, also after the host inputs change in place; the device input
    buffers are poisoned before each run, so every input must come through the copies.
    stacked: each kind's per-layer buffers are views of one [L, ...] tensor on both sides, so
    the step merges the copies of each layer group (11 layers: groups of 1, 1, 2, 4, 3)."""
    w = configs.ALL[cfg]() if cfg != 5 else configs.config5(num_layers=2)
    if cfg == 3:
        w = configs.config3(num_layers=len(layers))
    dw_ref = gpu.materialize(w, layers=layers, device=DEV)
    ref = make_step(w, dw_ref)
    dw = gpu.materialize(w, layers=layers, device=DEV)
    st = make_step(w, dw, stacked_outs=stacked)
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    if stacked:
        h_q, h_k, h_v = (list(pin(torch.stack(ts)).unbind(0))
                         for ts in (dw.queries, dw.keys_new, dw.values_new))
        h_out = list(torch.full((len(st.outs),) + tuple(st.outs[0].shape), float("nan"),
                                dtype=torch.float16).pin_memory().unbind(0))
    else:
        h_q, h_k, h_v = ([pin(t) for t in ts] for ts in (dw.queries, dw.keys_new, dw.values_new))
        h_out = [torch.full(o.shape, float("nan"), dtype=o.dtype).pin_memory() for o in st.outs]
    h_small = [pin(t) for t in (dw.block_tables, dw.context_lens, dw.token_seq, dw.token_pos)]
    st.bind_host(h_q, h_k, h_v, h_out, *h_small)
    n_copies = sum(len(r) for r in st.host["up_runs"].values()) + \
        sum(len(r) for r in st.host["down_runs"].values())
    n_groups = len(st.host["up_runs"])
    assert n_copies == (4 * n_groups if stacked else 4 * len(layers))

    def poison():
        for t in dw.queries + dw.keys_new + dw.values_new:
            t.fill_(float("nan"))
        dw.context_lens.zero_()
        dw.token_pos.zero_()

    if use_graph:
        st.capture(host=True)
    for rep in range(2):
        if rep == 1:                      # new queries, in place, on both sides
            for qr, qh in zip(dw_ref.queries, h_q):
                qr.mul_(-1.0)
                qh.mul_(-1.0)
        poison()
        ref.run()
        st.replay(host=True) if use_graph else st.run_host()
        torch.cuda.synchronize()
        for a, b in zip(ref.outs, h_out):
            assert torch.equal(a.cpu().view(torch.int16), b.view(torch.int16))
    for a, b in zip(dw_ref.key_caches + dw_ref.value_caches, dw.key_caches + dw.value_caches):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_bind_host_refuses_pageable_or_mismatched_buffers():
    w = configs.config1()
    dw = gpu.materialize(w, layers=[0], device=DEV)
    st = make_step(w, dw)
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    args = [[pin(dw.queries[0])], [pin(dw.keys_new[0])], [pin(dw.values_new[0])],
            [torch.empty(st.outs[0].shape, dtype=torch.float16).pin_memory()]] + \
        [pin(t) for t in (dw.block_tables, dw.context_lens, dw.token_seq, dw.token_pos)]
    st.bind_host(*args)
    bad = list(args)
    bad[0] = [dw.queries[0].cpu()]                       # pageable
    with pytest.raises(ValueError):
        st.bind_host(*bad)
    bad = list(args)
    bad[4] = pin(dw.block_tables[:, :1].contiguous())    # wrong shape
    with pytest.raises(ValueError):
        st.bind_host(*bad)
    with pytest.raises(RuntimeError):
        make_step(w, dw).run_host()

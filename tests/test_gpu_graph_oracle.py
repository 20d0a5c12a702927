"""The decode step replayed as a CUDA graph, checked against the oracle (not
against the eager step): every output within the decode tolerance and every
cache bit for bit, after each of two replays with the inputs changed in place
between them.  Covers the device-resident graph, the graph that reads its
inputs from pinned host buffers and writes its outputs back to them (the
bench's end-to-end path), FP8 caches, and the shared-prefix step with its
copy-on-write copies.

The oracle side replays the same history on the host: each warm-up run and
each replay writes the new tokens again (the write is a plain store, so a
repeated write of the same rows leaves the same pool), then decodes with the
oracle's own slot map, cache write and decode."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa
from oracle.block_model import shared_prefix_flow
from paged_kv_cache_158_gb300.pool import BlockManager
from paged_kv_cache_158_gb300.step import DecodeStep
from pa_testlib import decode_gate, materialize_fp8, u8, u16
from workloads import configs, gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"
SIGN16 = np.uint16(0x8000)


def make_step(w, dw, max_ctx=None, copy_pairs=None, fp8_scales=None, append=False):
    outs = [torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=torch.float16,
                       device=DEV) for _ in dw.layers]
    return DecodeStep(dw.key_caches, dw.value_caches, dw.queries, dw.keys_new, dw.values_new, outs,
                      dw.block_tables, dw.context_lens, dw.token_seq, dw.token_pos, w.block_size,
                      w.num_blocks, w.scale, int(w.context_lens.max()) if max_ctx is None else max_ctx,
                      copy_pairs, fp8_scales, append=append)


class OracleLayer:
    """One layer's pool on the host, advanced by the oracle's own calls."""

    def __init__(self, w, layer, fp8_scales=None):
        self.w, self.f8 = w, fp8_scales
        kc, vc = gpu.host_pool(w, layer)
        if fp8_scales is not None:
            kc, vc = oracle.quantize_e4m3(kc, fp8_scales[0]), oracle.quantize_e4m3(vc, fp8_scales[1])
        self.kc, self.vc = kc, vc

    def write(self, bt, seqs, pos, kn, vn):
        w = self.w
        slots, rc = oracle.slot_mapping(bt, seqs, pos, w.block_size, w.num_blocks)
        assert rc == 0
        if self.f8 is not None:
            assert oracle.reshape_and_cache_fp8(self.kc, self.vc, kn, vn, slots, w.block_size,
                                                *self.f8) == 0
        else:
            assert oracle.reshape_and_cache(self.kc, self.vc, kn, vn, slots, w.block_size) == 0

    def decode(self, q, bt, ctx):
        w = self.w
        if self.f8 is not None:
            _, ref64, rc = oracle.decode_fp8(q, self.kc, self.vc, bt, ctx, w.scale, *self.f8)
        else:
            _, ref64, rc = oracle.decode(q, self.kc, self.vc, bt, ctx, w.scale)
        assert rc == 0
        return ref64

    def check_pool(self, kc_dev, vc_dev, what):
        conv = u8 if self.f8 is not None else u16
        assert np.array_equal(conv(kc_dev), self.kc), f"{what}: key cache differs from the oracle"
        assert np.array_equal(conv(vc_dev), self.vc), f"{what}: value cache differs from the oracle"


def _second_step_inputs(w, dw, host=None):
    """Changes the step's inputs in place for the second replay: queries
    negated, each layer's new key/value rows replaced by the next layer's,
    and every sequence one token shorter (the new token is written at c - 2
    and decode attends over [0, c - 1)).  With host = the bound host buffers,
    the change is made there (the device buffers are refilled by the step).
    Returns the host-side copies (q, kn, vn per layer, ctx, pos) the oracle uses."""
    L = len(dw.layers)
    q = [gpu.host_small(w, l)[0] ^ SIGN16 for l in dw.layers]
    kn = [gpu.host_small(w, dw.layers[(i + 1) % L])[1] for i in range(L)]
    vn = [gpu.host_small(w, dw.layers[(i + 1) % L])[2] for i in range(L)]
    seqs, pos = w.new_tokens()
    ctx = (w.context_lens - 1).astype(np.int32)
    pos = (pos - 1).astype(np.int32)
    if host is None:
        tq, tk, tv, tctx, tpos = dw.queries, dw.keys_new, dw.values_new, dw.context_lens, dw.token_pos
    else:
        tq, tk, tv, tctx, tpos = host
    for i in range(L):
        tq[i].copy_(torch.from_numpy(q[i].view(np.int16)).view(torch.float16))
        tk[i].copy_(torch.from_numpy(kn[i].view(np.int16)).view(torch.float16))
        tv[i].copy_(torch.from_numpy(vn[i].view(np.int16)).view(torch.float16))
    tctx.copy_(torch.from_numpy(ctx))
    tpos.copy_(torch.from_numpy(pos))
    return q, kn, vn, ctx, seqs, pos


def _run_graph_against_oracle(w, dw, fp8_scales=None, host=False, append=False):
    st = make_step(w, dw, fp8_scales=fp8_scales, append=append)
    hb = None
    if host:
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        h_q, h_k, h_v = ([pin(t) for t in ts] for ts in (dw.queries, dw.keys_new, dw.values_new))
        h_small = [pin(t) for t in (dw.block_tables, dw.context_lens, dw.token_seq, dw.token_pos)]
        h_out = [torch.full(o.shape, float("nan"), dtype=o.dtype).pin_memory() for o in st.outs]
        st.bind_host(h_q, h_k, h_v, h_out, *h_small)
        hb = (h_q, h_k, h_v, h_small[1], h_small[3], h_out)
    st.capture(host=host)                     # two eager warm-up runs, then the capture
    orc = [OracleLayer(w, l, fp8_scales) for l in dw.layers]
    seqs, pos = w.new_tokens()
    for rep in range(2):
        if rep == 0:
            q = [gpu.host_small(w, l)[0] for l in dw.layers]
            kn = [gpu.host_small(w, l)[1] for l in dw.layers]
            vn = [gpu.host_small(w, l)[2] for l in dw.layers]
            ctx = w.context_lens
        else:
            q, kn, vn, ctx, seqs, pos = _second_step_inputs(
                w, dw, None if not host else (hb[0], hb[1], hb[2], hb[3], hb[4]))
        outs = hb[5] if host else st.outs
        for o in outs:
            o.fill_(float("nan"))
        if host:                              # every input must come through the step's copies
            for t in dw.queries + dw.keys_new + dw.values_new:
                t.fill_(float("nan"))
            dw.context_lens.zero_()
            dw.token_pos.zero_()
        st.replay(host=host)
        torch.cuda.synchronize()
        for i, o in enumerate(orc):
            o.write(w.block_tables, seqs, pos, kn[i], vn[i])
            ref64 = o.decode(q[i], w.block_tables, ctx)
            decode_gate(outs[i], ref64, f"graph{' (host)' if host else ''} {w.name} layer "
                                        f"{dw.layers[i]} replay {rep}")
            o.check_pool(dw.key_caches[i], dw.value_caches[i], f"layer {dw.layers[i]} replay {rep}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("append", [False, True])
def test_graph_step_13b_four_layers_against_oracle(append):
    """append: each layer's cache write fused into its decode (pa_decode_append)."""
    w = configs.config3(num_layers=4)
    _run_graph_against_oracle(w, gpu.materialize(w, device=DEV), append=append)


@pytest.mark.parametrize("append", [False, True])
def test_host_graph_step_13b_four_layers_against_oracle(append):
    """The end-to-end form: inputs from pinned host buffers, outputs to pinned
    host buffers, one captured graph; the device input buffers are poisoned
    before each replay."""
    w = configs.config3(num_layers=4)
    _run_graph_against_oracle(w, gpu.materialize(w, device=DEV), host=True, append=append)


@pytest.mark.parametrize("append", [False, True])
def test_graph_step_long_context_fp8_against_oracle(append):
    w = configs.config5(num_layers=2)
    sc = configs.fp8_scales(w)
    _run_graph_against_oracle(w, materialize_fp8(w, layers=[0, 1]), fp8_scales=sc, append=append)


def test_graph_step_shared_prefix_copy_on_write_against_oracle():
    """The shared-prefix step with its planned copy-on-write copies inside the
    graph.  Every run of the step (two warm-ups, two replays) copies the
    shared partial block again and writes the suffix tokens again; the oracle
    applies the pages' block manager plan the same number of times."""
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
    dw.context_lens = torch.from_numpy(bm.context_lens()).to(DEV)
    st = make_step(w, dw, copy_pairs=pairs)
    st.capture(warmup=2)

    model, appended = shared_prefix_flow(w.num_seqs, w.prefix_len, w.suffix_lens, w.num_blocks,
                                         w.block_size, w.free_order)
    mbt = model.table_array(range(w.num_seqs), w.max_blocks_per_seq)
    mctx = np.array([model.lengths[s] for s in range(w.num_seqs)], dtype=np.int32)
    seqs = np.array([s for s, _ in appended], dtype=np.int32)
    pos = np.array([p for _, p in appended], dtype=np.int32)
    o = OracleLayer(w, 0)
    q, kn, vn = gpu.host_small(w, 0)
    copies = np.array(model.copies, dtype=np.int64)
    runs = 2                                   # the eager warm-ups
    for rep in range(2):
        st.outs[0].fill_(float("nan"))
        st.replay()
        torch.cuda.synchronize()
        for _ in range(runs + 1):
            assert oracle.copy_blocks([o.kc], [o.vc], copies) == 0
            o.write(mbt, seqs, pos, kn, vn)
        runs = 0
        decode_gate(st.outs[0], o.decode(q, mbt, mctx), f"graph {w.name} replay {rep}")
        o.check_pool(dw.key_caches[0], dw.value_caches[0], f"{w.name} replay {rep}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)

"""GPU parity of multi-query paged attention (chunked prefill and mixed
prefill + decode batches, tensor cores) against the oracle: every output of
small ragged batches (chunks crossing tile boundaries, one-token chunks,
empty chunks, whole-context chunks, NaN in every dead slot), every output of
the 7B-shaped chunked prefill at full size (and sampled rows of it), and the
error reporting."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa
from pa_testlib import prefill_gate, live_slot_mask, poison_dead_slots_device, poison_dead_slots_host
from workloads import configs, gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean():
    pa.pa_check_errors()
    yield
    torch.cuda.synchronize()


def run_prefill(w, dv, max_q=None):
    tq = int(np.sum(w.extra["q_lens"]))
    out = torch.full((tq, w.num_heads, w.head_dim), float("nan"), dtype=torch.float16, device=DEV)
    pa.pa_prefill(out, dv["query"], dv["key_cache"], dv["value_cache"], dv["block_tables"],
                  dv["context_lens"], dv["query_start"], w.scale,
                  int(max(w.extra["q_lens"])) if max_q is None else max_q)
    return out


def oracle_prefill(w, poison_mask=None):
    kc, vc = gpu.host_pool(w, 0)
    if poison_mask is not None:
        poison_dead_slots_host(kc, vc, poison_mask)
    _, ref64, rc = oracle.prefill(gpu.host_queries(w), kc, vc, w.block_tables, w.context_lens,
                                  configs.query_start(w), w.scale)
    assert rc == 0
    return ref64


MIXED = ([130, 1, 0, 77, 300, 1], [130, 500, 40, 77, 700, 1])


@pytest.mark.parametrize("D,B", [(64, 8), (64, 16), (128, 16), (128, 32), (128, 8), (64, 32)])
def test_prefill_mixed_batch_all_outputs(D, B):
    """Whole-context chunk crossing a tile boundary, decode rows, an empty
    chunk, a short whole-context chunk, a chunk after a 400-token prefix, a
    one-token context; NaN in every slot no live token uses."""
    w = configs.prefill_workload(f"mixed_D{D}_B{B}", 4000 + D + B, *MIXED, 3, D, B)
    dv = gpu.materialize_prefill(w, DEV)
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, B)
    poison_dead_slots_device(dv["key_cache"], dv["value_cache"], mask)
    out = run_prefill(w, dv)
    ref64 = oracle_prefill(w, mask)
    prefill_gate(out, ref64, f"prefill D{D} B{B}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("q_len,ctx", [(128, 128), (129, 1000), (256, 256), (383, 2047), (1, 3000)])
def test_prefill_tile_edges(q_len, ctx):
    w = configs.prefill_workload(f"edge_{q_len}_{ctx}", 4100 + q_len, [q_len, 5], [ctx, 9], 2, 128, 16)
    dv = gpu.materialize_prefill(w, DEV)
    out = run_prefill(w, dv)
    prefill_gate(out, oracle_prefill(w), f"prefill q{q_len} c{ctx}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_prefill_deterministic_and_decode_rows_match_decode():
    w = configs.prefill_workload("det", 4200, [200, 1, 1, 1], [900, 333, 64, 1000], 4, 128, 16)
    dv = gpu.materialize_prefill(w, DEV)
    a = run_prefill(w, dv).clone()
    b = run_prefill(w, dv)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref64 = oracle_prefill(w)
    prefill_gate(a, ref64, "prefill det")
    # the one-token chunks against the decode kernel on the same cache
    qs = configs.query_start(w)
    rows = torch.from_numpy(qs[1:4].astype(np.int64)).to(DEV)
    q = dv["query"][rows].contiguous()
    bt = dv["block_tables"][1:4].contiguous()
    cl = dv["context_lens"][1:4].contiguous()
    outd = torch.empty_like(q)
    ws = pa.decode_workspace(3, w.num_heads, w.head_dim, 1000)
    pa.pa_decode(outd, q, dv["key_cache"], dv["value_cache"], bt, cl, w.scale, 1000, ws)
    prefill_gate(outd, ref64[qs[1:4]], "decode rows")


def test_prefill_7b_full_size_sampled_rows():
    """The 7B-shaped chunked prefill at full size; sampled 16-row windows of
    every sequence checked against the oracle on the causally truncated
    problem (rows j0..j0+15 only see positions up to their own)."""
    w = configs.prefill_7b()
    dv = gpu.materialize_prefill(w, DEV)
    out = run_prefill(w, dv)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    kc, vc = gpu.host_pool(w, 0)
    q = gpu.host_queries(w)
    qs = configs.query_start(w)
    rng = np.random.default_rng(61)
    for s in range(w.num_seqs):
        ql, c = int(w.extra["q_lens"][s]), int(w.context_lens[s])
        for j0 in (0, int(rng.integers(1, ql - 16)), ql - 16):
            p_last = c - ql + j0 + 15
            bt = w.block_tables[s:s + 1]
            _, ref64, rc = oracle.prefill(q[qs[s] + j0:qs[s] + j0 + 16], kc, vc, bt,
                                          np.array([p_last + 1], np.int32),
                                          np.array([0, 16], np.int32), w.scale)
            assert rc == 0
            prefill_gate(out[qs[s] + j0:qs[s] + j0 + 16], ref64, f"{w.name} s{s} rows {j0}..")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_prefill_7b_whole_call_against_oracle():
    """The 7B-shaped chunked prefill at full size (4 x 512 new tokens over 2048-token
    contexts, 32 heads): every output against the oracle (about 60 GFLOP in binary64 on the
    host cores)."""
    w = configs.prefill_7b()
    dv = gpu.materialize_prefill(w, DEV)
    out = run_prefill(w, dv)
    torch.cuda.synchronize()
    prefill_gate(out, oracle_prefill(w), f"{w.name} whole call")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_prefill_bad_inputs_flagged():
    w = configs.prefill_workload("bad", 4300, [40, 30], [100, 60], 2, 64, 16)
    dv = gpu.materialize_prefill(w, DEV)
    run_prefill(w, dv, max_q=32)                   # max_query_len below the real chunk lengths
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits & pa.PA_ERRBIT_CONTEXT
    w.block_tables[1, 0] = w.num_blocks + 7
    dv["block_tables"] = torch.from_numpy(w.block_tables).to(DEV)
    out = run_prefill(w, dv)
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits & pa.PA_ERRBIT_BLOCK_ID
    # the other sequence is unaffected
    w.block_tables[1, 0] = 0
    ref64 = oracle_prefill(w)
    prefill_gate(out[:40], ref64[:40], "unaffected sequence")


def test_prefill_long_chunk_and_many_decode_rows():
    """A 1000-token chunk over a 5000-token context (four query-tile pairs), a 700-token
    whole-context chunk and 150 one-token rows in one batch; every output."""
    q_lens = [1000] + [1] * 150 + [700]
    ctx = [5000] + [100 + 13 * i for i in range(150)] + [700]
    w = configs.prefill_workload("long_many", 4600, q_lens, ctx, 2, 128, 16)
    dv = gpu.materialize_prefill(w, DEV)
    out = run_prefill(w, dv)
    prefill_gate(out, oracle_prefill(w), "long chunk + 150 decode rows")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("scale", [0.4, 1.5, 4.0])
def test_prefill_large_logits_rescale_path(scale):
    """Logit scales far above 1/sqrt(D) make later tiles hold logits many base-2 units above
    the row's running reference, so weights overflow fp16 and the tile is redone against its
    maximum with O and l rescaled; every output still matches the oracle."""
    w = configs.prefill_workload(f"scale{scale}", 4700, *MIXED, 3, 128, 16)
    w.logit_scale = scale
    dv = gpu.materialize_prefill(w, DEV)
    out = run_prefill(w, dv)
    prefill_gate(out, oracle_prefill(w), f"prefill scale {scale}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def _fp8_copy(w, dv):
    ks, vs = configs.fp8_scales(w)
    for name, sc in (("key_cache", ks), ("value_cache", vs)):
        codes = torch.empty(dv[name].shape, dtype=torch.uint8, device=DEV)
        pa.pa_convert_cache_fp8(dv[name], codes, sc)
        dv[name] = codes
    return ks, vs


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("shape", ["mixed", "7b"])
def test_inputs_ready_back_to_back_calls_match_serial_calls(shape, fp8):
    """PA_PREFILL_INPUTS_READY as the bench uses it: calls over three independent copies of the
    inputs, three rounds back to back, each call behind the previous one (which writes only its
    own output), give the bits of the same calls made one at a time after a synchronize.  The
    7B-shaped batch has two waves of CTAs, so a call's first CTAs run beside the previous call's
    last ones; the mixed batch has decode rows.  The mixed batch's output is also held to the
    oracle."""
    if shape == "mixed":
        w = configs.prefill_workload("ready", 4300 + fp8, *MIXED, 4, 128, 16)
    else:
        w = configs.prefill_7b()
    copies = [gpu.materialize_prefill(w, DEV) for _ in range(3)]
    scales = [_fp8_copy(w, dv) for dv in copies] if fp8 else [None] * 3
    tq = int(np.sum(w.extra["q_lens"]))
    max_q = int(max(w.extra["q_lens"]))

    def call(dv, sc, out, flags):
        args = (out, dv["query"], dv["key_cache"], dv["value_cache"], dv["block_tables"],
                dv["context_lens"], dv["query_start"], w.scale)
        if fp8:
            pa.pa_prefill_fp8_ex(*args, sc[0], sc[1], max_q, flags=flags)
        else:
            pa.pa_prefill_ex(*args, max_q, flags=flags)

    refs = []
    for dv, sc in zip(copies, scales):
        refs.append(torch.full((tq, w.num_heads, w.head_dim), float("nan"), dtype=torch.float16,
                               device=DEV))
        call(dv, sc, refs[-1], 0)
        torch.cuda.synchronize()
    outs = [torch.full_like(r, float("nan")) for r in refs]
    for _ in range(3):
        for dv, sc, o in zip(copies, scales, outs):
            call(dv, sc, o, pa.PA_PREFILL_INPUTS_READY)
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert torch.equal(o.view(torch.int16), r.view(torch.int16))
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    if shape == "mixed" and not fp8:
        prefill_gate(outs[0], oracle_prefill(w), "prefill inputs_ready")


@pytest.mark.parametrize("nseq,q_len,H", [(3, 700, 8), (7, 128, 32), (32, 300, 4), (5, 512, 32)])
def test_prefill_uniform_chunks_every_output(nseq, q_len, H):
    """Batches whose sequences all bring the same number of query-tile pairs take the
    planner's closed form (the first wave's whole groups, then rank by rank); every output
    row against the oracle (a unit mapped twice would leave another unfilled)."""
    rng = np.random.default_rng(4400 + nseq)
    ctx = [q_len + int(rng.integers(0, 400)) for _ in range(nseq)]
    w = configs.prefill_workload("uniform", 4400 + nseq, [q_len] * nseq, ctx, H, 128, 16)
    dv = gpu.materialize_prefill(w, DEV)
    out = run_prefill(w, dv)
    torch.cuda.synchronize()
    prefill_gate(out, oracle_prefill(w), f"uniform S{nseq} q{q_len} H{H}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def _run_ex(w, dv, n_rows, max_q=None, fp8_scales=None):
    """pa_prefill_ex / pa_prefill_fp8_ex with the count of one-token sequences."""
    tq = int(np.sum(w.extra["q_lens"]))
    out = torch.full((tq, w.num_heads, w.head_dim), float("nan"), dtype=torch.float16, device=DEV)
    args = (out, dv["query"], dv["key_cache"], dv["value_cache"], dv["block_tables"],
            dv["context_lens"], dv["query_start"], w.scale)
    mq = int(max(w.extra["q_lens"])) if max_q is None else max_q
    if fp8_scales is not None:
        pa.pa_prefill_fp8_ex(*args, fp8_scales[0], fp8_scales[1], mq, n_rows)
    else:
        pa.pa_prefill_ex(*args, mq, n_rows)
    return out


def _oracle_any(w, fp8_scales):
    if fp8_scales is None:
        return oracle_prefill(w)
    kc, vc = gpu.host_pool(w, 0)
    ks, vs = fp8_scales
    _, ref64, rc = oracle.prefill_fp8(gpu.host_queries(w), oracle.quantize_e4m3(kc, ks),
                                      oracle.quantize_e4m3(vc, vs), w.block_tables,
                                      w.context_lens, configs.query_start(w), w.scale, ks, vs)
    assert rc == 0
    return ref64


# One-token rows over contexts from 1 token (one chunk: eleven of the twelve warps idle,
# most heads skipped by most warps) to several hundred, between chunks.
ROWS_Q = [1, 300, 1, 1, 0, 1, 77, 1, 1, 1]
ROWS_C = [1, 700, 20, 191, 40, 192, 77, 193, 650, 1000]


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("D,B,H", [(128, 16, 8), (128, 8, 6), (64, 32, 3), (64, 16, 5),
                                   (128, 32, 1)])
def test_prefill_decode_rows_grouped_every_output(D, B, H, fp8):
    """With the count of one-token sequences given, a CTA runs up to four heads of a row as
    one chunk stream (the last group of a row may be smaller); every output row of the batch
    against the oracle, with NaN in every slot no live token uses."""
    w = configs.prefill_workload(f"rows_D{D}_B{B}_H{H}", 4800 + D + B + H, ROWS_Q, ROWS_C, H, D, B)
    dv = gpu.materialize_prefill(w, DEV)
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, B)
    poison_dead_slots_device(dv["key_cache"], dv["value_cache"], mask)
    sc = _fp8_copy(w, dv) if fp8 else None
    n_rows = sum(1 for q in ROWS_Q if q == 1)
    out = _run_ex(w, dv, n_rows, fp8_scales=sc)
    torch.cuda.synchronize()
    if fp8:
        ref64 = _oracle_any(w, sc)   # dead slots hold NaN codes only on the device side
    else:
        ref64 = oracle_prefill(w, mask)
    prefill_gate(out, ref64, f"grouped rows D{D} B{B} H{H} {'fp8' if fp8 else 'fp16'}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill_all_rows_grouped_without_count(fp8):
    """max_query_len == 1: every sequence is a decode row or empty, so the launch groups four
    heads per CTA without being told the count; every output row."""
    rng = np.random.default_rng(4900 + fp8)
    S = 70
    q_lens = [0 if i % 9 == 4 else 1 for i in range(S)]
    ctx = [int(rng.integers(1, 1500)) for _ in range(S)]
    w = configs.prefill_workload("all_rows", 4900 + fp8, q_lens, ctx, 10, 128, 16)
    dv = gpu.materialize_prefill(w, DEV)
    sc = _fp8_copy(w, dv) if fp8 else None
    out = _run_ex(w, dv, -1, fp8_scales=sc)
    torch.cuda.synchronize()
    prefill_gate(out, _oracle_any(w, sc), f"all rows {'fp8' if fp8 else 'fp16'}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_prefill_wrong_decode_row_count():
    """A count below the true one still sizes a large enough launch (each row fits the
    chunks' bound): every output is right.  A count above it leaves the chunk's units past
    the grid: reported as PA_ERRBIT_CONTEXT (the kernel skips them, nothing is read or
    written out of range)."""
    w = configs.prefill_workload("wrong_rows", 4950, [300, 1, 1, 1], [700, 64, 500, 900], 4,
                                 128, 16)
    dv = gpu.materialize_prefill(w, DEV)
    out = _run_ex(w, dv, 0)
    torch.cuda.synchronize()
    prefill_gate(out, oracle_prefill(w), "count 0 of 3")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    out = _run_ex(w, dv, 2)
    torch.cuda.synchronize()
    prefill_gate(out, oracle_prefill(w), "count 2 of 3")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    _run_ex(w, dv, 4)
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits & pa.PA_ERRBIT_CONTEXT

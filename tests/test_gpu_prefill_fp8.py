"""GPU parity of multi-query paged attention over FP8 (E4M3) caches against the
oracle: every output of small ragged batches (chunks crossing tile
boundaries, one-token and empty chunks, NaN codes in every dead slot),
the 7B-shaped chunked prefill at full size (whole call, and sampled rows), and the
argument and error reporting.  The device codes come from the library's
conversion kernel (tested bit-exact on its own); the oracle quantises its
own host copy of the pool."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa
from pa_testlib import prefill_gate, live_slot_mask, poison_dead_slots_device_fp8, poison_dead_slots_host_fp8
from workloads import configs, gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean():
    pa.pa_check_errors()
    yield
    torch.cuda.synchronize()


def materialize_fp8(w):
    dv = gpu.materialize_prefill(w, DEV)
    ks, vs = configs.fp8_scales(w)
    for name, sc in (("key_cache", ks), ("value_cache", vs)):
        codes = torch.empty(dv[name].shape, dtype=torch.uint8, device=DEV)
        pa.pa_convert_cache_fp8(dv[name], codes, sc)
        dv[name] = codes
    return dv


def run(w, dv, max_q=None, scales=None):
    tq = int(np.sum(w.extra["q_lens"]))
    ks, vs = configs.fp8_scales(w) if scales is None else scales
    out = torch.full((tq, w.num_heads, w.head_dim), float("nan"), dtype=torch.float16, device=DEV)
    pa.pa_prefill_fp8(out, dv["query"], dv["key_cache"], dv["value_cache"], dv["block_tables"],
                      dv["context_lens"], dv["query_start"], w.scale, ks, vs,
                      int(max(w.extra["q_lens"])) if max_q is None else max_q)
    return out


def oracle_pool(w):
    ks, vs = configs.fp8_scales(w)
    kc16, vc16 = gpu.host_pool(w, 0)
    return oracle.quantize_e4m3(kc16, ks), oracle.quantize_e4m3(vc16, vs)


def oracle_out(w, kc8, vc8, q=None, bt=None, ctx=None, qs=None):
    ks, vs = configs.fp8_scales(w)
    _, ref64, rc = oracle.prefill_fp8(gpu.host_queries(w) if q is None else q, kc8, vc8,
                                      w.block_tables if bt is None else bt,
                                      w.context_lens if ctx is None else ctx,
                                      configs.query_start(w) if qs is None else qs, w.scale, ks, vs)
    assert rc == 0
    return ref64


MIXED = ([130, 1, 0, 77, 300, 1], [130, 500, 40, 77, 700, 1])


@pytest.mark.parametrize("D,B", [(64, 8), (128, 16), (128, 32), (64, 32), (128, 8)])
def test_prefill_fp8_mixed_batch_all_outputs(D, B):
    w = configs.prefill_workload(f"f8mixed_D{D}_B{B}", 6000 + D + B, *MIXED, 3, D, B)
    dv = materialize_fp8(w)
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, B)
    poison_dead_slots_device_fp8(dv["key_cache"], dv["value_cache"], mask)
    out = run(w, dv)
    kc8, vc8 = oracle_pool(w)
    poison_dead_slots_host_fp8(kc8, vc8, mask)
    prefill_gate(out, oracle_out(w, kc8, vc8), f"fp8 prefill D{D} B{B}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


@pytest.mark.parametrize("q_len,ctx", [(128, 128), (129, 1000), (383, 2047), (1, 3000)])
def test_prefill_fp8_tile_edges(q_len, ctx):
    w = configs.prefill_workload(f"f8edge_{q_len}_{ctx}", 6100 + q_len, [q_len, 5], [ctx, 9], 2, 128, 16)
    dv = materialize_fp8(w)
    out = run(w, dv)
    prefill_gate(out, oracle_out(w, *oracle_pool(w)), f"fp8 prefill q{q_len} c{ctx}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_prefill_fp8_7b_full_size_sampled_rows():
    """The 7B-shaped chunked prefill at full size over FP8 caches; sampled 16-row windows of
    every sequence against the oracle on the causally truncated problem."""
    w = configs.prefill_7b()
    dv = materialize_fp8(w)
    out = run(w, dv)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    kc8, vc8 = oracle_pool(w)
    q = gpu.host_queries(w)
    qs = configs.query_start(w)
    rng = np.random.default_rng(62)
    for s in range(w.num_seqs):
        ql, c = int(w.extra["q_lens"][s]), int(w.context_lens[s])
        for j0 in (0, int(rng.integers(1, ql - 16)), ql - 16):
            p_last = c - ql + j0 + 15
            ref64 = oracle_out(w, kc8, vc8, q[qs[s] + j0:qs[s] + j0 + 16], w.block_tables[s:s + 1],
                               np.array([p_last + 1], np.int32), np.array([0, 16], np.int32))
            prefill_gate(out[qs[s] + j0:qs[s] + j0 + 16], ref64, f"fp8 {w.name} s{s} rows {j0}..")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_prefill_fp8_7b_whole_call_against_oracle():
    """The 7B-shaped chunked prefill at full size over FP8 caches: every output against the
    oracle's dequantising prefill on its own quantised copy of the pool."""
    w = configs.prefill_7b()
    dv = materialize_fp8(w)
    out = run(w, dv)
    torch.cuda.synchronize()
    kc8, vc8 = oracle_pool(w)
    prefill_gate(out, oracle_out(w, kc8, vc8), f"fp8 {w.name} whole call")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)


def test_prefill_fp8_scales_checked_and_bad_block_flagged():
    w = configs.prefill_workload("f8bad", 6300, [40, 30], [100, 60], 2, 64, 16)
    dv = materialize_fp8(w)
    for bad in ((0.0, 1.0), (1.0, -2.0), (float("inf"), 1.0), (1.0, float("nan"))):
        with pytest.raises(pa.PAError) as e:
            run(w, dv, scales=bad)
        assert e.value.status == pa.PA_ERR_INVALID_ARG
    w.block_tables[1, 0] = w.num_blocks + 7
    dv["block_tables"] = torch.from_numpy(w.block_tables).to(DEV)
    out = run(w, dv)
    st, bits = pa.pa_check_errors()
    assert st == pa.PA_ERR_OUT_OF_RANGE and bits & pa.PA_ERRBIT_BLOCK_ID
    w.block_tables[1, 0] = 0
    kc8, vc8 = oracle_pool(w)
    prefill_gate(out[:40], oracle_out(w, kc8, vc8)[:40], "fp8 unaffected sequence")


@pytest.mark.parametrize("scale", [0.4, 4.0])
def test_prefill_fp8_large_logits_rescale_path(scale):
    w = configs.prefill_workload(f"f8scale{scale}", 6400, *MIXED, 3, 128, 16)
    w.logit_scale = scale
    dv = materialize_fp8(w)
    out = run(w, dv)
    prefill_gate(out, oracle_out(w, *oracle_pool(w)), f"fp8 prefill scale {scale}")
    assert pa.pa_check_errors() == (pa.PA_OK, 0)

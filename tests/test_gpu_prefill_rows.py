"""Multi-query attention batches whose one-token rows run on the kernel's
CUDA-core path and whose units are numbered densely: every output against the
oracle for decode rows of every block size and head size (fp16 and FP8
caches, ragged and long contexts, contexts of one token), chunk mixes whose
pair counts differ (the first-wave / later-rank order with uneven groups), and
more sequences than one launch takes."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_158_gb300 as pa
from pa_testlib import (live_slot_mask, materialize_fp8, poison_dead_slots_device,
                        poison_dead_slots_device_fp8, poison_dead_slots_host, poison_dead_slots_host_fp8,
                        prefill_gate)
from workloads import configs, gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean():
    pa.pa_check_errors()
    yield
    torch.cuda.synchronize()


def _fp8_pools(w, dv):
    ks, vs = configs.fp8_scales(w)
    for name, sc in (("key_cache", ks), ("value_cache", vs)):
        codes = torch.empty(dv[name].shape, dtype=torch.uint8, device=DEV)
        pa.pa_convert_cache_fp8(dv[name], codes, sc)
        dv[name] = codes
    kc, vc = gpu.host_pool(w, 0)
    return oracle.quantize_e4m3(kc, ks), oracle.quantize_e4m3(vc, vs)


def run_and_check(w, fp8=False, what=""):
    dv = gpu.materialize_prefill(w, DEV)
    mask = live_slot_mask(w.block_tables, w.context_lens, w.num_blocks, w.block_size)
    ks, vs = configs.fp8_scales(w)
    q = gpu.host_queries(w)
    qs = configs.query_start(w)
    if fp8:
        kc8, vc8 = _fp8_pools(w, dv)
        poison_dead_slots_device_fp8(dv["key_cache"], dv["value_cache"], mask)
        poison_dead_slots_host_fp8(kc8, vc8, mask)
    else:
        poison_dead_slots_device(dv["key_cache"], dv["value_cache"], mask)
        kc, vc = gpu.host_pool(w, 0)
        poison_dead_slots_host(kc, vc, mask)
    tq = int(qs[-1])
    out = torch.full((tq, w.num_heads, w.head_dim), float("nan"), dtype=torch.float16, device=DEV)
    max_q = int(max(w.extra["q_lens"]))
    if fp8:
        pa.pa_prefill_fp8(out, dv["query"], dv["key_cache"], dv["value_cache"], dv["block_tables"],
                          dv["context_lens"], dv["query_start"], w.scale, ks, vs, max_q)
        _, ref64, rc = oracle.prefill_fp8(q, kc8, vc8, w.block_tables, w.context_lens, qs, w.scale,
                                          ks, vs)
    else:
        pa.pa_prefill(out, dv["query"], dv["key_cache"], dv["value_cache"], dv["block_tables"],
                      dv["context_lens"], dv["query_start"], w.scale, max_q)
        _, ref64, rc = oracle.prefill(q, kc, vc, w.block_tables, w.context_lens, qs, w.scale)
    assert rc == 0
    prefill_gate(out, ref64, what)
    assert pa.pa_check_errors() == (pa.PA_OK, 0)
    return out


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("D,B", [(64, 8), (64, 16), (64, 32), (128, 8), (128, 16), (128, 32)])
def test_decode_rows_every_shape(D, B, fp8):
    """Decode rows only, contexts 1, 2, 15, 16, 17, 100, 777, 2050 tokens (one
    token, ragged chunks, several chunks per warp), plus one short chunk."""
    ctx = [1, 2, 15, 16, 17, 100, 777, 2050, 300]
    q_lens = [1] * 8 + [40]
    w = configs.prefill_workload(f"rows_D{D}_B{B}", 5000 + D + B + 7 * fp8, q_lens, ctx, 3, D, B)
    run_and_check(w, fp8, f"{'fp8 ' if fp8 else ''}decode rows D{D} B{B}")


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("B", [8, 16])
def test_decode_rows_long_contexts(B, fp8):
    """Contexts long enough that a warp's chunks span several windows of block
    ids (more than 32 chunks per warp)."""
    w = configs.prefill_workload(f"rows_long_B{B}", 5100 + B + fp8, [1, 1, 1], [9000, 6145, 3073],
                                 2, 128, B)
    run_and_check(w, fp8, f"{'fp8 ' if fp8 else ''}long decode rows B{B}")


def test_uneven_chunk_pairs_across_the_first_wave():
    """Chunks of 3, 2, 4, 1, 3 pairs of query tiles on 16 heads (208 units, more
    than one per SM), a few decode rows and an empty sequence between them."""
    q_lens = [600, 300, 1, 800, 0, 100, 1, 513]
    ctx = [700, 300, 50, 1200, 10, 900, 4000, 513]
    w = configs.prefill_workload("uneven", 5200, q_lens, ctx, 16, 64, 16)
    run_and_check(w, False, "uneven chunk pairs")


def test_more_sequences_than_one_launch():
    """5000 sequences (the kernel takes 4096 per launch): decode rows of short
    contexts and a chunk in each launch window."""
    rng = np.random.default_rng(53)
    S = 5000
    q_lens = np.ones(S, dtype=np.int32)
    ctx = rng.integers(1, 40, S).astype(np.int32)
    for s in (3, 4095, 4096, 4999):
        q_lens[s], ctx[s] = 70, 90
    w = configs.prefill_workload("many_seqs", 5300, q_lens, ctx, 2, 64, 16)
    run_and_check(w, False, "5000 sequences")

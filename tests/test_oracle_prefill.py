"""Pins for the oracle's multi-query paged attention (chunked prefill and
mixed prefill + decode batches), independent of the oracle's own code:

* equality with causal dense attention computed by numpy on contiguous K/V
  (the paged formula is the dense one on gathered K/V, "vLLM推理加速深度解读"
  §2.1 and §2.3, applied to each new token over the positions up to its own);
* closed forms: a whole-context chunk's first token returns V_0 exactly; a
  one-token chunk is the dense single-query attention over the context;
* causality: changing K/V after a token's position leaves its output
  bit-identical; mixed batches with empty chunks; bad input reported.
"""
import math

import numpy as np
import pytest

import oracle
from test_oracle_pins import dense_attention, paged_from_dense


def make_case(rng, q_lens, ctx, H, D, B, spare=2, sigma=1.0):
    ctx = np.asarray(ctx, dtype=np.int32)
    Kd = [(sigma * rng.standard_normal((int(c), H, D))).astype(np.float16) for c in ctx]
    Vd = [(sigma * rng.standard_normal((int(c), H, D))).astype(np.float16) for c in ctx]
    NB = sum(-(-int(c) // B) for c in ctx) + spare
    kc, vc, bt = paged_from_dense(Kd, Vd, ctx, B, NB, rng)
    qs = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = rng.standard_normal((int(qs[-1]), H, D)).astype(np.float16)
    return q, kc, vc, bt, ctx, qs, Kd, Vd


def dense_causal(q, Kd, Vd, ctx, qs, scale):
    TQ, H, D = q.shape
    out = np.zeros((TQ, H, D))
    for s in range(len(ctx)):
        c, ql = int(ctx[s]), int(qs[s + 1] - qs[s])
        for j in range(ql):
            p = c - ql + j
            for h in range(H):
                out[qs[s] + j, h] = dense_attention(q[qs[s] + j, h].astype(np.float64),
                                                    Kd[s][:p + 1, h].astype(np.float64),
                                                    Vd[s][:p + 1, h].astype(np.float64), scale)
    return out


@pytest.mark.parametrize("q_lens,ctx,H,D,B", [
    ([5, 1, 17, 0], [9, 30, 40, 12], 2, 64, 4),
    ([33, 1, 1], [33, 70, 5], 3, 32, 16),
    ([8, 20], [100, 20], 1, 16, 8),
])
def test_prefill_equals_causal_dense_attention(q_lens, ctx, H, D, B):
    rng = np.random.default_rng(sum(q_lens) + D)
    q, kc, vc, bt, ctx, qs, Kd, Vd = make_case(rng, q_lens, ctx, H, D, B)
    scale = 1.0 / math.sqrt(D)
    out16, out64, rc = oracle.prefill(q, kc, vc, bt, ctx, qs, scale)
    assert rc == 0
    ref = dense_causal(q, Kd, Vd, ctx, qs, scale)
    np.testing.assert_allclose(out64, ref, rtol=1e-12, atol=1e-14)
    assert np.array_equal(out16, out64.astype(np.float16).view(np.uint16))


def test_first_token_of_a_whole_context_chunk_returns_v0():
    rng = np.random.default_rng(3)
    q, kc, vc, bt, ctx, qs, Kd, Vd = make_case(rng, [12, 7], [12, 7], 2, 64, 4)
    out16, out64, rc = oracle.prefill(q, kc, vc, bt, ctx, qs, 0.125)
    assert rc == 0
    for s in range(2):
        assert np.array_equal(out16[qs[s]], Vd[s][0].view(np.uint16))


def test_one_token_chunks_are_single_query_attention():
    rng = np.random.default_rng(4)
    q, kc, vc, bt, ctx, qs, Kd, Vd = make_case(rng, [1, 1, 1], [5, 33, 64], 2, 32, 8)
    _, out64, rc = oracle.prefill(q, kc, vc, bt, ctx, qs, 0.3)
    assert rc == 0
    for s in range(3):
        for h in range(2):
            ref = dense_attention(q[s, h].astype(np.float64), Kd[s][:, h].astype(np.float64),
                                  Vd[s][:, h].astype(np.float64), 0.3)
            np.testing.assert_allclose(out64[s, h], ref, rtol=1e-12, atol=1e-14)


def test_causality_later_positions_do_not_matter():
    rng = np.random.default_rng(5)
    q, kc, vc, bt, ctx, qs, Kd, Vd = make_case(rng, [10], [25], 2, 32, 8)
    a16, _, _ = oracle.prefill(q, kc, vc, bt, ctx, qs, 0.2)
    last = int(ctx[0]) - 1
    blk, off = bt[0, last // 8], last % 8
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[blk, :, off] = np.float16(7.0)
    vc2[blk, :, off] = np.float16(-3.0)
    b16, _, _ = oracle.prefill(q, kc2, vc2, bt, ctx, qs, 0.2)
    assert np.array_equal(a16[:9], b16[:9])          # tokens before the changed position
    assert not np.array_equal(a16[9], b16[9])        # the last token sees it


def test_bad_inputs_are_reported():
    rng = np.random.default_rng(6)
    q, kc, vc, bt, ctx, qs, _, _ = make_case(rng, [4], [4], 1, 16, 4)
    _, _, rc = oracle.prefill(q, kc, vc, bt, np.array([3], np.int32), qs, 0.5)   # q_len > c
    assert rc != 0
    bt2 = bt.copy()
    bt2[0, 0] = kc.shape[0] + 3
    _, _, rc = oracle.prefill(q, kc, vc, bt2, ctx, qs, 0.5)
    assert rc != 0

"""Pins for the oracle's multi-query paged attention over FP8 (E4M3) caches,
independent of the oracle's own code:

* equality with causal dense attention computed by numpy on contiguous K/V
  dequantised by PyTorch's ``float8_e4m3fn`` conversion (a library routine)
  and scaled, with different key and value scales (swapping them fails), on
  mixed batches with empty, one-token and whole-context chunks;
* closed form: a whole-context chunk's first token returns E4M3(V_0) times
  the value scale exactly;
* bad input (a block id out of range, q_len > context) is reported.
"""
import math

import numpy as np
import pytest

import oracle
from test_oracle_fp8 import torch_e4m3_decode
from test_oracle_prefill import dense_causal


def fp8_case(rng, q_lens, ctx, H, D, B, spare=2):
    """Random non-NaN codes in a paged pool with random block placement."""
    ctx = np.asarray(ctx, dtype=np.int32)
    NB = sum(-(-int(c) // B) for c in ctx) + spare
    codes = lambda: (rng.integers(0, 0x7E, (NB, H, B, D)) |  # noqa: E731
                     (rng.integers(0, 2, (NB, H, B, D)) << 7)).astype(np.uint8)
    kc, vc = codes(), codes()
    perm = rng.permutation(NB)
    nbs = [-(-int(c) // B) for c in ctx]
    bt = np.full((len(ctx), max(1, max(nbs))), -1, dtype=np.int32)
    off = 0
    for s, nb in enumerate(nbs):
        bt[s, :nb] = perm[off:off + nb]
        off += nb
    qs = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = rng.standard_normal((int(qs[-1]), H, D)).astype(np.float16)
    return q, kc, vc, bt, ctx, qs


def dense_of(pool, bt, ctx, B, H, D):
    """Per-sequence contiguous [c, H, D] arrays gathered with numpy fancy indexing."""
    out = []
    for s, c in enumerate(ctx):
        blocks = bt[s, :-(-int(c) // B)] if c > 0 else np.zeros(0, dtype=np.int32)
        out.append(pool[blocks].transpose(0, 2, 1, 3).reshape(-1, H, D)[:int(c)])
    return out


@pytest.mark.parametrize("q_lens,ctx,H,D,B", [
    ([5, 1, 17, 0], [9, 30, 40, 12], 2, 64, 4),
    ([33, 1, 1], [33, 70, 5], 3, 32, 16),
    ([8, 20], [100, 20], 1, 128, 8),
])
def test_prefill_fp8_equals_causal_dense_attention_on_dequantised_kv(q_lens, ctx, H, D, B):
    rng = np.random.default_rng(sum(q_lens) + D + 7)
    q, kc, vc, bt, ctx, qs = fp8_case(rng, q_lens, ctx, H, D, B)
    k_scale, v_scale, scale = 0.011, 0.0047, 1.0 / math.sqrt(D)
    out16, out64, rc = oracle.prefill_fp8(q, kc, vc, bt, ctx, qs, scale, k_scale, v_scale)
    assert rc == 0
    Kd = dense_of(torch_e4m3_decode(kc) * k_scale, bt, ctx, B, H, D)
    Vd = dense_of(torch_e4m3_decode(vc) * v_scale, bt, ctx, B, H, D)
    ref = dense_causal(q, Kd, Vd, ctx, qs, scale)
    np.testing.assert_allclose(out64, ref, rtol=1e-12, atol=1e-15)
    assert np.array_equal(out16, out64.astype(np.float16).view(np.uint16))


def test_prefill_fp8_first_token_of_whole_context_chunk_is_v0():
    rng = np.random.default_rng(5)
    q, kc, vc, bt, ctx, qs = fp8_case(rng, [24], [24], 2, 64, 8)
    _, out64, rc = oracle.prefill_fp8(q, kc, vc, bt, ctx, qs, 0.125, 0.02, 0.003)
    assert rc == 0
    v0 = torch_e4m3_decode(vc[bt[0, 0], :, 0]) * 0.003      # position 0 of every head
    assert np.array_equal(out64[0], v0)


def test_prefill_fp8_bad_inputs_reported():
    rng = np.random.default_rng(6)
    q, kc, vc, bt, ctx, qs = fp8_case(rng, [4, 3], [10, 3], 1, 32, 4)
    assert oracle.prefill_fp8(q, kc, vc, bt, ctx, qs, 0.1, 1.0, 1.0)[2] == 0
    bad = bt.copy()
    bad[0, 1] = kc.shape[0] + 3
    assert oracle.prefill_fp8(q, kc, vc, bad, ctx, qs, 0.1, 1.0, 1.0)[2] == -1
    assert oracle.prefill_fp8(q, kc, vc, bt, np.array([10, 2], np.int32), qs, 0.1, 1.0, 1.0)[2] == -1

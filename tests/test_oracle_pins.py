"""Pins for the oracle: checks against what the pages and mathematics fix,
independent of the oracle's own code.

* fp16 conversions against numpy's IEEE 754 conversions (library routine),
  every binary16 pattern and the rounding ties;
* paged decode against dense attention computed by numpy on contiguous,
  un-paged K/V ("vLLM推理加速深度解读" §2.1 and §2.3: the paged formula is
  the dense one applied to gathered K/V);
* invariance under relabelling physical blocks, identity of shared and
  privately copied prefixes;
* closed forms (one token; equal keys; constant values; a dominant logit;
  a hand-computed two-token case) and brute force on tiny shapes;
* the worked block-table example and the cache-write / block-copy loops
  against numpy indexing.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from workloads import configs, synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------- fp16

def test_half_to_double_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, ours[0x8000]) == -1.0


def test_double_to_half_roundtrip_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    back = oracle.double_to_half(vals)
    finite = ~np.isnan(vals)
    assert np.array_equal(back[finite], bits[finite])
    assert np.all((back[~finite] & 0x7C00) == 0x7C00) and np.all((back[~finite] & 0x3FF) != 0)


def test_double_to_half_rounding_matches_ieee():
    rng = np.random.default_rng(5)
    # Wide random range, including subnormal and overflow territory.
    x = rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 17, 200000))
    # Exact midpoints between neighbouring halves (ties go to even), and
    # points a hair either side of them.
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2
    special = np.array([65504.0, 65519.999, 65520.0, 65536.0, 1e300, 2.0 ** -24, 2.0 ** -25,
                        3 * 2.0 ** -26, 2.0 ** -26, 0.0, -0.0, np.inf, -np.inf])
    allx = np.concatenate([x, -x, mid, -mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf),
                           special])
    ours = oracle.double_to_half(allx)
    ref = allx.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------ helpers

def dense_attention(q, K, V, scale):
    """softmax(q K^T * scale) V with numpy (q [D], K/V [c, D], float64)."""
    x = (K @ q) * scale
    w = np.exp(x - x.max())
    return (w @ V) / w.sum()


def paged_from_dense(Kd, Vd, ctx, B, NB, rng):
    """Build a paged pool [NB, H, B, D] and block tables from contiguous per-sequence
    K/V [S][c, H, D] by reshaping each sequence into [nb, B, H, D] blocks,
    transposing to [nb, H, B, D] and placing them at a random set of physical ids."""
    S = len(Kd)
    H, D = Kd[0].shape[1], Kd[0].shape[2]
    kc = np.full((NB, H, B, D), np.float16(np.nan), dtype=np.float16)
    vc = kc.copy()
    nbs = [-(-int(c) // B) for c in ctx]
    mb = max(1, max(nbs))
    perm = rng.permutation(NB)
    bt = np.full((S, mb), -1, dtype=np.int32)
    off = 0
    for s in range(S):
        nb = nbs[s]
        ids = perm[off:off + nb]
        off += nb
        bt[s, :nb] = ids
        for X, pool in ((Kd[s], kc), (Vd[s], vc)):
            pad = np.zeros((nb * B, H, D), dtype=np.float16)
            pad[:X.shape[0]] = X
            pool[ids] = pad.reshape(nb, B, H, D).transpose(0, 2, 1, 3)
    return kc, vc, bt


def random_case(rng, S, H, D, B, cmax, cmin=1, spare=3, sigma=1.0):
    ctx = rng.integers(cmin, cmax + 1, S).astype(np.int32)
    Kd = [(sigma * rng.standard_normal((int(c), H, D))).astype(np.float16) for c in ctx]
    Vd = [(sigma * rng.standard_normal((int(c), H, D))).astype(np.float16) for c in ctx]
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    NB = sum(-(-int(c) // B) for c in ctx) + spare
    kc, vc, bt = paged_from_dense(Kd, Vd, ctx, B, NB, rng)
    return q, kc, vc, bt, ctx, Kd, Vd


# ------------------------------------------------------------ decode pins

@pytest.mark.parametrize("S,H,D,B,cmax", [(3, 2, 64, 4, 40), (2, 3, 128, 16, 70),
                                          (4, 1, 32, 32, 100), (2, 2, 16, 8, 33)])
def test_decode_equals_dense_attention(S, H, D, B, cmax):
    rng = np.random.default_rng(S * 1000 + D + B)
    q, kc, vc, bt, ctx, Kd, Vd = random_case(rng, S, H, D, B, cmax)
    scale = 1.0 / math.sqrt(D)
    out16, out64, rc = oracle.decode(q, kc, vc, bt, ctx, scale)
    assert rc == 0
    for s in range(S):
        for h in range(H):
            ref = dense_attention(q[s, h].astype(np.float64), Kd[s][:, h].astype(np.float64),
                                  Vd[s][:, h].astype(np.float64), scale)
            np.testing.assert_allclose(out64[s, h], ref, rtol=1e-12, atol=1e-14)
            # the fp16 output is the double result rounded once (numpy's RNE)
            assert np.array_equal(out16[s, h], out64[s, h].astype(np.float16).view(np.uint16))


def test_decode_scale_is_applied():
    """A wrong or missing scale changes the result: compare two scales against numpy."""
    rng = np.random.default_rng(11)
    q, kc, vc, bt, ctx, Kd, Vd = random_case(rng, 1, 1, 8, 4, 12, cmin=12)
    for scale in (0.125, 0.9):
        _, out64, _ = oracle.decode(q, kc, vc, bt, ctx, scale)
        ref = dense_attention(q[0, 0].astype(np.float64), Kd[0][:, 0].astype(np.float64),
                              Vd[0][:, 0].astype(np.float64), scale)
        np.testing.assert_allclose(out64[0, 0], ref, rtol=1e-12, atol=1e-14)


def test_decode_permutation_invariance():
    rng = np.random.default_rng(21)
    q, kc, vc, bt, ctx, _, _ = random_case(rng, 4, 3, 32, 4, 50)
    a16, a64, _ = oracle.decode(q, kc, vc, bt, ctx, 0.2)
    NB = kc.shape[0]
    pi = rng.permutation(NB)                    # physical id b moves to pi[b]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    bt2 = np.where(bt >= 0, pi[np.maximum(bt, 0)], -1).astype(np.int32)
    b16, b64, _ = oracle.decode(q, kc2, vc2, bt2, ctx, 0.2)
    assert np.array_equal(a16, b16) and np.array_equal(a64, b64)


def test_decode_shared_prefix_identity():
    """Sequences that share prefix blocks by reference give the same bits as
    sequences holding private copies of the prefix."""
    rng = np.random.default_rng(31)
    S, H, D, B, P = 3, 2, 16, 4, 10          # prefix of 10 tokens: 2 full blocks + 2 tokens
    suffix = [5, 1, 9]
    NBp = 3
    prefix_k = rng.standard_normal((NBp, H, B, D)).astype(np.float16)
    prefix_v = rng.standard_normal((NBp, H, B, D)).astype(np.float16)
    ctx = np.array([P + n for n in suffix], dtype=np.int32)
    nbs = [-(-int(c) // B) for c in ctx]
    # Shared layout: blocks 0,1 shared by all; each seq has a private copy of the
    # partial block (copy-on-write) plus its own later blocks.
    NB = 2 + sum(nb - 2 for nb in nbs)
    kc = rng.standard_normal((NB, H, B, D)).astype(np.float16)
    vc = rng.standard_normal((NB, H, B, D)).astype(np.float16)
    kc[:2], vc[:2] = prefix_k[:2], prefix_v[:2]
    bt = np.full((S, max(nbs)), -1, dtype=np.int32)
    nxt = 2
    for s in range(S):
        bt[s, 0], bt[s, 1] = 0, 1
        for j in range(2, nbs[s]):
            bt[s, j] = nxt
            if j == 2:      # the copied partial block keeps the prefix's first 2 tokens
                kc[nxt, :, :2] = prefix_k[2, :, :2]
                vc[nxt, :, :2] = prefix_v[2, :, :2]
            nxt += 1
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    a16, a64, _ = oracle.decode(q, kc, vc, bt, ctx, 0.25)
    # Private layout: every sequence gets its own copy of blocks 0 and 1.
    kc2 = np.concatenate([kc] + [kc[:2]] * S)
    vc2 = np.concatenate([vc] + [vc[:2]] * S)
    bt2 = bt.copy()
    for s in range(S):
        bt2[s, 0], bt2[s, 1] = NB + 2 * s, NB + 2 * s + 1
    b16, b64, _ = oracle.decode(q, kc2, vc2, bt2, ctx, 0.25)
    assert np.array_equal(a16, b16) and np.array_equal(a64, b64)


def test_decode_single_token_returns_value_exactly():
    rng = np.random.default_rng(41)
    q, kc, vc, bt, ctx, Kd, Vd = random_case(rng, 5, 2, 64, 16, 1)
    out16, _, _ = oracle.decode(q, kc, vc, bt, ctx, 0.125)
    for s in range(5):
        assert np.array_equal(out16[s], Vd[s][0].view(np.uint16))


def test_decode_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(51)
    S, H, D, B = 2, 2, 32, 8
    ctx = np.array([13, 30], dtype=np.int32)
    krow = rng.standard_normal((H, D)).astype(np.float16)
    Kd = [np.broadcast_to(krow, (int(c), H, D)).copy() for c in ctx]
    Vd = [rng.standard_normal((int(c), H, D)).astype(np.float16) for c in ctx]
    NB = sum(-(-int(c) // B) for c in ctx)
    kc, vc, bt = paged_from_dense(Kd, Vd, ctx, B, NB, rng)
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    _, out64, _ = oracle.decode(q, kc, vc, bt, ctx, 0.3)
    for s in range(S):
        np.testing.assert_allclose(out64[s], Vd[s].astype(np.float64).mean(axis=0), rtol=1e-13,
                                   atol=1e-15)


def test_decode_constant_values_give_that_constant():
    rng = np.random.default_rng(61)
    S, H, D, B = 2, 3, 16, 4
    ctx = np.array([7, 22], dtype=np.int32)
    vrow = rng.standard_normal((H, D)).astype(np.float16)
    Kd = [rng.standard_normal((int(c), H, D)).astype(np.float16) for c in ctx]
    Vd = [np.broadcast_to(vrow, (int(c), H, D)).copy() for c in ctx]
    NB = sum(-(-int(c) // B) for c in ctx) + 2
    kc, vc, bt = paged_from_dense(Kd, Vd, ctx, B, NB, rng)
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    out16, out64, _ = oracle.decode(q, kc, vc, bt, ctx, 0.7)
    for s in range(S):
        np.testing.assert_allclose(out64[s], vrow.astype(np.float64), rtol=1e-14, atol=0)
        assert np.array_equal(out16[s], vrow.view(np.uint16))


def test_decode_dominant_logit_selects_its_value():
    """q aligned with one key at a large scale: softmax puts all weight on it.
    Logits reach ~1e4, so a softmax without max subtraction would overflow."""
    rng = np.random.default_rng(71)
    S, H, D, B, c = 1, 1, 8, 4, 11
    Kd = [rng.standard_normal((c, H, D)).astype(np.float16)]
    Vd = [rng.standard_normal((c, H, D)).astype(np.float16)]
    j = 6
    Kd[0][j, 0] = np.float16(8.0)
    q = np.full((1, 1, D), 8.0, dtype=np.float16)
    kc, vc, bt = paged_from_dense(Kd, Vd, np.array([c]), B, 4, rng)
    out16, out64, _ = oracle.decode(q, kc, vc, bt, np.array([c], dtype=np.int32), 20.0)
    assert np.all(np.isfinite(out64))
    assert np.array_equal(out16[0, 0], Vd[0][j, 0].view(np.uint16))


def test_decode_two_tokens_by_hand():
    """D=2, c=2: q=(1,0), K=[(1,0),(0,1)], V=[(1,0),(0,1)], scale 1/sqrt(2):
    logits (1/sqrt2, 0), so out = (sigma, 1 - sigma) with sigma = 1/(1+e^{-1/sqrt2})."""
    kc = np.zeros((1, 1, 4, 2), dtype=np.float16)
    vc = np.zeros((1, 1, 4, 2), dtype=np.float16)
    kc[0, 0, 0], kc[0, 0, 1] = (1, 0), (0, 1)
    vc[0, 0, 0], vc[0, 0, 1] = (1, 0), (0, 1)
    q = np.array([[[1, 0]]], dtype=np.float16)
    _, out64, _ = oracle.decode(q, kc, vc, np.array([[0]], np.int32), np.array([2], np.int32),
                                1 / math.sqrt(2))
    sig = 1.0 / (1.0 + math.exp(-1.0 / math.sqrt(2.0)))
    assert abs(out64[0, 0, 0] - sig) < 1e-15 and abs(out64[0, 0, 1] - (1 - sig)) < 1e-15
    assert abs(sig - 0.6697615493266569) < 1e-15


def test_decode_empty_context_gives_zero_row():
    q = np.ones((2, 1, 8), dtype=np.float16)
    kc = np.ones((2, 1, 4, 8), dtype=np.float16)
    out16, out64, rc = oracle.decode(q, kc, kc, np.array([[0], [1]], np.int32),
                                     np.array([0, 3], np.int32), 0.5)
    assert rc == 0 and np.all(out64[0] == 0) and np.all(out16[0] == 0)
    np.testing.assert_allclose(out64[1], 1.0)


def _brute_force(q, kc, vc, bt, ctx, scale):
    S, H, D = q.shape
    B = kc.shape[2]
    out = np.zeros((S, H, D))
    for s in range(S):
        for h in range(H):
            c = int(ctx[s])
            logits = []
            for i in range(c):
                phys = int(bt[s][i // B])
                logits.append(sum(float(q[s, h, d]) * float(kc[phys, h, i % B, d]) for d in range(D))
                              * scale)
            if c == 0:
                continue
            m = max(logits)
            ws = [math.exp(x - m) for x in logits]
            tot = sum(ws)
            for d in range(D):
                out[s, h, d] = sum(ws[i] * float(vc[int(bt[s][i // B]), h, i % B, d])
                                   for i in range(c)) / tot
    return out


@pytest.mark.parametrize("B", [1, 2, 4])
def test_decode_brute_force_tiny_grid(B):
    rng = np.random.default_rng(100 + B)
    for S in (1, 2):
        for H in (1, 2):
            for cmax in (1, 4, 9):
                q, kc, vc, bt, ctx, _, _ = random_case(rng, S, H, 4, B, cmax, cmin=0)
                _, out64, rc = oracle.decode(q, kc, vc, bt, ctx, 0.5)
                assert rc == 0
                np.testing.assert_allclose(out64, _brute_force(q, kc, vc, bt, ctx, 0.5),
                                           rtol=1e-12, atol=1e-14)


def test_decode_reads_only_live_slots():
    """NaN everywhere outside the live tokens (unused blocks and the tail of each
    last block) must not reach the output."""
    rng = np.random.default_rng(81)
    q, kc, vc, bt, ctx, _, _ = random_case(rng, 4, 2, 16, 4, 30, spare=5)
    out16, out64, _ = oracle.decode(q, kc, vc, bt, ctx, 0.25)
    assert np.all(np.isfinite(out64))


# ------------------------------------------------------- address map pins

def test_worked_example_slots():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_block_table.json")))
    B = g["block_size"]
    bt = np.array([g["block_table_A"]], dtype=np.int32)
    for pos, blk, off in g["position_to_block_offset"]:
        slots, rc = oracle.slot_mapping(bt, np.array([0], np.int32), np.array([pos], np.int32), B, 8)
        assert rc == 0 and slots[0] == blk * B + off
    for pos, slot in g["slot_of_position"]:
        slots, _ = oracle.slot_mapping(bt, np.array([0], np.int32), np.array([pos], np.int32), B, 8)
        assert slots[0] == slot


def test_slot_mapping_against_table_lookup():
    w = configs.config2()
    seqs, pos = w.new_tokens()
    slots, rc = oracle.slot_mapping(w.block_tables, seqs, pos, w.block_size, w.num_blocks)
    assert rc == 0
    # every slot lies in the block the table names, at the right offset
    blocks = slots // w.block_size
    offs = slots % w.block_size
    assert np.array_equal(blocks, w.block_tables[seqs, pos // w.block_size])
    assert np.array_equal(offs, pos % w.block_size)
    # padding tokens and out-of-range entries
    s2, rc2 = oracle.slot_mapping(w.block_tables, np.array([-1, 0], np.int32),
                                  np.array([0, 10 ** 6], np.int32), w.block_size, w.num_blocks)
    assert s2[0] == -1 and s2[1] == -1 and rc2 != 0


# ---------------------------------------------- cache write / copy pins

def test_reshape_and_cache_matches_numpy_scatter():
    rng = np.random.default_rng(91)
    NB, H, B, D, T = 9, 3, 4, 16, 20
    kc = rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint64).astype(np.uint16)
    vc = rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint64).astype(np.uint16)
    k = rng.integers(0, 1 << 16, (T, H, D), dtype=np.uint64).astype(np.uint16)
    v = rng.integers(0, 1 << 16, (T, H, D), dtype=np.uint64).astype(np.uint16)
    slots = rng.permutation(NB * B)[:T].astype(np.int64)
    slots[[3, 11]] = -1                                   # padding tokens
    ek, ev = kc.copy(), vc.copy()
    live = slots >= 0
    # numpy's view: the pool as [NB, B, H, D] slots, flattened to [NB*B] x [H, D]
    ekv = ek.transpose(0, 2, 1, 3).reshape(NB * B, H, D).copy()
    evv = ev.transpose(0, 2, 1, 3).reshape(NB * B, H, D).copy()
    ekv[slots[live]] = k[live]
    evv[slots[live]] = v[live]
    ek = ekv.reshape(NB, B, H, D).transpose(0, 2, 1, 3)
    ev = evv.reshape(NB, B, H, D).transpose(0, 2, 1, 3)
    rc = oracle.reshape_and_cache(kc, vc, k, v, slots, B)
    assert rc == 0
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_copy_blocks_matches_numpy():
    rng = np.random.default_rng(93)
    L, NB, H, B, D = 3, 12, 2, 4, 8
    kcs = [rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint64).astype(np.uint16) for _ in range(L)]
    vcs = [rng.integers(0, 1 << 16, (NB, H, B, D), dtype=np.uint64).astype(np.uint16) for _ in range(L)]
    pairs = np.array([[0, 5], [3, 7], [2, 11]], dtype=np.int64)
    ek = [x.copy() for x in kcs]
    ev = [x.copy() for x in vcs]
    for src, dst in pairs:
        for l in range(L):
            ek[l][dst] = ek[l][src]
            ev[l][dst] = ev[l][src]
    assert oracle.copy_blocks(kcs, vcs, pairs) == 0
    for l in range(L):
        assert np.array_equal(kcs[l], ek[l]) and np.array_equal(vcs[l], ev[l])


# ------------------------------------------------- generator sanity (inputs)

def test_generator_matches_splitmix64_definition():
    # Published first outputs of SplitMix64 seeded with 0.
    assert synth.splitmix_at(0, 0) == 0xE220A8397B1DCDAF
    assert synth.splitmix_at(0, 1) == 0x6E789E6AA1B965F4
    lib = synth._lib()
    for x0, i in [(0, 0), (12345, 7), (2 ** 63 + 5, 10 ** 9)]:
        assert lib.synth_splitmix64_at(x0, i) == synth.splitmix_at(x0, i)
    bank = synth.fp16_bank(7, 1.0)
    vals = synth.host_values(7, 3, 1000, 64, bank)
    base = synth.stream_base(7, 3)
    expect = [bank[synth.splitmix_at(base, 1000 + i) >> (64 - synth.BANK_BITS)] for i in range(64)]
    assert np.array_equal(vals, np.array(expect, dtype=np.uint16))
    z = synth.normal_bank(7)
    assert abs(z.mean()) < 2e-3 and abs(z.std() - 1) < 2e-3


def test_swap_blocks_matches_numpy():
    """Swap out then in between pools of different sizes (block-id spaces) and
    element types: each destination block equals its source block byte for byte."""
    rng = np.random.default_rng(11)
    dev = [rng.integers(0, 1 << 16, (12, 2, 4, 8), dtype=np.uint16) for _ in range(3)]
    host = [np.zeros((7, 2, 4, 8), dtype=np.uint16) for _ in range(3)]
    out_map = np.array([[3, 0], [11, 6], [0, 2]], dtype=np.int64)
    assert oracle.swap_blocks(host, dev, out_map) == 0
    for c in range(3):
        assert np.array_equal(host[c][[0, 6, 2]], dev[c][[3, 11, 0]])
        assert not host[c][[1, 3, 4, 5]].any()
    dev2 = [np.zeros_like(d) for d in dev]
    in_map = np.array([[6, 1], [0, 9]], dtype=np.int64)
    assert oracle.swap_blocks(dev2, host, in_map) == 0
    for c in range(3):
        assert np.array_equal(dev2[c][1], dev[c][11]) and np.array_equal(dev2[c][9], dev[c][3])
    # byte pools (FP8 caches) and out-of-range ids
    a = rng.integers(0, 256, (5, 64), dtype=np.uint8)
    b = np.zeros((4, 64), dtype=np.uint8)
    assert oracle.swap_blocks([b], [a], np.array([[4, 3], [5, 0], [1, 4]], np.int64)) == -1
    assert np.array_equal(b[3], a[4]) and not b[0].any()

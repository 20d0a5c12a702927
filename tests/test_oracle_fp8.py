"""Pins for the oracle's FP8 (E4M3) KV-cache functions, independent of the
oracle's own code.

* E4M3 decoding of all 256 codes against PyTorch's ``float8_e4m3fn``
  conversion (library routine) and the format's closed forms;
* E4M3 encoding (round to nearest even) against PyTorch's conversion inside
  the finite range, including every midpoint and its neighbours; saturation
  to +-448 beyond it from the closed form (PyTorch gives NaN there);
* the FP8 cache write against numpy scatter of PyTorch-quantised values;
* FP8 decode against dense numpy attention on the dequantised K/V, with
  different key and value scales so that swapping them fails.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import dense_attention, random_case


def torch_e4m3_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_e4m3_encode_f32(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_double(codes)
    ref = torch_e4m3_decode(codes)
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e4m3_closed_forms():
    v = oracle.e4m3_to_double(np.array([0x7E, 0x08, 0x01, 0x07, 0x38, 0x40, 0x30, 0xB8],
                                       dtype=np.uint8))
    # largest finite; smallest normal 2^-6; smallest subnormal 2^-9; largest
    # subnormal 7 * 2^-9; 1; 2; 1/2; -1
    assert list(v) == [448.0, 2.0 ** -6, 2.0 ** -9, 7 * 2.0 ** -9, 1.0, 2.0, 0.5, -1.0]


def test_e4m3_encode_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = torch_e4m3_decode(codes)
    assert np.array_equal(oracle.double_to_e4m3(vals), codes)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(200000) * np.exp2(rng.uniform(-12, 8.5, 200000))).astype(np.float32)
    codes = np.arange(0, 0x7E, dtype=np.uint8)
    lo = torch_e4m3_decode(codes)
    hi = torch_e4m3_decode(codes + 1)
    mid = ((lo + hi) / 2).astype(np.float32)          # exact: 5 significant bits
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)
    special = np.array([448.0, 450.0, 463.9, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11,
                        2.0 ** -11, 0.0, -0.0], dtype=np.float32)
    allx = np.concatenate([x, -x, mid, -mid, np.nextafter(mid, np.float32(np.inf)),
                           np.nextafter(mid, np.float32(-np.inf)), special])
    allx = allx[np.abs(allx) < 464.0]                 # PyTorch's conversion is NaN beyond
    ours = oracle.double_to_e4m3(allx.astype(np.float64))
    assert np.array_equal(ours, torch_e4m3_encode_f32(allx))
    # ties go to the even code
    t = oracle.double_to_e4m3(np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10]))
    assert list(t) == [0x38, 0x3A, 0x00, 0x02]


def test_e4m3_encode_saturates():
    x = np.array([464.0, 465.0, 1e6, np.inf, -464.0, -1e30, -np.inf])
    assert list(oracle.double_to_e4m3(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0xFE]
    assert oracle.double_to_e4m3(np.array([np.nan]))[0] == 0x7F


@pytest.mark.parametrize("D,B", [(64, 16), (128, 32)])
def test_fp8_cache_write_matches_torch_quantisation(D, B):
    rng = np.random.default_rng(D + B)
    T, H, NB = 37, 3, 8
    key = (rng.standard_normal((T, H, D)) * 2).astype(np.float16)
    value = (rng.standard_normal((T, H, D)) * 0.5).astype(np.float16)
    slots = rng.choice(NB * B, T, replace=False).astype(np.int64)
    slots[5] = -1                                     # padding token
    k_scale, v_scale = 0.0625, 0.01171875
    kc = np.full((NB, H, B, D), 0xAB, dtype=np.uint8)
    vc = kc.copy()
    assert oracle.reshape_and_cache_fp8(kc, vc, key, value, slots, B, k_scale, v_scale) == 0
    ek, ev = kc.copy(), vc.copy()
    ek.fill(0xAB)
    ev.fill(0xAB)
    qk = torch_e4m3_encode_f32(key.astype(np.float32) / np.float32(k_scale))
    qv = torch_e4m3_encode_f32(value.astype(np.float32) / np.float32(v_scale))
    for t in range(T):
        if slots[t] < 0:
            continue
        ek[slots[t] // B, :, slots[t] % B] = qk[t]
        ev[slots[t] // B, :, slots[t] % B] = qv[t]
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


@pytest.mark.parametrize("S,H,D,B,cmax", [(3, 2, 64, 16, 90), (2, 3, 128, 32, 130)])
def test_fp8_decode_equals_dense_attention_on_dequantised_kv(S, H, D, B, cmax):
    rng = np.random.default_rng(S * 100 + D)
    q, kc16, vc16, bt, ctx, _, _ = random_case(rng, S, H, D, B, cmax)
    # an arbitrary byte pattern per slot (NaN codes excluded) stands for the cache
    kc = rng.integers(0, 0x7E, kc16.shape).astype(np.uint8) | (rng.integers(0, 2, kc16.shape) << 7).astype(np.uint8)
    vc = rng.integers(0, 0x7E, vc16.shape).astype(np.uint8) | (rng.integers(0, 2, vc16.shape) << 7).astype(np.uint8)
    k_scale, v_scale = 0.01, 0.003
    scale = 1.0 / math.sqrt(D)
    out16, out64, rc = oracle.decode_fp8(q, kc, vc, bt, ctx, scale, k_scale, v_scale)
    assert rc == 0
    Kf = torch_e4m3_decode(kc) * k_scale
    Vf = torch_e4m3_decode(vc) * v_scale
    for s in range(S):
        c = int(ctx[s])
        blocks = bt[s, :-(-c // B)]
        Kd = Kf[blocks].transpose(0, 2, 1, 3).reshape(-1, H, D)[:c]
        Vd = Vf[blocks].transpose(0, 2, 1, 3).reshape(-1, H, D)[:c]
        for h in range(H):
            ref = dense_attention(q[s, h].astype(np.float64), Kd[:, h], Vd[:, h], scale)
            np.testing.assert_allclose(out64[s, h], ref, rtol=1e-12, atol=1e-15)
            assert np.array_equal(out16[s, h], out64[s, h].astype(np.float16).view(np.uint16))


def test_fp8_decode_empty_context_and_bad_block():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((2, 1, 64)).astype(np.float16)
    kc = np.zeros((2, 1, 16, 64), dtype=np.uint8)
    bt = np.array([[0], [0]], dtype=np.int32)
    out16, _, rc = oracle.decode_fp8(q, kc, kc, bt, np.array([0, 3], np.int32), 0.1, 1.0, 1.0)
    assert rc == 0 and not out16[0].any()
    bt[1, 0] = 5
    _, _, rc = oracle.decode_fp8(q, kc, kc, bt, np.array([0, 3], np.int32), 0.1, 1.0, 1.0)
    assert rc != 0


@pytest.mark.parametrize("scale", [1.0, 0.37, 0.0625, 3.0])
def test_quantize_every_fp16_pattern_matches_torch(scale):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x16 = bits.view(np.float16)
    finite = np.isfinite(x16)
    ours = oracle.quantize_e4m3(bits[finite], scale)
    q32 = x16[finite].astype(np.float32) / np.float32(scale)      # IEEE binary32 division
    inrange = np.abs(q32) < 464.0
    assert np.array_equal(ours[inrange], torch_e4m3_encode_f32(q32[inrange]))
    # beyond the finite range: +-448 with the value's sign
    big = ~inrange
    assert np.all(ours[big] == np.where(q32[big] > 0, 0x7E, 0xFE))
    inf = oracle.quantize_e4m3(np.array([0x7C00, 0xFC00], dtype=np.uint16), scale)
    assert list(inf) == [0x7E, 0xFE]

"""Pins of the FP8 (E4M3) parts of the oracle, independent of the oracle's
own arithmetic:
  * every one of the 256 codes decodes to the value torch's independent
    float8_e4m3fn conversion gives (NaN codes included), and the format's
    landmarks hold (largest 448, smallest subnormal 2^-9, smallest normal
    2^-6, 1.0 = 0x38, 126 positive finite non-zero codes, strictly monotone);
  * encoding agrees with torch's round-to-nearest-even conversion on random
    values, on every midpoint between neighbouring codes (ties to the even
    code) and on every code value itself, and saturates to +-448 where torch
    (which does not saturate) gives NaN;
  * the rounding error is at most half a grid step;
  * the quantizing scatter equals torch's conversion of (x / scale) computed
    in fp32, element by element;
  * the dequantized decode reduces exactly to the bf16 oracle (already pinned)
    when the pool holds values that bf16 represents exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_218_gb300 import workload as W


def torch_e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_values_match_an_independent_decoder():
    ref = torch_e4m3_values()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and nan.sum() == 2
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def test_e4m3_landmarks():
    v = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert v[0x7E] == 448.0 and v[1] == 2.0 ** -9 and v[8] == 2.0 ** -6 and v[0x38] == 1.0
    assert all(a < b for a, b in zip(v, v[1:])) and sum(1 for x in v if x > 0) == 126
    assert np.isnan(oracle.e4m3_value(0x7F)) and np.isnan(oracle.e4m3_value(0xFF))


def torch_encode(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_rounding():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(4000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x.astype(np.float32)
    x = x[np.abs(x) < 448]
    mine = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    assert np.array_equal(mine, torch_encode(x))


def test_e4m3_encode_ties_and_exact_values():
    vals = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    for sign in (1.0, -1.0):
        exact = (sign * vals).astype(np.float32)
        assert np.array_equal(np.array([oracle.e4m3_encode(v) for v in exact], np.uint8),
                              torch_encode(exact))
        mids = (sign * (vals[:-1] + vals[1:]) / 2).astype(np.float32)  # exact in fp32
        got = np.array([oracle.e4m3_encode(v) for v in mids], np.uint8)
        assert np.array_equal(got, torch_encode(mids))
        assert np.all(got % 2 == 0)  # ties go to the even code


def test_e4m3_encode_saturates():
    for v, code in ((448.0, 0x7E), (463.99, 0x7E), (464.0, 0x7E), (1e6, 0x7E),
                    (float("inf"), 0x7E), (-500.0, 0xFE), (float("-inf"), 0xFE)):
        assert oracle.e4m3_encode(v) == code, v
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_e4m3_rounding_error_is_at_most_half_a_step():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * 40).astype(np.float32)
    x = x[np.abs(x) < 448]
    q = np.array([oracle.e4m3_value(oracle.e4m3_encode(v)) for v in x])
    a = np.abs(x.astype(np.float64))
    k = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    step = 2.0 ** (k - 3)
    assert np.all(np.abs(q - x) <= step / 2)


def test_quantizing_scatter_is_elementwise_torch_conversion():
    rng = np.random.default_rng(5)
    T, Hkv, D, nb = 20, 3, 32, 4
    key, value = W.normal_bf16(rng, (T, Hkv, D)), W.normal_bf16(rng, (T, Hkv, D))
    ks = np.array([0.01, 0.02, 0.0031], np.float32)
    vs = np.array([0.5, 0.007, 1.0], np.float32)
    slots = rng.permutation(nb * 16)[:T].astype(np.int64)
    slots[3] = -1
    kc, vc = oracle.reshape_and_cache_fp8(key, value, np.zeros((nb, 16, Hkv, D), np.uint8),
                                          np.zeros((nb, 16, Hkv, D), np.uint8), slots, ks, vs)
    kf = W.bf16_bits_to_f32(key)
    vf = W.bf16_bits_to_f32(value)
    for t in range(T):
        s = slots[t]
        if s < 0:
            continue
        for x, sc, pool in ((kf, ks, kc), (vf, vs, vc)):
            r = (x[t] / sc[:, None]).astype(np.float32)  # fp32 division, as specified
            want = np.where(np.abs(r) >= 448, np.where(r < 0, 0xFE, 0x7E), torch_encode(r))
            assert np.array_equal(pool[s // 16, s % 16], want.astype(np.uint8))
    assert np.all(kc.reshape(-1, Hkv, D)[np.setdiff1d(np.arange(nb * 16), slots[slots >= 0])] == 0)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (8, 8), (6, 1)])
def test_dequantized_decode_reduces_to_the_bf16_oracle(Hq, Hkv):
    """Codes times power-of-two scales are exact in bf16, so the fp8 oracle
    must equal the bf16 oracle on the dequantized pool."""
    rng = np.random.default_rng(9)
    D, nb, S = 32, 12, 3
    kc = rng.integers(0, 256, (nb, 16, Hkv, D)).astype(np.uint8)
    vc = rng.integers(0, 256, (nb, 16, Hkv, D)).astype(np.uint8)
    for pool in (kc, vc):  # no NaN codes where the tokens live
        pool[(pool & 0x7F) == 0x7F] = 0x3C
    ks = (2.0 ** rng.integers(-8, 3, Hkv)).astype(np.float32)
    vs = (2.0 ** rng.integers(-8, 3, Hkv)).astype(np.float32)
    lens = np.array([1, 17, 70], np.int32)
    bt = np.full((S, 5), -1, np.int32)
    ids = rng.permutation(nb)
    k = 0
    for s_, n in enumerate(lens):
        for j in range(-(-n // 16)):
            bt[s_, j] = ids[k]
            k += 1
    q = W.normal_bf16(rng, (S, Hq, D))

    def deq(pool, sc):
        v = np.vectorize(oracle.e4m3_value)(pool) * sc[None, None, :, None]
        return W.f32_to_bf16_bits(v.astype(np.float32))

    kb, vb = deq(kc, ks), deq(vc, vs)
    assert np.array_equal(W.bf16_bits_to_f32(kb), (np.vectorize(oracle.e4m3_value)(kc)
                                                   * ks[None, None, :, None]).astype(np.float32))
    o8, l8 = oracle.decode_fp8(q, kc, vc, ks, vs, bt, lens, 0.17)
    o16, l16 = oracle.decode(q, kb, vb, bt, lens, 0.17)
    np.testing.assert_allclose(o8, o16, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l8, l16, rtol=1e-12, atol=1e-12)

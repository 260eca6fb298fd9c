"""Pins for the oracle's e4m3 format, block quantiser and FP8 attention
("GPU 内核与 FlashAttention" §15.5).

The e4m3 decoder is checked against values the format definition fixes
(1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals below 2^-6,
one NaN pattern, largest finite 448); the encoder against round-trips,
rounding-to-nearest with ties to the even mantissa, and saturation; the FP8
attention against the already-pinned bf16 oracle on inputs that e4m3
represents exactly, and against the scale's closed-form effect.
"""
import numpy as np
import pytest
import torch

from attention_forward_fa2_gb300 import inputs as I


def test_e4m3_values_fixed_by_the_format(oracle_mod):
    d = oracle_mod.e4m3_decode
    assert d(0x38) == 1.0 and d(0x40) == 2.0 and d(0x30) == 0.5
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert d(0x08) == 2.0 ** -6                      # smallest normal
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9   # subnormals
    assert d(0x00) == 0.0 and np.signbit(d(0x80))
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    vals = d(np.arange(0x7F))
    assert np.all(np.diff(vals) > 0)                  # codes 0..0x7e increase
    assert np.array_equal(d(np.arange(0x80, 0xFF)), -vals)


def test_e4m3_encode_round_trip_and_rounding(oracle_mod):
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = oracle_mod.e4m3_decode(codes)
    assert np.array_equal(oracle_mod.e4m3_encode(vals), codes)
    assert np.array_equal(oracle_mod.e4m3_encode(-vals[1:]), codes[1:] | 0x80)
    # midpoints go to the even mantissa, anything else to the nearer value
    mids = (vals[:-1] + vals[1:]) / 2
    enc = oracle_mod.e4m3_encode(mids)
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(enc, even)
    rng = np.random.default_rng(3)
    x = rng.uniform(0, 448, 2000)
    e = oracle_mod.e4m3_decode(oracle_mod.e4m3_encode(x))
    gap = np.abs(vals[None, :] - x[:, None]).min(axis=1)
    assert np.allclose(np.abs(e - x), gap)
    assert list(oracle_mod.e4m3_encode([448.0, 460.0, 1e6, -1e6])) == [0x7E, 0x7E, 0x7E, 0xFE]
    # zeros and values that round to zero keep their sign (round to nearest is sign-symmetric)
    assert list(oracle_mod.e4m3_encode([0.0, -0.0, 2.0 ** -11, -(2.0 ** -11), 2.0 ** -10, -(2.0 ** -10)])) == \
        [0x00, 0x80, 0x00, 0x80, 0x00, 0x80]
    assert list(oracle_mod.e4m3_encode([1.5 * 2.0 ** -10, -1.5 * 2.0 ** -10])) == [0x01, 0x81]


def test_block_quantiser_bounds(oracle_mod):
    g = torch.Generator().manual_seed(4)
    q = I.randn_bf16((1, 200, 2, 128), g) * 3
    k = I.randn_bf16((1, 130, 1, 128), g)
    v = I.randn_bf16((1, 130, 1, 128), g)
    q8, k8, vt8, qs, ks, vs = oracle_mod.quantize_fp8(I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v))
    assert vt8.shape == (1, 1, 128, 144) and np.all(vt8[..., 130:] == 0)
    qf = q.float().numpy()
    for blk in range(2):
        x = qf[0, blk * 128:(blk + 1) * 128, 0]
        s = qs[0, 0, blk]
        assert s == np.float32(np.abs(x).max() / np.float32(448))
        y = oracle_mod.e4m3_decode(q8[0, blk * 128:(blk + 1) * 128, 0]) * s
        # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 above 2^-6 * s
        big = np.abs(x) >= 2 ** -6 * s
        assert np.all(np.abs(y - x)[big] <= 2 ** -4 * np.abs(x)[big] + 1e-12)
        assert np.all(np.abs(y - x)[~big] <= 2 ** -10 * s + 1e-12)
        assert np.abs(oracle_mod.e4m3_decode(q8[0, blk * 128:(blk + 1) * 128, 0])).max() == 448.0
    # V is stored transposed: [b, hk, c, j] holds key j, feature c
    v_back = oracle_mod.e4m3_decode(vt8[0, 0, :, :130]).T * vs[0, 0]
    assert np.allclose(v_back, v.float().numpy()[0, :, 0], rtol=2 ** -4, atol=2 ** -10 * vs[0, 0])


def _exact_codes(shape, seed, oracle_mod):
    """Random codes whose values are moderate (|x| in [2^-3, 4]), as numbers and codes."""
    rng = np.random.default_rng(seed)
    pool = np.array([c for c in range(0x7F) if 0.125 <= oracle_mod.e4m3_decode(c) <= 4.0], np.uint8)
    codes = rng.choice(pool, size=shape) | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)
    return codes


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_attention_equals_bf16_oracle_on_exact_values(oracle_mod, causal):
    B, Nq, Nk, H, Hk, d = 1, 70, 150, 2, 1, 128
    q8 = _exact_codes((B, Nq, H, d), 1, oracle_mod)
    k8 = _exact_codes((B, Nk, Hk, d), 2, oracle_mod)
    v8 = _exact_codes((B, Nk, Hk, d), 3, oracle_mod)
    nkp = (Nk + 15) // 16 * 16
    vt8 = np.zeros((B, Hk, d, nkp), np.uint8)
    vt8[:, :, :, :Nk] = v8.transpose(0, 2, 3, 1)
    ones = lambda *s: np.ones(s, np.float32)
    o8, l8 = oracle_mod.attn_fp8_dense(q8, k8, vt8, ones(B, H, 1), ones(B, Hk, 2), ones(B, Hk), Nq, Nk,
                                       scale=0.05, causal=causal)
    bf = lambda c: I.bf16_bits(torch.from_numpy(oracle_mod.e4m3_decode(c).astype(np.float32)).to(torch.bfloat16))
    ob, lb = oracle_mod.attn_dense(bf(q8), bf(k8), bf(v8), scale=0.05, causal=causal)
    assert np.allclose(o8, ob, rtol=1e-13, atol=1e-13)
    assert np.allclose(l8, lb, rtol=1e-13, atol=1e-13)


def test_fp8_scales_act_as_multipliers(oracle_mod):
    """Doubling every query scale equals doubling the softmax scale; a V scale
    multiplies O and leaves the LSE alone."""
    B, Nq, Nk, H, d = 1, 40, 90, 1, 128
    q8 = _exact_codes((B, Nq, H, d), 4, oracle_mod)
    k8 = _exact_codes((B, Nk, H, d), 5, oracle_mod)
    vt8 = np.zeros((B, H, d, 96), np.uint8)
    vt8[..., :Nk] = _exact_codes((B, H, d, Nk), 6, oracle_mod)
    one = lambda *s: np.ones(s, np.float32)
    o1, l1 = oracle_mod.attn_fp8_dense(q8, k8, vt8, one(B, H, 1) * 2, one(B, H, 1), one(B, H) * 3, Nq, Nk, scale=0.02)
    o2, l2 = oracle_mod.attn_fp8_dense(q8, k8, vt8, one(B, H, 1), one(B, H, 1), one(B, H), Nq, Nk, scale=0.04)
    assert np.allclose(o1, 3 * o2, rtol=1e-12, atol=1e-12)
    assert np.allclose(l1, l2, rtol=1e-12, atol=1e-12)

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


def _dequant(oracle_mod, q8, k8, vt8, qs, ks, vs, Nq, Nk):
    """Dequantised q [B, Nq, H, d], k [B, Nk, Hk, d], v [B, Nk, Hk, d] in float64."""
    dec = oracle_mod.e4m3_decode
    q = dec(q8) * np.repeat(qs, 128, axis=2)[:, :, :Nq].transpose(0, 2, 1)[..., None]
    k = dec(k8) * np.repeat(ks, 128, axis=2)[:, :, :Nk].transpose(0, 2, 1)[..., None]
    v = dec(vt8[..., :Nk]).transpose(0, 3, 1, 2) * vs[:, None, :, None]
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_bound_terms_brute_force(oracle_mod, causal):
    """Row maximum and sum_j P_ij |v_j| against a direct numpy evaluation."""
    B, Nq, Nk, H, Hk, d = 2, 9, 7, 4, 2, 128
    g = torch.Generator().manual_seed(12)
    q, k, v = (I.randn_bf16(s, g) for s in ((B, Nq, H, d), (B, Nk, Hk, d), (B, Nk, Hk, d)))
    codes = oracle_mod.quantize_fp8(I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v))
    o, lse, m, a = oracle_mod.attn_fp8_dense(*codes, Nq, Nk, causal=causal, with_bound_terms=True)
    qf, kf, vf = _dequant(oracle_mod, *codes, Nq, Nk)
    sc = 1 / np.sqrt(d)
    for b in range(B):
        for h in range(H):
            s = sc * qf[b, :, h] @ kf[b, :, h // 2].T
            if causal:
                s[np.arange(Nk)[None, :] > np.arange(Nq)[:, None] + Nk - Nq] = -np.inf
            mx = s.max(axis=1)
            assert np.allclose(m[b, h], mx, rtol=1e-13, atol=1e-13)
            seen = np.isfinite(mx)
            p = np.exp(s[seen] - mx[seen, None])
            p /= p.sum(axis=1, keepdims=True)
            assert np.allclose(a[b, seen, h], p @ np.abs(vf[b, :, h // 2]), rtol=1e-12, atol=1e-13)
            assert np.allclose(o[b, seen, h], p @ vf[b, :, h // 2], rtol=1e-12, atol=1e-13)
            assert np.all(a[b, ~seen, h] == 0) and np.all(np.isneginf(m[b, h][~seen]))
    # the log-sum-exp lies between the row maximum and the maximum plus log(keys seen)
    fin = np.isfinite(lse)
    assert np.all(lse[fin] >= m[fin] - 1e-12) and np.all(lse[fin] <= m[fin] + np.log(Nk) + 1e-12)


def test_fp8_bound_terms_invariants(oracle_mod):
    """V with non-negative codes: sum_j P_ij |v_j| equals O; flipping the sign
    of every V code negates O and leaves the magnitudes' sum alone."""
    B, Nq, Nk, H, d = 1, 30, 70, 2, 128
    q8 = _exact_codes((B, Nq, H, d), 7, oracle_mod)
    k8 = _exact_codes((B, Nk, H, d), 8, oracle_mod)
    vt8 = np.zeros((B, H, d, 80), np.uint8)
    vt8[..., :Nk] = _exact_codes((B, H, d, Nk), 9, oracle_mod) & 0x7F
    one = lambda *s: np.ones(s, np.float32)
    args = (one(B, H, 1), one(B, H, 1), one(B, H), Nq, Nk)
    o, _, _, a = oracle_mod.attn_fp8_dense(q8, k8, vt8, *args, scale=0.03, with_bound_terms=True)
    assert np.allclose(a, o, rtol=1e-13, atol=0)
    o2, _, _, a2 = oracle_mod.attn_fp8_dense(q8, k8, vt8 | 0x80, *args, scale=0.03, with_bound_terms=True)
    assert np.array_equal(o2, -o) and np.array_equal(a2, a)


def _blocky_codes(oracle_mod, seed, Nq=256, Nk=512, H=2, Hk=1):
    """N(0,1) inputs whose 128-key blocks differ in amplitude (ratios up to 1.33)."""
    g = torch.Generator().manual_seed(seed)
    q = I.randn_bf16((1, Nq, H, 128), g)
    k = I.randn_bf16((1, Nk, Hk, 128), g)
    v = I.randn_bf16((1, Nk, Hk, 128), g)
    amp = torch.tensor([1.0, 1.2, 0.9, 1.1]).repeat_interleave(128)[:Nk]
    k = (k.float() * amp[None, :, None, None]).to(torch.bfloat16)
    return oracle_mod.quantize_fp8(I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v))


def test_fp8_bar_holds_for_rounded_weights(oracle_mod):
    """The bar covers what it claims: weights relative to a reference below the
    row maximum (by up to the rescale threshold, 8 in log2 units), rounded to
    e4m3, with the sum of the unrounded weights, stay within it."""
    from fa_testutil import fp8_bound
    Nq, Nk = 64, 512
    codes = _blocky_codes(oracle_mod, 21, Nq=Nq, Nk=Nk, H=1)
    o_ref, _, bound = fp8_bound(oracle_mod, *codes, Nq, Nk)
    qf, kf, vf = _dequant(oracle_mod, *codes, Nq, Nk)
    s = qf[0, :, 0] @ kf[0, :, 0].T / np.sqrt(128)
    lag = np.random.default_rng(5).uniform(0, 8 * np.log(2), Nq)   # reference below the maximum
    p = np.exp(s - (s.max(axis=1) - lag)[:, None])
    assert p.max() <= 256.0 * (1 + 1e-12)
    p8 = oracle_mod.e4m3_decode(oracle_mod.e4m3_encode(p))
    o_emul = (p8 @ vf[0, :, 0]) / p.sum(axis=1, keepdims=True)
    err = np.abs(o_emul - o_ref[0, :, 0])
    assert np.all(err <= bound[0, :, 0]), float((err - bound[0, :, 0]).max())


def test_fp8_bar_rejects_a_neighbouring_block_scale(oracle_mod):
    """An output computed with one key block's scale taken from the next block
    (what a kernel indexing the scales one block off would write) breaks the
    per-element bar, while the earlier global bar 2^-4 max|v| + 2e-2 on O
    would have let it through."""
    from fa_testutil import fp8_bound
    Nq, Nk = 256, 512
    q8, k8, vt8, qs, ks, vs = _blocky_codes(oracle_mod, 1, Nq=Nq, Nk=Nk)
    o_ref, _, bound = fp8_bound(oracle_mod, q8, k8, vt8, qs, ks, vs, Nq, Nk)
    ks_bad = ks.copy()
    ks_bad[0, 0, 1] = ks[0, 0, 2]
    o_bad, _ = oracle_mod.attn_fp8_dense(q8, k8, vt8, qs, ks_bad, vs, Nq, Nk)
    err = np.abs(o_bad - o_ref)
    assert np.any(err > bound)
    vmax = np.abs(oracle_mod.e4m3_decode(vt8) * vs[:, :, None, None]).max()
    assert err.max() <= 2.0 ** -4 * vmax + 2e-2

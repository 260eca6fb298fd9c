"""GPU parity of the FP8 path (fa_quantize_fp8, fa_fwd_fp8) against the oracle.

Quantiser: codes and scales must equal the oracle's bit for bit (both divide
in float32 and round to the nearest e4m3 code, ties to even, saturating).

Forward: compared with the attention definition evaluated in fp64 on the
dequantised codes (the same codes and scales the kernel reads).  The one
rounding step not in that definition is P -> e4m3 before O += P V: each
weight is off by at most 2^-4 of itself (3 mantissa bits; below 2^-6 the
absolute error is at most 2^-10), and the row sum uses the unrounded weights,
so |dO| <= 2^-4 * max|v| + 2^-10 * sum|v| / l; with the bf16 output rounding
the bar is max|dO| <= 2^-4 * max|v| + 2e-2.  The LSE comes from fp32 scores
and sums: |dLSE| <= 1e-3 as for bf16.
"""
import numpy as np
import pytest
import torch

import attention_forward_fa2_gb300 as fa
from attention_forward_fa2_gb300 import build as fabuild
from attention_forward_fa2_gb300 import inputs as I
from fa_testutil import sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    fabuild.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(B, Nq, Nk, H, Hk, seed):
    g = torch.Generator().manual_seed(seed)
    return (I.randn_bf16((B, Nq, H, 128), g), I.randn_bf16((B, Nk, Hk, 128), g),
            I.randn_bf16((B, Nk, Hk, 128), g))


def _gpu_quant(q, k, v):
    t = fa.quantize_fp8(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    B, Nq, Nk, H, Hk, d = t.B, t.Nq, t.Nk, t.H, t.Hk, t.d
    n = fa.fp8_sizes(B, Nq, Nk, H, Hk, d)
    nkp = n[2] // (B * Hk * d)
    cpu = lambda x, m: x[:m].cpu().numpy()
    return t, (cpu(t.q8, n[0]).reshape(B, Nq, H, d), cpu(t.k8, n[1]).reshape(B, Nk, Hk, d),
               cpu(t.vt8, n[2]).reshape(B, Hk, d, nkp), cpu(t.q_scale, n[3]).reshape(B, H, -1),
               cpu(t.k_scale, n[4]).reshape(B, Hk, -1), cpu(t.v_scale, n[5]).reshape(B, Hk))


@pytest.mark.parametrize("B,Nq,Nk,H,Hk", [(1, 200, 130, 2, 1), (2, 257, 300, 3, 3), (1, 64, 4096, 1, 1)])
def test_quantiser_matches_oracle_bit_for_bit(oracle_mod, B, Nq, Nk, H, Hk):
    q, k, v = _inputs(B, Nq, Nk, H, Hk, 40 + Nq)
    q = q * 5  # a wider range: exercises saturation-free large codes and subnormals
    _, got = _gpu_quant(q, k, v)
    ref = oracle_mod.quantize_fp8(I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v))
    for name, a, b in zip(("q8", "k8", "vt8", "q_scale", "k_scale", "v_scale"), got, ref):
        assert a.shape == b.shape, name
        assert np.array_equal(a, b), name


def _check(o, lse, o_ref, lse_ref, vmax, what):
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    assert np.all(np.isfinite(o)), what
    err = np.abs(o - o_ref).max()
    bound = 2.0 ** -4 * vmax + 2e-2
    assert err <= bound, "%s: max|dO| %.4g > %.4g" % (what, err, bound)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), what
    el = np.abs(np.where(empty, 0, lse) - np.where(empty, 0, lse_ref)).max()
    assert el <= 1e-3, "%s: max|dLSE| %.3g" % (what, el)
    return err


@pytest.mark.parametrize("B,Nq,Nk,H,Hk,causal", [
    (1, 256, 256, 2, 2, False),
    (1, 256, 256, 2, 2, True),
    (2, 300, 517, 4, 2, False),
    (2, 300, 517, 4, 2, True),
    (1, 130, 70, 2, 1, True),      # more queries than keys: rows with no key
    (1, 64, 4096, 1, 1, False),    # the 64 x 4096 slice
])
def test_fp8_forward_matches_oracle(oracle_mod, B, Nq, Nk, H, Hk, causal):
    q, k, v = _inputs(B, Nq, Nk, H, Hk, 60 + Nq + Nk + causal)
    t, (q8, k8, vt8, qs, ks, vs) = _gpu_quant(q, k, v)
    o, lse = fa.forward_fp8(t, causal=causal)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    o_ref, lse_ref = oracle_mod.attn_fp8_dense(q8, k8, vt8, qs, ks, vs, Nq, Nk, causal=causal)
    vmax = np.abs(oracle_mod.e4m3_decode(vt8) * vs[:, :, None, None]).max()
    _check(o, lse, o_ref, lse_ref, vmax, "B%d Nq%d Nk%d H%d Hk%d causal%d" % (B, Nq, Nk, H, Hk, causal))


def test_fp8_forward_page_workload_sampled_heads(oracle_mod):
    """The page workload (B16 N4096 H16 d128) in one call, two heads checked in full."""
    w = I.PAGE
    q, k, v, _, _ = I.make(w)
    t, (q8, k8, vt8, qs, ks, vs) = _gpu_quant(q, k, v)
    o, lse = fa.forward_fp8(t)
    assert fa.check_status()[0] == fa.FA_OK
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        o_ref, lse_ref = oracle_mod.attn_fp8_dense(q8[b:b + 1, :, h:h + 1].copy(), k8[b:b + 1, :, h:h + 1].copy(),
                                                   vt8[b:b + 1, h:h + 1].copy(), qs[b:b + 1, h:h + 1].copy(),
                                                   ks[b:b + 1, h:h + 1].copy(), vs[b:b + 1, h:h + 1].copy(),
                                                   w.Nq, w.Nk)
        vmax = np.abs(oracle_mod.e4m3_decode(vt8[b, h]) * vs[b, h]).max()
        _check(o[b:b + 1, :, h:h + 1], lse[b:b + 1, h:h + 1], o_ref, lse_ref, vmax, "page b%d h%d" % (b, h))


def test_fp8_errors():
    with pytest.raises(fa.FaError) as e:
        fa.fp8_sizes(1, 64, 64, 1, 1, 64)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    q = torch.randn(1, 64, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError):
        fa.quantize_fp8(q, q, q)

"""GPU parity of the FP8 path (fa_quantize_fp8, fa_fwd_fp8) against the oracle.

Quantiser: codes and scales must equal the oracle's bit for bit (both divide
in float32 and round to the nearest e4m3 code, ties to even, saturating).

Forward: compared with the attention definition evaluated in fp64 on the
dequantised codes (the same codes and scales the kernel reads).  The one
rounding step not in that definition is P -> e4m3 before O += P V: each
weight is off by at most 2^-4 of itself (3 mantissa bits; below 2^-6 the
absolute error is at most 2^-10), and the row sum uses the unrounded weights,
so per element |dO_ic| <= 2^-4 sum_j P_ij |v_jc| + 2^-10 sum_j |v_jc| / l_i,
plus the bf16 output rounding and the fp32 sums (fa_testutil.fp8_bound; the
oracle supplies sum_j P_ij |v_jc| and the row maximum that gives l_i).  The
LSE comes from fp32 scores and sums: |dLSE| <= 1e-3 as for bf16.
"""
import numpy as np
import pytest
import torch

import attention_forward_fa2_gb300 as fa
from attention_forward_fa2_gb300 import build as fabuild
from attention_forward_fa2_gb300 import inputs as I
from fa_testutil import fp8_bound, sample_rows

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


def _regime_rows(kind, rows, heads, gen):
    """bf16 [rows, heads, 128] values of one quantisation regime."""
    shape = (rows, heads, 128)
    z = torch.randn(shape, generator=gen)
    if kind == "normal":
        x = z * 3
    elif kind == "tiny":        # scale below 2^-60: the quotients take the rescaled path
        x = z * 1e-36
    elif kind == "subnormal":   # bf16 subnormals only: a subnormal scale
        x = z * 1e-39
    elif kind == "spread":      # magnitudes 2^-140 .. 2^20 in one block, subnormals included
        e = torch.randint(-140, 21, shape, generator=gen).double()
        x = (torch.sign(z) * torch.exp2(e) * (1 + torch.rand(shape, generator=gen))).float()
    elif kind == "signed_zeros":  # +0 and -0 with a few ordinary values
        x = torch.where(torch.rand(shape, generator=gen) < 0.5, torch.tensor(0.0), torch.tensor(-0.0))
        x[::17, :, ::5] = z[::17, :, ::5]
    elif kind == "zeros":       # an all-zero block (scale 1), both signs
        x = torch.where(torch.rand(shape, generator=gen) < 0.5, torch.tensor(0.0), torch.tensor(-0.0))
    else:                       # "large"
        x = z * 1e30
    return x.to(torch.bfloat16)


def test_quantiser_edge_regimes_bit_for_bit(oracle_mod):
    """Blocks in every regime the quantiser's quotient distinguishes (ordinary values, scales
    below 2^-60 and subnormal ones, bf16 subnormals, magnitudes over 160 binades, signed zeros,
    all-zero blocks, huge values): codes and scales equal the oracle's bit for bit."""
    kinds = ("normal", "tiny", "subnormal", "spread", "signed_zeros", "zeros", "large")
    g = torch.Generator().manual_seed(606)
    H, Hk = 2, 2
    q = torch.cat([_regime_rows(k, 128, H, g) for k in kinds])[None]
    k = torch.cat([_regime_rows(k, 128, Hk, g) for k in reversed(kinds)])[None]
    v = torch.cat([_regime_rows(k, 128, Hk, g) for k in kinds[:3]])[None]
    v = torch.cat([v, torch.zeros_like(k[:, 384:])], dim=1)  # V maxima: a subnormal-scale head...
    v[:, :, 1] = k[:, :, 1]                                  # ...and one spanning every regime
    _, got = _gpu_quant(q, k, v)
    ref = oracle_mod.quantize_fp8(I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v))
    for name, a, b in zip(("q8", "k8", "vt8", "q_scale", "k_scale", "v_scale"), got, ref):
        assert a.shape == b.shape, name
        assert np.array_equal(a, b), (name, np.argwhere(a != b)[:5])


def _check(o, lse, o_ref, lse_ref, bound, what):
    """O within the per-element bar (fa_testutil.fp8_bound), LSE within 1e-3."""
    o = o.double().cpu().numpy() if torch.is_tensor(o) else o
    lse = lse.double().cpu().numpy() if torch.is_tensor(lse) else lse
    assert np.all(np.isfinite(o)), what
    diff = np.abs(o - o_ref)
    err = diff.max() if diff.size else 0.0
    worst = (diff / bound).max() if diff.size else 0.0
    assert worst <= 1.0, "%s: |dO| %.4g exceeds its bar (ratio %.3g)" % (what, err, worst)
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
    o_ref, lse_ref, bound = fp8_bound(oracle_mod, q8, k8, vt8, qs, ks, vs, Nq, Nk, causal=causal)
    _check(o, lse, o_ref, lse_ref, bound, "B%d Nq%d Nk%d H%d Hk%d causal%d" % (B, Nq, Nk, H, Hk, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_blocks_of_different_amplitude(oracle_mod, causal):
    """Key blocks whose amplitudes differ (so their scales differ by up to a
    third), queries likewise: a scale applied to the wrong block moves O past
    the per-element bar and the LSE past 1e-3."""
    B, Nq, Nk, H, Hk = 2, 384, 640, 4, 2
    q, k, v = _inputs(B, Nq, Nk, H, Hk, 90 + causal)
    amp_k = torch.tensor([1.0, 1.2, 0.9, 1.1, 0.8]).repeat_interleave(128)
    amp_q = torch.tensor([1.1, 0.9, 1.25]).repeat_interleave(128)
    k = (k.float() * amp_k[None, :, None, None]).to(torch.bfloat16)
    q = (q.float() * amp_q[None, :, None, None]).to(torch.bfloat16)
    t, (q8, k8, vt8, qs, ks, vs) = _gpu_quant(q, k, v)
    o, lse = fa.forward_fp8(t, causal=causal)
    assert fa.check_status()[0] == fa.FA_OK
    o_ref, lse_ref, bound = fp8_bound(oracle_mod, q8, k8, vt8, qs, ks, vs, Nq, Nk, causal=causal)
    _check(o, lse, o_ref, lse_ref, bound, "blocky causal%d" % causal)


def test_fp8_forward_page_workload_every_head(oracle_mod):
    """The page workload (B16 N4096 H16 d128) in one call; every element of
    every head against the oracle (one batch at a time to bound memory)."""
    w = I.PAGE
    q, k, v, _, _ = I.make(w)
    t, (q8, k8, vt8, qs, ks, vs) = _gpu_quant(q, k, v)
    o, lse = fa.forward_fp8(t)
    assert fa.check_status()[0] == fa.FA_OK
    o, lse = o.cpu(), lse.cpu()
    for b in range(w.B):
        sl = slice(b, b + 1)
        o_ref, lse_ref, bound = fp8_bound(oracle_mod, q8[sl], k8[sl], vt8[sl], qs[sl], ks[sl], vs[sl], w.Nq, w.Nk)
        _check(o[sl].double().numpy(), lse[sl].double().numpy(), o_ref, lse_ref, bound, "page b%d" % b)


def test_fp8_errors():
    with pytest.raises(fa.FaError) as e:
        fa.fp8_sizes(1, 64, 64, 1, 1, 64)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    q = torch.randn(1, 64, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError):
        fa.quantize_fp8(q, q, q)


# ------------------------------------------------------- packed sequences
def _col0(cu_b, b):
    """First V^T column of sequence b (the packed FP8 layout of include/fa.h)."""
    return (int(cu_b) + 15) // 16 * 16 + 16 * b


def _varlen_inputs(lens_q, lens_k, H, Hk, seed):
    g = torch.Generator().manual_seed(seed)
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    q = I.randn_bf16((int(cu_q[-1]), H, 128), g)
    k = I.randn_bf16((int(cu_k[-1]), Hk, 128), g)
    v = I.randn_bf16((int(cu_k[-1]), Hk, 128), g)
    return q, k, v, cu_q, cu_k


def _gpu_quant_varlen(q, k, v, cu_q, cu_k):
    t = fa.quantize_fp8_varlen(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cu_q).cuda(),
                               torch.from_numpy(cu_k).cuda(), int(np.diff(cu_q).max()), int(np.diff(cu_k).max()))
    torch.cuda.synchronize()
    n = fa.fp8_varlen_sizes(t.B, t.total_q, t.total_k, t.max_seqlen_q, t.max_seqlen_k, t.H, t.Hk, t.d)
    kp = n[2] // (t.Hk * t.d)
    cpu = lambda x, m: x[:m].cpu().numpy()
    return t, (cpu(t.q8, n[0]).reshape(t.total_q, t.H, t.d), cpu(t.k8, n[1]).reshape(t.total_k, t.Hk, t.d),
               cpu(t.vt8, n[2]).reshape(t.Hk, t.d, kp), cpu(t.q_scale, n[3]).reshape(t.B, t.H, -1),
               cpu(t.k_scale, n[4]).reshape(t.B, t.Hk, -1), cpu(t.v_scale, n[5]).reshape(t.B, t.Hk))


def _seq_codes(codes, cu_q, cu_k, b):
    """Codes and scales of sequence b in the dense layouts of quantize_fp8 (batch of one)."""
    q8, k8, vt8, qs, ks, vs = codes
    lq, lk = int(cu_q[b + 1] - cu_q[b]), int(cu_k[b + 1] - cu_k[b])
    c0 = _col0(cu_k[b], b)
    return (q8[cu_q[b]:cu_q[b + 1]][None], k8[cu_k[b]:cu_k[b + 1]][None],
            vt8[None, :, :, c0:c0 + (lk + 15) // 16 * 16], qs[b:b + 1, :, :(lq + 127) // 128],
            ks[b:b + 1, :, :(lk + 127) // 128], vs[b:b + 1]), lq, lk


LENS_Q = [1, 127, 128, 129, 300, 0, 513, 64, 17]
LENS_K = [3, 130, 128, 1, 300, 40, 257, 0, 700]


def test_varlen_quantiser_matches_oracle_per_sequence(oracle_mod):
    """Packed codes and scales equal the oracle's quantisation of each sequence on its own."""
    H, Hk = 4, 2
    q, k, v, cu_q, cu_k = _varlen_inputs(LENS_Q, LENS_K, H, Hk, 501)
    q = q * 3
    t, codes = _gpu_quant_varlen(q, k, v, cu_q, cu_k)
    vt8, qs, ks = codes[2], codes[3], codes[4]
    bits = I.bf16_bits
    for b in range(len(LENS_Q)):
        got, lq, lk = _seq_codes(codes, cu_q, cu_k, b)
        ref = oracle_mod.quantize_fp8(bits(q[cu_q[b]:cu_q[b + 1]][None]), bits(k[cu_k[b]:cu_k[b + 1]][None]),
                                      bits(v[cu_k[b]:cu_k[b + 1]][None]))
        for name, a, r in zip(("q8", "k8", "vt8", "q_scale", "k_scale", "v_scale"), got, ref):
            assert a.shape == r.shape, (b, name)
            assert np.array_equal(a, r), (b, name)
        # Blocks past the sequence have scale 1; V^T columns after its keys are zero.
        assert np.all(qs[b, :, (lq + 127) // 128:] == 1.0) and np.all(ks[b, :, (lk + 127) // 128:] == 1.0)
        c0, c1 = _col0(cu_k[b], b), _col0(cu_k[b + 1], b + 1)
        assert np.all(vt8[:, :, c0 + (lk + 15) // 16 * 16:c1] == 0), b
    assert vt8.shape[2] == _col0(cu_k[-1], len(LENS_Q))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_varlen_forward_matches_oracle(oracle_mod, causal):
    H, Hk = 4, 2
    q, k, v, cu_q, cu_k = _varlen_inputs(LENS_Q, LENS_K, H, Hk, 502 + causal)
    t, codes = _gpu_quant_varlen(q, k, v, cu_q, cu_k)
    lse0 = torch.full((t.B, H, t.max_seqlen_q), 123.0, device="cuda")
    o, lse = fa.forward_fp8_varlen(t, causal=causal, lse=lse0)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    for b in range(len(LENS_Q)):
        (q8, k8, vt8, qs, ks, vs), lq, lk = _seq_codes(codes, cu_q, cu_k, b)
        assert np.all(lse[b, :, lq:] == 123.0), b  # entries past the length untouched
        if lq == 0:
            continue
        if lk == 0:
            assert np.all(o[cu_q[b]:cu_q[b + 1]] == 0.0) and np.all(np.isneginf(lse[b, :, :lq])), b
            continue
        o_ref, lse_ref, bound = fp8_bound(oracle_mod, q8, k8, vt8, qs, ks, vs, lq, lk, causal=causal)
        _check(o[cu_q[b]:cu_q[b + 1]][None], lse[b:b + 1, :, :lq],
               o_ref, lse_ref, bound, "seq %d (lq %d, lk %d, causal %d)" % (b, lq, lk, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_varlen_equal_lengths_bitwise_equal_to_dense(causal):
    """Sequences of one length run the same tiles as the dense form: identical codes and outputs."""
    B, L, H, Hk = 3, 300, 4, 2
    q, k, v, cu_q, cu_k = _varlen_inputs([L] * B, [L] * B, H, Hk, 503)
    t, codes = _gpu_quant_varlen(q, k, v, cu_q, cu_k)
    td, dense = _gpu_quant(q.reshape(B, L, H, 128), k.reshape(B, L, Hk, 128), v.reshape(B, L, Hk, 128))
    assert np.array_equal(codes[0].reshape(B, L, H, 128), dense[0])
    assert np.array_equal(codes[1].reshape(B, L, Hk, 128), dense[1])
    for x, y in zip(codes[3:], dense[3:]):
        assert np.array_equal(x, y)
    for b in range(B):
        c0 = _col0(cu_k[b], b)
        assert np.array_equal(codes[2][:, :, c0:c0 + 304], dense[2][b])
    o, lse = fa.forward_fp8_varlen(t, causal=causal)
    od, lsed = fa.forward_fp8(td, causal=causal)
    assert fa.check_status()[0] == fa.FA_OK
    assert torch.equal(o.view(torch.int16).reshape(B, L, H, 128), od.view(torch.int16))
    assert torch.equal(lse, lsed)


def test_fp8_varlen_workload_every_element(oracle_mod):
    """The variable-length workload (32 sequences of 128..4096 tokens, H16 d128) in one call;
    every head of every sequence checked in full against the oracle."""
    w = I.VARLEN
    q, k, v, cu_q, cu_k = I.make(w)
    cu_q, cu_k = cu_q.numpy(), cu_k.numpy()
    t, codes = _gpu_quant_varlen(q, k, v, cu_q, cu_k)
    o, lse = fa.forward_fp8_varlen(t)
    assert fa.check_status()[0] == fa.FA_OK
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    for b in range(w.B):
        (q8, k8, vt8, qs, ks, vs), lq, lk = _seq_codes(codes, cu_q, cu_k, b)
        o_ref, lse_ref, bound = fp8_bound(oracle_mod, q8, k8, vt8, qs, ks, vs, lq, lk)
        _check(o[cu_q[b]:cu_q[b + 1]][None], lse[b:b + 1, :, :lq], o_ref, lse_ref, bound,
               "varlen seq %d (len %d)" % (b, lq))


def test_fp8_varlen_bad_seqlens_are_reported():
    """A sequence longer than the stated maximum, or past the packed rows, is reported; nothing faults."""
    H = 2
    q, k, v, cu_q, cu_k = _varlen_inputs([100, 200], [100, 200], H, H, 504)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    # Second sequence: 200 rows > maximum 150; then 220 rows ending at row 320 of 300.
    for max_q, cq in ((150, cu_q), (250, np.array([0, 100, 320], np.int32))):
        cqt = torch.from_numpy(cq).cuda()
        t = fa.quantize_fp8_varlen(dq, dk, dv, cqt, torch.from_numpy(cu_k).cuda(), max_q, 200)
        fa.forward_fp8_varlen(t)
        rc, _ = fa.check_status()
        assert rc == fa.FA_ERR_BAD_SEQLENS, (max_q, cq)
    assert fa.check_status()[0] == fa.FA_OK

"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a brute-force
evaluation of the plain (non-max-shifted) softmax definition on tiny inputs,
torch's float64 softmax, closed forms, and invariants.  They are chosen so that
a dropped term, a wrong sign or index, or a transposed operand in attn_ref.c
fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from attention_forward_fa2_gb300 import inputs as I


def _f(bits):
    """bf16 bit patterns -> exact float64 values."""
    return I.bits_to_bf16(bits).to(torch.float64).numpy()


def _bits_from_values(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16)
    back = t.to(torch.float64).numpy()
    assert np.array_equal(back, np.asarray(x, dtype=np.float64)), "values must be bf16-exact"
    return I.bf16_bits(t)


def _rand_dense(B, Nq, Nk, H, d, seed):
    q, k, v = I.make_dense(B, Nq, Nk, H, d, seed)
    return I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v)


# ---------------------------------------------------------------- brute force
def _brute_plain(qf, kf, vf, scale):
    """o = sum_j e^{s_j} v_j / sum_j e^{s_j}, lse = log sum_j e^{s_j}: the plain
    softmax definition WITHOUT the max shift, exact sums via math.fsum.
    Valid for small scores only (no overflow)."""
    B, Nq, H, d = qf.shape
    Nk = kf.shape[1]
    o = np.zeros((B, Nq, H, d))
    lse = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                e = []
                for j in range(Nk):
                    s = scale * math.fsum(qf[b, i, h, c] * kf[b, j, h, c] for c in range(d))
                    e.append(math.exp(s))
                den = math.fsum(e)
                lse[b, h, i] = math.log(den)
                for c in range(d):
                    o[b, i, h, c] = math.fsum(e[j] * vf[b, j, h, c] for j in range(Nk)) / den
    return o, lse


@pytest.mark.parametrize("B,Nq,Nk,H,d,seed", [(2, 3, 5, 3, 4, 11), (1, 4, 1, 2, 3, 12),
                                              (3, 1, 4, 1, 2, 13), (1, 2, 7, 2, 8, 14)])
def test_brute_force_tiny(oracle_mod, B, Nq, Nk, H, d, seed):
    qb, kb, vb = _rand_dense(B, Nq, Nk, H, d, seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attn_dense(qb, kb, vb)
    o_bf, lse_bf = _brute_plain(_f(qb), _f(kb), _f(vb), scale)
    np.testing.assert_allclose(o, o_bf, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_bf, rtol=0, atol=1e-13)


def test_brute_force_explicit_scale(oracle_mod):
    qb, kb, vb = _rand_dense(2, 3, 4, 2, 5, 21)
    o, lse = oracle_mod.attn_dense(qb, kb, vb, scale=0.37)
    o_bf, lse_bf = _brute_plain(_f(qb), _f(kb), _f(vb), 0.37)
    np.testing.assert_allclose(o, o_bf, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_bf, rtol=0, atol=1e-13)


# ------------------------------------------------------------- library check
@pytest.mark.parametrize("B,Nq,Nk,H,d", [(2, 37, 45, 3, 16), (1, 130, 129, 2, 64),
                                         (1, 64, 300, 1, 128)])
def test_torch_float64_softmax(oracle_mod, B, Nq, Nk, H, d):
    qb, kb, vb = _rand_dense(B, Nq, Nk, H, d, 31 + d)
    o, lse = oracle_mod.attn_dense(qb, kb, vb)
    qt = torch.from_numpy(_f(qb)).permute(0, 2, 1, 3)  # [B, H, N, d]
    kt = torch.from_numpy(_f(kb)).permute(0, 2, 1, 3)
    vt = torch.from_numpy(_f(vb)).permute(0, 2, 1, 3)
    s = (qt @ kt.transpose(-1, -2)) * (1.0 / math.sqrt(d))
    ref_o = (torch.softmax(s, dim=-1) @ vt).permute(0, 2, 1, 3).numpy()
    ref_lse = torch.logsumexp(s, dim=-1).numpy()
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


# --------------------------------------------------------------- closed forms
def test_zero_query_gives_mean_of_values(oracle_mod):
    B, Nq, Nk, H, d = 2, 5, 9, 3, 16
    _, kb, vb = _rand_dense(B, Nq, Nk, H, d, 41)
    qb = np.zeros((B, Nq, H, d), np.uint16)  # +0.0 in bf16
    o, lse = oracle_mod.attn_dense(qb, kb, vb)
    vf = _f(vb)
    mean = vf.mean(axis=1)  # [B, H, d]
    for i in range(Nq):
        np.testing.assert_allclose(o[:, i], mean, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.full_like(lse, math.log(Nk)), rtol=0, atol=1e-14)


def test_one_key(oracle_mod):
    B, Nq, H, d = 2, 4, 3, 8
    qb, kb, vb = _rand_dense(B, Nq, 1, H, d, 42)
    o, lse = oracle_mod.attn_dense(qb, kb, vb)
    qf, kf, vf = _f(qb), _f(kb), _f(vb)
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                np.testing.assert_array_equal(o[b, i, h], vf[b, 0, h])
                s = math.fsum(qf[b, i, h] * kf[b, 0, h]) / math.sqrt(d)
                assert abs(lse[b, h, i] - s) < 1e-13


def test_two_keys_logistic(oracle_mod):
    # s1, s2 chosen by hand; P = (sigmoid(s1 - s2), sigmoid(s2 - s1)).
    d = 2
    q = _bits_from_values(np.array([1.0, 0.5]).reshape(1, 1, 1, d))
    k = _bits_from_values(np.array([[2.0, 0.0], [0.0, -4.0]]).reshape(1, 2, 1, d))
    v = _bits_from_values(np.array([[1.0, 0.0], [0.0, 1.0]]).reshape(1, 2, 1, d))
    scale = 0.75
    o, lse = oracle_mod.attn_dense(q, k, v, scale=scale)
    s1, s2 = scale * 2.0, scale * (-2.0)
    p1 = 1.0 / (1.0 + math.exp(s2 - s1))
    assert abs(o[0, 0, 0, 0] - p1) < 1e-15
    assert abs(o[0, 0, 0, 1] - (1.0 - p1)) < 1e-15
    assert abs(lse[0, 0, 0] - (s1 + math.log1p(math.exp(s2 - s1)))) < 1e-15


def test_identical_value_rows(oracle_mod):
    B, Nq, Nk, H, d = 1, 6, 33, 2, 16
    qb, kb, _ = _rand_dense(B, Nq, Nk, H, d, 43)
    row = np.linspace(-3, 3, d)
    vals = np.broadcast_to(row, (B, Nk, H, d)).copy()
    vals = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    vb = _bits_from_values(vals)
    o, _ = oracle_mod.attn_dense(qb, kb, vb)
    np.testing.assert_allclose(o, np.broadcast_to(vals[:, :1], o.shape), rtol=0, atol=1e-14)


def test_rows_sum_to_one(oracle_mod):
    """V = 1 everywhere gives O = sum_j P_ij = 1."""
    B, Nq, Nk, H, d = 2, 7, 50, 2, 4
    qb, kb, _ = _rand_dense(B, Nq, Nk, H, d, 44)
    vb = _bits_from_values(np.ones((B, Nk, H, d)))
    o, _ = oracle_mod.attn_dense(qb, kb, vb)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


# ----------------------------------------------------------------- invariants
def test_key_shift_invariance(oracle_mod):
    """K -> K + 1 c^T shifts every score of row i by scale * q_i . c: O is
    unchanged and LSE_i moves by exactly that amount."""
    rng = np.random.default_rng(5)
    B, Nq, Nk, H, d = 2, 5, 11, 2, 8
    qv = rng.integers(-4, 5, size=(B, Nq, H, d)) / 4.0
    kv = rng.integers(-4, 5, size=(B, Nk, H, d)) / 4.0
    vv = rng.integers(-8, 9, size=(B, Nk, H, d)) / 8.0
    c = rng.integers(-2, 3, size=(d,)) / 4.0
    qb, kb, vb = _bits_from_values(qv), _bits_from_values(kv), _bits_from_values(vv)
    kb2 = _bits_from_values(kv + c)
    o1, l1 = oracle_mod.attn_dense(qb, kb, vb)
    o2, l2 = oracle_mod.attn_dense(qb, kb2, vb)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    shift = np.einsum("bihc,c->bhi", qv, c) / math.sqrt(d)
    np.testing.assert_allclose(l2 - l1, shift, rtol=0, atol=1e-13)


def test_joint_permutation_invariance(oracle_mod):
    B, Nq, Nk, H, d = 2, 4, 23, 3, 16
    qb, kb, vb = _rand_dense(B, Nq, Nk, H, d, 45)
    perm = np.random.default_rng(6).permutation(Nk)
    o1, l1 = oracle_mod.attn_dense(qb, kb, vb)
    o2, l2 = oracle_mod.attn_dense(qb, kb[:, perm].copy(), vb[:, perm].copy())
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)


def test_value_linearity(oracle_mod):
    """O(2 V + 1) = 2 O(V) + 1 and LSE does not depend on V."""
    rng = np.random.default_rng(7)
    B, Nq, Nk, H, d = 1, 6, 19, 2, 8
    qb, kb, _ = _rand_dense(B, Nq, Nk, H, d, 46)
    vv = rng.integers(-16, 17, size=(B, Nk, H, d)) / 16.0
    o1, l1 = oracle_mod.attn_dense(qb, kb, _bits_from_values(vv))
    o2, l2 = oracle_mod.attn_dense(qb, kb, _bits_from_values(2.0 * vv + 1.0))
    np.testing.assert_allclose(o2, 2.0 * o1 + 1.0, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(l2, l1)


def test_heads_and_batches_are_independent(oracle_mod):
    """Changing the inputs of one (b, h) slice changes only that slice."""
    B, Nq, Nk, H, d = 3, 5, 6, 4, 8
    qb, kb, vb = _rand_dense(B, Nq, Nk, H, d, 47)
    o1, l1 = oracle_mod.attn_dense(qb, kb, vb)
    q2, k2, v2 = qb.copy(), kb.copy(), vb.copy()
    q3, k3, v3 = _rand_dense(B, Nq, Nk, H, d, 48)
    q2[1, :, 2] = q3[1, :, 2]
    k2[1, :, 2] = k3[1, :, 2]
    v2[1, :, 2] = v3[1, :, 2]
    o2, l2 = oracle_mod.attn_dense(q2, k2, v2)
    mask = np.ones((B, H), bool)
    mask[1, 2] = False
    for b in range(B):
        for h in range(H):
            same = np.array_equal(o1[b, :, h], o2[b, :, h]) and np.array_equal(l1[b, h], l2[b, h])
            assert same == mask[b, h], (b, h)


def test_large_scores_do_not_overflow(oracle_mod):
    """Scores near +-2000: exp without the max shift would overflow; safe
    softmax ("GPU 内核与 FlashAttention" §11.1) must return the dominant key's V."""
    d = 16
    q = _bits_from_values(np.full((1, 2, 1, d), 8.0))
    kv = np.zeros((1, 3, 1, d))
    kv[0, 0, 0, :] = 4.0    # s = 8*4*16*scale
    kv[0, 1, 0, :] = 3.0
    kv[0, 2, 0, :] = -4.0
    vv = np.zeros((1, 3, 1, d))
    vv[0, 0, 0, :] = 1.5
    vv[0, 1, 0, :] = -2.0
    scale = 4.0
    o, lse = oracle_mod.attn_dense(q, _bits_from_values(kv), _bits_from_values(vv), scale=scale)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    s0 = scale * 8.0 * 4.0 * d
    np.testing.assert_allclose(o[0, :, 0, :], 1.5, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], s0, rtol=1e-15)


# ----------------------------------------------- blockwise recurrence is exact
@pytest.mark.parametrize("block", [1, 7, 64, 128, 1000])
def test_online_recurrence_equals_full(oracle_mod, block):
    """"GPU 内核与 FlashAttention" §11.3: after the last block the recurrence
    gives the exact result, not an approximation."""
    qb, kb, vb = _rand_dense(2, 9, 300, 2, 32, 50)
    o, lse = oracle_mod.attn_dense(qb, kb, vb)
    o2, lse2 = oracle_mod.attn_online(qb, kb, vb, block)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)


def test_two_block_merge_is_associative():
    """§11.2: (m, l) pairs merge by m = max(m1, m2), l = l1 e^{m1-m} + l2 e^{m2-m};
    merging three blocks in either grouping gives the same pair as one pass."""
    x = np.random.default_rng(8).normal(size=30) * 5

    def ml(seg):
        m = max(seg)
        return m, math.fsum(math.exp(t - m) for t in seg)

    def merge(a, b):
        m = max(a[0], b[0])
        return m, a[1] * math.exp(a[0] - m) + b[1] * math.exp(b[0] - m)

    a, b, c = ml(x[:7]), ml(x[7:19]), ml(x[19:])
    full = ml(x)
    for m, l in (merge(merge(a, b), c), merge(a, merge(b, c))):
        assert m == full[0]
        assert abs(l - full[1]) < 1e-12 * full[1]


# --------------------------------------------------------- rows and varlen
def test_rows_match_dense(oracle_mod):
    B, Nq, Nk, H, d = 2, 40, 70, 3, 16
    qb, kb, vb = _rand_dense(B, Nq, Nk, H, d, 51)
    o, lse = oracle_mod.attn_dense(qb, kb, vb)
    rows = np.array([[0, 0, 0], [1, 2, 39], [1, 0, 17], [0, 1, 5]])
    orow, lrow = oracle_mod.attn_dense_rows(qb, kb, vb, rows)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(orow[r], o[b, i, h])
        assert lrow[r] == lse[b, h, i]


def test_varlen_against_brute_force(oracle_mod):
    lens_q = [3, 1, 0, 4]
    lens_k = [2, 5, 3, 1]
    H, d = 2, 4
    q, k, v, cu_q, cu_k = I.make_varlen(lens_q, H, d, 52, lengths_k=lens_k)
    qb, kb, vb = I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v)
    maxq = max(lens_q)
    o, lse = oracle_mod.attn_varlen(qb, kb, vb, cu_q.numpy(), cu_k.numpy(), maxq)
    qf, kf, vf = _f(qb), _f(kb), _f(vb)
    scale = 1.0 / math.sqrt(d)
    cq, ck = cu_q.numpy(), cu_k.numpy()
    for b in range(len(lens_q)):
        qs = qf[cq[b]:cq[b + 1]][None]
        ks = kf[ck[b]:ck[b + 1]][None]
        vs = vf[ck[b]:ck[b + 1]][None]
        ob, lb = _brute_plain(qs, ks, vs, scale)
        np.testing.assert_allclose(o[cq[b]:cq[b + 1]], ob[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b, :, :lens_q[b]], lb[0], rtol=0, atol=1e-13)
        assert np.all(np.isnan(lse[b, :, lens_q[b]:]))  # untouched beyond the length


def test_varlen_empty_keys_convention(oracle_mod):
    """A query sequence with no keys: o = 0 and LSE = -inf (log of an empty sum)."""
    q, k, v, cu_q, cu_k = I.make_varlen([2, 3], 1, 4, 53, lengths_k=[0, 2])
    o, lse = oracle_mod.attn_varlen(I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v),
                                    cu_q.numpy(), cu_k.numpy(), 3)
    assert np.all(o[:2] == 0.0)
    assert np.all(np.isneginf(lse[0, :, :2]))
    assert np.all(np.isfinite(o[2:]))


# ------------------------------------------------------- causal and GQA
def _brute_causal(qf, kf, vf, scale, Hk):
    """Plain softmax over the visible keys j <= i + (Nk - Nq) (no max shift,
    math.fsum); rows that see no key give o = 0, lse = -inf."""
    B, Nq, H, d = qf.shape
    Nk = kf.shape[1]
    G = H // Hk
    o = np.zeros((B, Nq, H, d))
    lse = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                vis = [j for j in range(Nk) if j <= i + Nk - Nq]
                if not vis:
                    lse[b, h, i] = -math.inf
                    continue
                e = [math.exp(scale * math.fsum(qf[b, i, h, c] * kf[b, j, h // G, c] for c in range(d)))
                     for j in vis]
                den = math.fsum(e)
                lse[b, h, i] = math.log(den)
                for c in range(d):
                    o[b, i, h, c] = math.fsum(e[n] * vf[b, j, h // G, c] for n, j in enumerate(vis)) / den
    return o, lse


@pytest.mark.parametrize("B,Nq,Nk,H,Hk,d", [(1, 5, 5, 2, 2, 4), (2, 3, 7, 4, 2, 3),
                                             (1, 6, 4, 3, 1, 4), (1, 4, 4, 4, 1, 2)])
def test_causal_and_grouped_heads_brute_force(oracle_mod, B, Nq, Nk, H, Hk, d):
    g = torch.Generator().manual_seed(60 + Nq + Nk + Hk)
    q = I.randn_bf16((B, Nq, H, d), g)
    k = I.randn_bf16((B, Nk, Hk, d), g)
    v = I.randn_bf16((B, Nk, Hk, d), g)
    qb, kb, vb = I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attn_dense(qb, kb, vb, causal=True)
    o_bf, lse_bf = _brute_causal(_f(qb), _f(kb), _f(vb), scale, Hk)
    np.testing.assert_allclose(o, o_bf, rtol=0, atol=1e-13)
    fin = np.isfinite(lse_bf)
    np.testing.assert_allclose(lse[fin], lse_bf[fin], rtol=0, atol=1e-13)
    assert np.all(np.isneginf(lse[~fin]))
    if Hk == H:
        o_nc, _ = oracle_mod.attn_dense(qb, kb, vb, causal=False)
        o_bf_nc, _ = _brute_plain(_f(qb), _f(kb), _f(vb), scale)
        np.testing.assert_allclose(o_nc, o_bf_nc, rtol=0, atol=1e-13)


def test_causal_row_is_prefix_attention(oracle_mod):
    """With equal lengths, causal row i is plain attention of q_i over the first
    i + 1 keys ("GPU 内核与 FlashAttention" §14.4): compare with the unmasked
    definition evaluated on the truncated key set."""
    B, N, H, d = 1, 40, 2, 16
    qb, kb, vb = _rand_dense(B, N, N, H, d, 61)
    o, lse = oracle_mod.attn_dense(qb, kb, vb, causal=True)
    for i in (0, 1, 17, 39):
        op, lp = oracle_mod.attn_dense(qb[:, i:i + 1].copy(), kb[:, :i + 1].copy(), vb[:, :i + 1].copy())
        np.testing.assert_allclose(o[:, i], op[:, 0], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[:, :, i], lp[:, :, 0], rtol=0, atol=1e-14)


def test_causal_first_row_sees_one_key(oracle_mod):
    B, N, H, d = 2, 9, 3, 8
    qb, kb, vb = _rand_dense(B, N, N, H, d, 62)
    o, lse = oracle_mod.attn_dense(qb, kb, vb, causal=True)
    np.testing.assert_array_equal(o[:, 0], _f(vb)[:, 0])
    s0 = np.einsum("bhc,bhc->bh", _f(qb)[:, 0], _f(kb)[:, 0]) / math.sqrt(d)
    np.testing.assert_allclose(lse[:, :, 0], s0, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads_equal_repeated_heads(oracle_mod, causal):
    """Query head h reads key/value head h / G: identical to plain multi-head
    attention on K, V with every head repeated G times."""
    B, Nq, Nk, H, Hk, d = 2, 33, 47, 6, 2, 16
    g = torch.Generator().manual_seed(63)
    q = I.bf16_bits(I.randn_bf16((B, Nq, H, d), g))
    k = I.bf16_bits(I.randn_bf16((B, Nk, Hk, d), g))
    v = I.bf16_bits(I.randn_bf16((B, Nk, Hk, d), g))
    o, lse = oracle_mod.attn_dense(q, k, v, causal=causal)
    G = H // Hk
    o2, lse2 = oracle_mod.attn_dense(q, np.repeat(k, G, axis=2), np.repeat(v, G, axis=2), causal=causal)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_causal_rows_and_varlen_match_dense(oracle_mod):
    B, Nq, Nk, H, Hk, d = 2, 30, 45, 4, 2, 8
    g = torch.Generator().manual_seed(64)
    q = I.bf16_bits(I.randn_bf16((B, Nq, H, d), g))
    k = I.bf16_bits(I.randn_bf16((B, Nk, Hk, d), g))
    v = I.bf16_bits(I.randn_bf16((B, Nk, Hk, d), g))
    o, lse = oracle_mod.attn_dense(q, k, v, causal=True)
    rows = np.array([[0, 0, 0], [1, 3, 29], [0, 2, 11], [1, 1, 7]])
    orow, lrow = oracle_mod.attn_dense_rows(q, k, v, rows, causal=True)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(orow[r], o[b, i, h])
        assert lrow[r] == lse[b, h, i]
    # the same batch as a packed variable-length batch of two equal sequences
    cu_q = np.array([0, Nq, 2 * Nq], np.int32)
    cu_k = np.array([0, Nk, 2 * Nk], np.int32)
    ov, lv = oracle_mod.attn_varlen(q.reshape(B * Nq, H, d), k.reshape(B * Nk, Hk, d),
                                    v.reshape(B * Nk, Hk, d), cu_q, cu_k, Nq, causal=True)
    np.testing.assert_array_equal(ov.reshape(o.shape), o)
    np.testing.assert_array_equal(lv, lse)

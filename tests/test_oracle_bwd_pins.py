"""Pins for the fp64 oracle's backward pass ("GPU 内核与 FlashAttention" §13.1).

The backward formulas are checked against things other than themselves: the
numerical derivative of the forward definition (central differences), torch's
float64 autograd through an explicit softmax, the identity D_i = do_i . o_i
that §13.1 derives (the oracle computes D from its definition sum_j P_ij dP_ij),
closed forms (one key, Q = 0), and invariants (the key gradients of a head sum
to zero because every softmax row's Jacobian annihilates constants; grouped
heads equal repeated heads).  A dropped D, a missing scale, a transposed dS or
a wrong head mapping fails at least one of them.
"""
import numpy as np
import pytest
import torch

from attention_forward_fa2_gb300 import inputs as I


def _f(bits):
    return I.bits_to_bf16(bits).to(torch.float64).numpy()


def _rand(B, Nq, Nk, H, Hk, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = I.randn_bf16((B, Nq, H, d), g)
    k = I.randn_bf16((B, Nk, Hk, d), g)
    v = I.randn_bf16((B, Nk, Hk, d), g)
    do = I.randn_bf16((B, Nq, H, d), g)
    return tuple(I.bf16_bits(t) for t in (q, k, v, do))


def _torch_forward(q, k, v, scale, causal):
    """o = softmax(scale q k^T) v in float64, [B, N, H, d] layout, grouped heads
    by repeating K/V; the causal mask is bottom-right aligned."""
    B, Nq, H, d = q.shape
    Nk, Hk = k.shape[1], k.shape[2]
    G = H // Hk
    kr = k.repeat_interleave(G, dim=2)
    vr = v.repeat_interleave(G, dim=2)
    s = torch.einsum("bihc,bjhc->bhij", q, kr) * scale
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        s = s.masked_fill(j > i + (Nk - Nq), float("-inf"))
    p = torch.softmax(s, dim=-1)
    p = torch.nan_to_num(p, nan=0.0)  # rows that see no key
    return torch.einsum("bhij,bjhc->bihc", p, vr)


@pytest.mark.parametrize("B,Nq,Nk,H,Hk,d,causal", [
    (1, 5, 7, 2, 2, 4, False),
    (2, 9, 6, 4, 2, 8, True),
    (1, 6, 9, 3, 1, 5, True),
    (1, 11, 11, 2, 1, 16, False),
])
def test_against_torch_autograd(oracle_mod, B, Nq, Nk, H, Hk, d, causal):
    q, k, v, do = _rand(B, Nq, Nk, H, Hk, d, 3 + Nq + 7 * Hk + causal)
    scale = 0.3
    dq, dk, dv, _ = oracle_mod.attn_bwd_dense(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.tensor(_f(x), requires_grad=True) for x in (q, k, v))
    o = _torch_forward(tq, tk, tv, scale, causal)
    o.backward(torch.tensor(_f(do)))
    assert np.allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_central_differences(oracle_mod):
    """d phi / d x for phi = sum(dO * O(q, k, v)), one coordinate at a time."""
    B, Nq, Nk, H, Hk, d = 1, 4, 6, 2, 1, 3
    q, k, v, do = _rand(B, Nq, Nk, H, Hk, d, 21)
    scale = 0.7
    dq, dk, dv, _ = oracle_mod.attn_bwd_dense(q, k, v, do, scale, True)
    base = [torch.tensor(_f(x)) for x in (q, k, v)]
    dof = torch.tensor(_f(do))

    def phi(xs):
        return float((_torch_forward(*xs, scale, True) * dof).sum())

    rng = np.random.default_rng(5)
    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in base[which].shape)
            xs_p = [t.clone() for t in base]
            xs_m = [t.clone() for t in base]
            xs_p[which][idx] += eps
            xs_m[which][idx] -= eps
            num = (phi(xs_p) - phi(xs_m)) / (2 * eps)
            assert abs(num - grad[idx]) < 1e-7, (which, idx, num, grad[idx])


def test_delta_equals_do_dot_o(oracle_mod):
    """§13.1: D_i = sum_j P_ij dP_ij simplifies to do_i . o_i."""
    q, k, v, do = _rand(2, 13, 17, 4, 2, 16, 8)
    _, _, _, delta = oracle_mod.attn_bwd_dense(q, k, v, do, None, True)
    o, _ = oracle_mod.attn_dense(q, k, v, causal=True)
    ref = np.einsum("bihc,bihc->bhi", _f(do), o)
    assert np.allclose(delta, ref, rtol=1e-12, atol=1e-13)


def test_key_gradients_sum_to_zero(oracle_mod):
    """Every softmax row's Jacobian maps constants to zero, so sum_j dS_ij = 0
    and therefore sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0."""
    q, k, v, do = _rand(2, 10, 12, 4, 2, 8, 9)
    for causal in (False, True):
        _, dk, _, _ = oracle_mod.attn_bwd_dense(q, k, v, do, None, causal)
        assert np.abs(dk.sum(axis=1)).max() < 1e-12


def test_one_key(oracle_mod):
    """One key: P = 1, so dS = 0 (dQ = dK = 0) and dV = sum_i do_i."""
    q, k, v, do = _rand(1, 6, 1, 2, 2, 4, 10)
    dq, dk, dv, _ = oracle_mod.attn_bwd_dense(q, k, v, do)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    assert np.allclose(dv[:, 0], _f(do).sum(axis=1), rtol=1e-14, atol=1e-14)


def test_zero_queries_closed_form(oracle_mod):
    """Q = 0: uniform P = 1/Nk.  dV_j = (1/Nk) sum_i do_i, dK = 0 and
    dQ_i = (scale/Nk) sum_j (do_i . (v_j - vbar)) k_j."""
    B, Nq, Nk, H, d = 1, 5, 8, 2, 4
    _, k, v, do = _rand(B, Nq, Nk, H, H, d, 11)
    q = np.zeros((B, Nq, H, d), np.uint16)
    scale = 0.5
    dq, dk, dv, _ = oracle_mod.attn_bwd_dense(q, k, v, do, scale)
    kf, vf, dof = _f(k), _f(v), _f(do)
    assert np.allclose(dv, np.broadcast_to(dof.sum(axis=1, keepdims=True) / Nk, dv.shape), atol=1e-14)
    assert np.abs(dk).max() < 1e-15
    vbar = vf.mean(axis=1, keepdims=True)
    ref = scale / Nk * np.einsum("bihc,bjhc,bjhe->bihe", dof, vf - vbar, kf)
    assert np.allclose(dq, ref, rtol=1e-12, atol=1e-13)


def test_causal_first_row_has_no_query_gradient(oracle_mod):
    """Causal, Nq = Nk: row 0 sees key 0 only, P_0 = e_0, dS_0 = 0 -> dQ_0 = 0."""
    q, k, v, do = _rand(1, 7, 7, 2, 2, 4, 12)
    dq, _, _, _ = oracle_mod.attn_bwd_dense(q, k, v, do, None, True)
    assert np.abs(dq[:, 0]).max() < 1e-15
    assert np.abs(dq[:, 1:]).max() > 1e-3


def test_grouped_heads_equal_repeated_heads(oracle_mod):
    """GQA: the gradient of a shared K/V head is the sum of the gradients of
    the query heads reading it, as if K/V were repeated per head."""
    B, Nq, Nk, H, Hk, d = 1, 9, 10, 6, 2, 8
    q, k, v, do = _rand(B, Nq, Nk, H, Hk, d, 13)
    G = H // Hk
    for causal in (False, True):
        dq, dk, dv, _ = oracle_mod.attn_bwd_dense(q, k, v, do, None, causal)
        kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
        dq2, dk2, dv2, _ = oracle_mod.attn_bwd_dense(q, kr, vr, do, None, causal)
        assert np.allclose(dq, dq2, rtol=1e-13, atol=1e-14)
        assert np.allclose(dk, dk2.reshape(B, Nk, Hk, G, d).sum(axis=3), rtol=1e-12, atol=1e-13)
        assert np.allclose(dv, dv2.reshape(B, Nk, Hk, G, d).sum(axis=3), rtol=1e-12, atol=1e-13)


def test_gradients_are_linear_in_dout(oracle_mod):
    q, k, v, do = _rand(1, 6, 5, 2, 1, 4, 14)
    r1 = oracle_mod.attn_bwd_dense(q, k, v, do)
    do2 = I.bf16_bits(I.bits_to_bf16(do) * 2)  # exact in bf16
    r2 = oracle_mod.attn_bwd_dense(q, k, v, do2)
    for a, b in zip(r1, r2):
        assert np.allclose(2 * a, b, rtol=1e-13, atol=1e-15)

"""Shared helpers for the GPU parity tests: run the CUDA path through the
binding on seeded CPU inputs, and compare against the fp64 oracle."""
import numpy as np
import torch

import attention_forward_fa2_gb300 as fa
from attention_forward_fa2_gb300 import inputs as I

# Acceptance bar: max-abs error on O (bf16 output) and on LSE (fp32).
O_TOL = 2e-2
LSE_TOL = 1e-3


def gpu_dense(q, k, v, scale=None, causal=False):
    """CPU bf16 q [B,Nq,H,d], k/v [B,Nk,Hk,d] -> (o float64 [B,Nq,H,d], lse float64 [B,H,Nq])."""
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.forward_qk(dq, dk, dv, scale, causal=causal)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    return o.to(torch.float64).cpu().numpy(), lse.to(torch.float64).cpu().numpy()


def gpu_varlen(q, k, v, cu_q, cu_k, max_q, max_k, scale=None, causal=False):
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.forward_qk(dq, dk, dv, scale, cu_q.cuda(), cu_k.cuda(), max_q, max_k, causal=causal)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    return o.to(torch.float64).cpu().numpy(), lse.to(torch.float64).cpu().numpy()


def max_errs(o, lse, o_ref, lse_ref):
    assert np.all(np.isfinite(o)), "non-finite O"
    eo = float(np.max(np.abs(o - o_ref))) if o.size else 0.0
    el = float(np.max(np.abs(lse - lse_ref))) if lse.size else 0.0
    return eo, el


def assert_close(o, lse, o_ref, lse_ref, what=""):
    # Rows that see no key: LSE must be -inf on both sides (compared separately).
    lse, lse_ref = np.asarray(lse), np.asarray(lse_ref)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), "%s: rows without keys differ" % what
    lse, lse_ref = np.where(empty, 0.0, lse), np.where(empty, 0.0, lse_ref)
    eo, el = max_errs(o, lse, o_ref, lse_ref)
    assert eo <= O_TOL and el <= LSE_TOL, "%s: max|dO|=%.3g (tol %g) max|dLSE|=%.3g (tol %g)" % (
        what, eo, O_TOL, el, LSE_TOL)
    return eo, el


def sample_rows(B, Nq, H, n_random=48, seed=0):
    """Deterministic (b, h, i) rows: corners, tile and CTA boundaries, plus random."""
    special_i = sorted({0, 1, 63, 64, 127, 128, 129, 255, 256, 257, Nq // 2, Nq - 129, Nq - 128,
                        Nq - 2, Nq - 1} & set(range(Nq)))
    rows = set()
    for b in {0, B - 1}:
        for h in {0, H - 1}:
            for i in special_i:
                rows.add((b, h, i))
    rng = np.random.default_rng(seed)
    for _ in range(n_random):
        rows.add((int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(Nq))))
    return np.array(sorted(rows), dtype=np.int64)


def bits(t):
    return I.bf16_bits(t)


def fp8_bound(oracle_mod, q8, k8, vt8, qs, ks, vs, Nq, Nk, causal=False, scale=None):
    """Oracle output of the FP8 forward and the per-element bar it must meet.

    Returns (o_ref, lse_ref, bound) with bound [B, Nq, H, d].  The kernel
    computes the definition on the dequantised codes except that each weight
    p_j (relative to the kernel's reference maximum, which never exceeds the
    row maximum m) is rounded to e4m3 before O += P V: off by at most 2^-4 of
    itself (3 mantissa bits), or by 2^-10 absolute below the smallest normal
    2^-6.  The row sum uses the unrounded weights, so with l = sum_j e^(s_j - m)
    (the kernel's own sum is at least l):
        |dO_ic| <= 2^-4 sum_j P_ij |v_jc| + 2^-10 sum_{j seen by i} |v_jc| / l
    plus the bf16 rounding of the output (2^-9 of |O|, taken as 2^-8) and an
    absolute 1e-3 for the fp32 sums.  l = e^(m - LSE) comes from the oracle's
    row maximum and log-sum-exp."""
    o, lse, m, a = oracle_mod.attn_fp8_dense(q8, k8, vt8, qs, ks, vs, Nq, Nk, scale=scale, causal=causal,
                                             with_bound_terms=True)
    B, _, H, d = o.shape
    Hk = vt8.shape[1]
    G = H // Hk
    vabs = np.abs(oracle_mod.e4m3_decode(vt8[..., :Nk])) * np.asarray(vs, np.float64)[:, :, None, None]
    csum = np.cumsum(vabs, axis=3)                      # [B, Hk, d, Nk]: sum over keys 0..j
    fin = np.isfinite(lse)
    inv_l = np.exp(np.where(fin, m, 0.0) - np.where(fin, lse, 0.0)) * fin  # [B, H, Nq]; 0 without keys
    bound = 2.0 ** -4 * a + 2.0 ** -8 * np.abs(o) + 1e-3
    i = np.arange(Nq)
    last = np.minimum(Nk - 1, i + Nk - Nq) if causal else np.full(Nq, Nk - 1)
    for h in range(H):
        vsum = np.where(last[None, :, None] >= 0,
                        np.transpose(csum[:, h // G][:, :, np.maximum(last, 0)], (0, 2, 1)), 0.0)  # [B, Nq, d]
        bound[:, :, h, :] += 2.0 ** -10 * inv_l[:, h, :, None] * vsum
    return o, lse, bound

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

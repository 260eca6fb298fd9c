"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small cases compare every output element; the ten sweep workloads compare every
element of four whole heads and sampled rows of the others, in the same launch
configuration the benchmark times (the page and variable-length workloads are
compared on every element in test_parity_full_gpu.py).  Bar: max|dO| <= 2e-2,
max|dLSE| <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import attention_forward_fa2_gb300 as fa
from attention_forward_fa2_gb300 import inputs as I
from fa_testutil import (LSE_TOL, O_TOL, assert_close, bits, gpu_dense, gpu_varlen,
                         sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_forward_fa2_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.set_config(None)
    yield
    fa.set_config(None)


def _oracle_dense(oracle_mod, q, k, v, scale=None):
    return oracle_mod.attn_dense(bits(q), bits(k), bits(v), scale=scale)


# ----------------------------------------------------------- named workloads
def test_tiny_full_parity(oracle_mod):
    w = I.TINY
    q, k, v, _, _ = I.make(w)
    o, lse = gpu_dense(q, k, v)
    o_ref, lse_ref = _oracle_dense(oracle_mod, q, k, v)
    assert_close(o, lse, o_ref, lse_ref, "tiny")


def test_slice_full_parity(oracle_mod):
    w = I.SLICE
    q, k, v, _, _ = I.make(w)
    o, lse = gpu_dense(q, k, v)
    o_ref, lse_ref = _oracle_dense(oracle_mod, q, k, v)
    assert_close(o, lse, o_ref, lse_ref, "slice 64x4096")


@pytest.mark.parametrize("w", I.SWEEP, ids=[w.name for w in I.SWEEP])
def test_sweep_heads_full_and_rows_sampled(oracle_mod, w):
    """Each sweep workload in one launch (the benchmark's configuration): every element of
    four whole (b, h) heads -- (0, 0), (B-1, H-1) and two seeded ones -- plus sampled rows
    (corners, tile and CTA boundaries, random) over the other heads."""
    q, k, v, _, _ = I.make(w)
    o, lse = gpu_dense(q, k, v)
    rng = np.random.default_rng(w.seed + 7)
    heads = [(0, 0), (w.B - 1, w.H - 1)] + [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(2)]
    b = np.array([x[0] for x in heads])
    h = np.array([x[1] for x in heads])
    qb, kb, vb = bits(q), bits(k), bits(v)
    sel = lambda t: np.ascontiguousarray(t[b, :, h, :][:, :, None, :])  # heads as a batch of one-head problems
    o_ref, lse_ref = oracle_mod.attn_dense(sel(qb), sel(kb), sel(vb))
    assert_close(o[b, :, h, :][:, :, None, :], lse[b, h, :][:, None, :], o_ref, lse_ref, w.name + " heads")
    rows = sample_rows(w.B, w.Nq, w.H, n_random=24, seed=w.seed)
    o_rows, lse_rows = oracle_mod.attn_dense_rows(qb, kb, vb, rows)
    rb, rh, ri = rows[:, 0], rows[:, 1], rows[:, 2]
    assert_close(o[rb, ri, rh, :], lse[rb, rh, ri], o_rows, lse_rows, w.name + " rows")


# ----------------------------------------------------------------- edge cases
@pytest.mark.parametrize("B,Nq,Nk,H,d", [
    (1, 1, 1, 1, 128), (1, 1, 5, 1, 64), (2, 127, 129, 3, 128), (1, 128, 128, 2, 64),
    (1, 129, 127, 1, 128), (1, 255, 300, 2, 128), (1, 256, 256, 1, 64), (1, 257, 1, 2, 128),
    (3, 300, 513, 2, 64), (1, 64, 4096, 1, 64), (2, 513, 384, 1, 128), (1, 1000, 1000, 1, 128),
])
def test_ragged_shapes_full_parity(oracle_mod, B, Nq, Nk, H, d):
    q, k, v = I.make_dense(B, Nq, Nk, H, d, seed=1000 + Nq + Nk + d)
    o, lse = gpu_dense(q, k, v)
    o_ref, lse_ref = _oracle_dense(oracle_mod, q, k, v)
    assert_close(o, lse, o_ref, lse_ref, "ragged %s" % ((B, Nq, Nk, H, d),))


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_ragged_full_parity(oracle_mod, d):
    lens_q = [1, 127, 128, 129, 255, 256, 257, 300, 5, 700]
    lens_k = [3, 130, 128, 1, 255, 600, 257, 300, 129, 64]
    H = 3
    q, k, v, cu_q, cu_k = I.make_varlen(lens_q, H, d, 77 + d, lengths_k=lens_k)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, max(lens_q), max(lens_k))
    o_ref, lse_ref = oracle_mod.attn_varlen(bits(q), bits(k), bits(v), cu_q.numpy(), cu_k.numpy(),
                                            max(lens_q))
    valid = ~np.isnan(lse_ref)
    assert_close(o, lse[valid], o_ref, lse_ref[valid], "varlen ragged d%d" % d)


def test_varlen_empty_sequences(oracle_mod):
    lens_q = [0, 3, 200, 0, 130]
    lens_k = [4, 0, 131, 0, 300]
    q, k, v, cu_q, cu_k = I.make_varlen(lens_q, 2, 128, 91, lengths_k=lens_k)
    lse_init = torch.full((5, 2, 200), 123.0, device="cuda")
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.forward_qk(dq, dk, dv, None, cu_q.cuda(), cu_k.cuda(), 200, 300, lse=lse_init)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, info
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    o_ref, lse_ref = oracle_mod.attn_varlen(bits(q), bits(k), bits(v), cu_q.numpy(), cu_k.numpy(), 200)
    valid = ~np.isnan(lse_ref)
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lse[valid & ~fin]))       # sequence with no keys
    assert np.all(o[0:3] == 0.0)                           # its O rows are zero
    assert_close(o, lse[valid & fin], o_ref, lse_ref[valid & fin], "varlen empty")
    assert np.all(lse[~valid] == 123.0)                    # rows past a length untouched


def test_empty_problem_writes_nothing():
    o = torch.full((2, 4, 1, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((2, 1, 4), 7.0, device="cuda")
    z = torch.zeros((2, 0, 1, 128), dtype=torch.bfloat16, device="cuda")
    rc = fa.fa_fwd(z.data_ptr(), z.data_ptr(), z.data_ptr(), o.data_ptr(), lse.data_ptr(),
                   2, 0, 1, 128, 0.1, None, torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)


# ----------------------------------------------------- invariants on the GPU
def test_zero_query_gives_mean_of_values():
    B, N, H, d = 1, 300, 2, 128
    _, k, v = I.make_dense(B, N, N, H, d, 5)
    q = torch.zeros_like(k)
    o, lse = gpu_dense(q, k, v)
    mean = v.double().mean(dim=1).numpy()
    for i in (0, 150, 299):
        assert np.max(np.abs(o[:, i] - mean)) <= O_TOL
    assert np.max(np.abs(lse - math.log(N))) <= LSE_TOL


def test_identical_value_rows():
    B, N, H, d = 1, 400, 1, 64
    q, k, _ = I.make_dense(B, N, N, H, d, 6)
    row = torch.linspace(-2, 2, d).to(torch.bfloat16)
    v = row.expand(B, N, H, d).contiguous()
    o, _ = gpu_dense(q, k, v)
    assert np.max(np.abs(o - row.double().numpy())) <= O_TOL


def test_key_value_permutation_invariance():
    B, N, H, d = 1, 512, 2, 128
    q, k, v = I.make_dense(B, N, N, H, d, 8)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(N))
    o1, l1 = gpu_dense(q, k, v)
    o2, l2 = gpu_dense(q, k[:, perm].contiguous(), v[:, perm].contiguous())
    assert np.max(np.abs(o1 - o2)) <= O_TOL and np.max(np.abs(l1 - l2)) <= LSE_TOL


def test_large_scores_stay_finite(oracle_mod):
    """Scores of order 1e3: the online max keeps every exponent <= 0."""
    B, N, H, d = 1, 256, 1, 128
    q, k, v = I.make_dense(B, N, N, H, d, 9)
    q = (q.float() * 8).to(torch.bfloat16)
    o, lse = gpu_dense(q, k, v, scale=2.0)
    o_ref, lse_ref = oracle_mod.attn_dense(bits(q), bits(k), bits(v), scale=2.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert np.max(np.abs(o - o_ref)) <= O_TOL
    assert np.max(np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))) <= LSE_TOL


@pytest.mark.parametrize("spec", [None, "threshold=0", "reduce=quad,threshold=8"])
def test_reference_maximum_paths(oracle_mod, spec):
    """Key tiles whose scores step up by 0, 6, 20 and 21 (log2 units: the scale
    ln 2 makes a raw score r contribute 2^r): the second tile's block sum
    exceeds 2^8 while its maximum stays within the rescale threshold (the
    reference maximum must stay), the third and fourth move it.  Every
    output must still match the definition."""
    B, N, H, d = 1, 512, 2, 128
    q, k, v = I.make_dense(B, N, N, H, d, 31)
    q = torch.zeros_like(q)
    q[..., 0] = 1.0
    k = torch.zeros_like(k)
    for t, r in enumerate((0.0, 6.0, 20.0, 21.0)):
        k[:, 128 * t:128 * (t + 1), :, 0] = r
    fa.set_config(spec)
    try:
        o, lse = gpu_dense(q, k, v, scale=math.log(2.0))
    finally:
        fa.set_config(None)
    o_ref, lse_ref = oracle_mod.attn_dense(bits(q), bits(k), bits(v), scale=math.log(2.0))
    assert_close(o, lse, o_ref, lse_ref, "reference maximum paths %s" % spec)


def test_deterministic():
    q, k, v = I.make_dense(2, 700, 700, 2, 128, 10)
    o1, l1 = gpu_dense(q, k, v)
    o2, l2 = gpu_dense(q, k, v)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ------------------------------------------------------------ configurations
CONFIG_SPACE = ["br=%d,bc=%d,stages=%d,threshold=%d" % (br, bc, st, th)
                for br in (256, 128) for bc in (128, 64) for st in (2, 3, 4) for th in (0, 8)]
CONFIG_SPACE += ["reduce=quad,threshold=0", "reduce=quad,threshold=8"]


@pytest.mark.parametrize("spec", CONFIG_SPACE)
@pytest.mark.parametrize("d", [64, 128])
def test_every_config(oracle_mod, spec, d):
    fa.set_config(spec)
    try:
        q, k, v = I.make_dense(2, 333, 517, 2, d, 11 + d)
        o, lse = gpu_dense(q, k, v)
        o_ref, lse_ref = _oracle_dense(oracle_mod, q, k, v)
        assert_close(o, lse, o_ref, lse_ref, spec)
        lens = [129, 1, 384, 77]
        q, k, v, cu_q, cu_k = I.make_varlen(lens, 2, d, 12 + d)
        o, lse = gpu_varlen(q, k, v, cu_q, cu_k, 384, 384)
        o_ref, lse_ref = oracle_mod.attn_varlen(bits(q), bits(k), bits(v), cu_q.numpy(), cu_k.numpy(), 384)
        valid = ~np.isnan(lse_ref)
        assert_close(o, lse[valid], o_ref, lse_ref[valid], spec + " varlen")
    finally:
        fa.set_config(None)


def test_autotune_keeps_parity(oracle_mod):
    q, k, v = I.make_dense(1, 1024, 1024, 4, 128, 13)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    spec = fa.autotune(dq, dk, dv)
    assert spec.startswith("br=")
    o, lse = gpu_dense(q, k, v)
    o_ref, lse_ref = _oracle_dense(oracle_mod, q, k, v)
    assert_close(o, lse, o_ref, lse_ref, "autotuned " + spec)


# ------------------------------------------------------- failure detection
def test_device_checked_seqlens_error():
    """A sequence longer than the declared maximum is refused by the kernel's
    own check (nothing is read or written for it) and reported."""
    lens = [100, 300]
    q, k, v, cu_q, cu_k = I.make_varlen(lens, 1, 128, 14)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o = torch.zeros_like(dq)
    lse = torch.zeros((2, 1, 256), device="cuda")
    rc = fa.fa_fwd(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                   2, 256, 1, 128, 0.1, cu_q.cuda().data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    code, _ = fa.check_status()
    assert code == fa.FA_ERR_BAD_SEQLENS
    assert fa.check_status()[0] == fa.FA_OK  # cleared


def test_wait_timeout_is_reported_and_device_stays_usable(oracle_mod):
    rc = fa.fa_selftest_wait_timeout(20_000_000, torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    code, info = fa.check_status()
    assert code == fa.FA_ERR_TIMEOUT and info[2] == 99
    q, k, v = I.make_dense(1, 200, 200, 1, 128, 15)
    o, lse = gpu_dense(q, k, v)
    o_ref, lse_ref = _oracle_dense(oracle_mod, q, k, v)
    assert_close(o, lse, o_ref, lse_ref, "after timeout")


# ------------------------------------------------- causal and grouped heads
def _make_gqa(B, Nq, Nk, H, Hk, d, seed):
    g = torch.Generator().manual_seed(seed)
    return (I.randn_bf16((B, Nq, H, d), g), I.randn_bf16((B, Nk, Hk, d), g),
            I.randn_bf16((B, Nk, Hk, d), g))


@pytest.mark.parametrize("B,Nq,Nk,H,Hk,d", [
    (1, 256, 256, 2, 2, 128), (2, 300, 300, 2, 1, 128), (1, 129, 513, 2, 2, 64),
    (1, 513, 129, 2, 2, 128), (1, 1000, 1000, 4, 2, 128), (1, 1, 1, 1, 1, 128),
    (1, 64, 4096, 1, 1, 128), (2, 700, 700, 3, 3, 64), (1, 384, 256, 2, 1, 64),
])
def test_causal_full_parity(oracle_mod, B, Nq, Nk, H, Hk, d):
    q, k, v = _make_gqa(B, Nq, Nk, H, Hk, d, 2000 + Nq + Nk + d)
    o, lse = gpu_dense(q, k, v, causal=True)
    o_ref, lse_ref = oracle_mod.attn_dense(bits(q), bits(k), bits(v), causal=True)
    assert_close(o, lse, o_ref, lse_ref, "causal %s" % ((B, Nq, Nk, H, Hk, d),))


@pytest.mark.parametrize("H,Hk,d", [(8, 1, 128), (8, 2, 128), (8, 4, 64), (6, 3, 128)])
def test_grouped_heads_full_parity(oracle_mod, H, Hk, d):
    q, k, v = _make_gqa(2, 300, 517, H, Hk, d, 3000 + H + Hk + d)
    o, lse = gpu_dense(q, k, v)
    o_ref, lse_ref = oracle_mod.attn_dense(bits(q), bits(k), bits(v))
    assert_close(o, lse, o_ref, lse_ref, "gqa H%d Hk%d d%d" % (H, Hk, d))


@pytest.mark.parametrize("Hk", [3, 1])
def test_causal_varlen_full_parity(oracle_mod, Hk):
    lens_q = [1, 127, 128, 129, 300, 256, 40, 700]
    lens_k = [1, 130, 128, 100, 300, 600, 260, 700]
    H, d = 3, 128
    cu_q = torch.tensor([0] + list(np.cumsum(lens_q)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(np.cumsum(lens_k)), dtype=torch.int32)
    g = torch.Generator().manual_seed(70 + Hk)
    q = I.randn_bf16((int(cu_q[-1]), H, d), g)
    k = I.randn_bf16((int(cu_k[-1]), Hk, d), g)
    v = I.randn_bf16((int(cu_k[-1]), Hk, d), g)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, max(lens_q), max(lens_k), causal=True)
    o_ref, lse_ref = oracle_mod.attn_varlen(bits(q), bits(k), bits(v), cu_q.numpy(), cu_k.numpy(),
                                            max(lens_q), causal=True)
    valid = ~np.isnan(lse_ref)
    assert_close(o, lse[valid], o_ref, lse_ref[valid], "causal varlen Hk%d" % Hk)


@pytest.mark.parametrize("spec", ["stages=2,threshold=0", "stages=4,threshold=8",
                                  "br=128,bc=64,stages=3,threshold=8"])
def test_causal_gqa_configs(oracle_mod, spec):
    fa.set_config(spec)
    try:
        for d in (64, 128):
            q, k, v = _make_gqa(1, 400, 333, 4, 2, d, 80 + d)
            o, lse = gpu_dense(q, k, v, causal=True)
            o_ref, lse_ref = oracle_mod.attn_dense(bits(q), bits(k), bits(v), causal=True)
            assert_close(o, lse, o_ref, lse_ref, spec + " d%d" % d)
    finally:
        fa.set_config(None)


# ------------------------------------------------------------ key-split form
def _gpu_split(q, k, v, causal=False, num_splits=None):
    o, lse = fa.forward_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=causal, num_splits=num_splits)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def test_splitkv_slice_full_parity(oracle_mod):
    w = I.SLICE
    q, k, v, _, _ = I.make(w)
    assert fa.splitkv_num_splits(w.B, w.Nq, w.Nk, w.H, w.d) > 1
    o, lse = _gpu_split(q, k, v)
    o_ref, lse_ref = oracle_mod.attn_dense(bits(q), bits(k), bits(v))
    assert_close(o, lse, o_ref, lse_ref, "split slice")


@pytest.mark.parametrize("splits", [1, 2, 5, 16, 32])
@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_counts(oracle_mod, splits, causal):
    q, k, v = _make_gqa(1, 64, 4096, 2, 1, 128, 90 + splits)
    o, lse = _gpu_split(q, k, v, causal=causal, num_splits=splits)
    o_ref, lse_ref = oracle_mod.attn_dense(bits(q), bits(k), bits(v), causal=causal)
    assert_close(o, lse, o_ref, lse_ref, "split %d causal %s" % (splits, causal))


@pytest.mark.parametrize("B,Nq,Nk,H,Hk,d,causal", [
    (2, 300, 1000, 4, 2, 64, False), (1, 257, 999, 3, 3, 128, True), (1, 1, 129, 1, 1, 128, False),
    (3, 100, 2048, 2, 1, 64, True), (1, 513, 384, 2, 2, 128, True),
])
def test_splitkv_shapes(oracle_mod, B, Nq, Nk, H, Hk, d, causal):
    q, k, v = _make_gqa(B, Nq, Nk, H, Hk, d, 95 + Nq + Nk)
    o, lse = _gpu_split(q, k, v, causal=causal)
    o_ref, lse_ref = oracle_mod.attn_dense(bits(q), bits(k), bits(v), causal=causal)
    assert_close(o, lse, o_ref, lse_ref, "split %s" % ((B, Nq, Nk, H, Hk, d, causal),))


def test_splitkv_rejects_small_or_misaligned_workspace():
    q, k, v = _make_gqa(1, 64, 1024, 1, 1, 128, 99)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(dq)
    lse = torch.empty((1, 1, 64), device="cuda")
    n = fa.splitkv_num_splits(1, 64, 1024, 1, 128, 4)
    need = fa.splitkv_workspace_bytes(1, 64, 1, 128, n)
    ws = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = (dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 64, 1024, 1, 1,
            128, 0.1, 0, 4)
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need - 4, s) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr() + 8, need, s) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need, s) == fa.FA_OK
    assert fa.check_status()[0] == fa.FA_OK


# ------------------------------------------------------------ maximum sizes
def _device_bf16(shape, gen):
    return torch.randn(shape, generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)


def test_tensors_above_two_to_the_31_elements(oracle_mod):
    """B128 N4096 H32 d128: every input and the output hold 2^31 elements
    (4.3 GB each), so the last heads sit past any 32-bit element offset.  The
    first and the last (batch, head) are checked in full against the oracle."""
    B, N, H, d = 128, 4096, 32, 128
    gen = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = (_device_bf16((B, N, H, d), gen) for _ in range(3))
    assert q.numel() >= 2 ** 31
    o, lse = fa.forward_qk(q, k, v)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    for b, h in ((0, 0), (B - 1, H - 1)):
        sl = lambda t: bits(t[b:b + 1, :, h:h + 1].contiguous().cpu())
        o_ref, lse_ref = oracle_mod.attn_dense(sl(q), sl(k), sl(v))
        assert_close(o[b:b + 1, :, h:h + 1].double().cpu().numpy(), lse[b:b + 1, h:h + 1].double().cpu().numpy(),
                     o_ref, lse_ref, "b%d h%d" % (b, h))
    del q, k, v, o, lse
    torch.cuda.empty_cache()

"""GPU parity of the backward pass (fa_bwd through the C ABI) against the fp64 oracle.

Bar (derived from the arithmetic): P and dS enter the tensor-core products as
bf16 (relative rounding 2^-9, unbiased), accumulation is fp32 and the outputs
are rounded to bf16 (2^-9 relative), so each gradient tensor must satisfy
max|g - g_ref| <= 2e-2 * max|g_ref| and rms(g - g_ref) <= 1e-2 * rms(g_ref),
plus an absolute floor of 1e-4 (1e-5 for the rms) for gradients that vanish
exactly (one key: dQ = 0), where fp32 rounding of dP - D is all that is left.
The forward O and LSE that feed the backward come from the GPU forward.
"""
import numpy as np
import pytest
import torch

import attention_forward_fa2_gb300 as fa
from attention_forward_fa2_gb300 import build as fabuild
from attention_forward_fa2_gb300 import inputs as I

pytestmark = pytest.mark.gpu

MAX_REL = 2e-2
RMS_REL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    fabuild.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(B, Nq, Nk, H, Hk, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = I.randn_bf16((B, Nq, H, d), g)
    k = I.randn_bf16((B, Nk, Hk, d), g)
    v = I.randn_bf16((B, Nk, Hk, d), g)
    do = I.randn_bf16((B, Nq, H, d), g)
    return q, k, v, do


def _gpu_grads(q, k, v, do, causal):
    dq_, dk_, dv_, ddo = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.forward_qk(dq_, dk_, dv_, causal=causal)
    gq, gk, gv = fa.backward(dq_, dk_, dv_, o, lse, ddo, causal=causal)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    return tuple(t.double().cpu().numpy() for t in (gq, gk, gv))


def _assert_grads(got, ref, what):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(g)), "%s %s: non-finite" % (what, name)
        mx = float(np.abs(r).max()) if r.size else 0.0
        err = float(np.abs(g - r).max()) if r.size else 0.0
        rms_r = float(np.sqrt(np.mean(r ** 2))) if r.size else 0.0
        rms_e = float(np.sqrt(np.mean((g - r) ** 2))) if r.size else 0.0
        assert err <= MAX_REL * mx + 1e-4, "%s %s: max err %.3g vs max|ref| %.3g" % (what, name, err, mx)
        assert rms_e <= RMS_REL * rms_r + 1e-5, "%s %s: rms err %.3g vs rms ref %.3g" % (what, name, rms_e, rms_r)


@pytest.mark.parametrize("B,Nq,Nk,H,Hk", [
    (1, 256, 256, 2, 2),     # tiny: two key blocks, four query steps
    (2, 200, 333, 4, 2),     # ragged in both lengths, grouped heads
    (1, 1, 1, 1, 1),         # one query, one key
    (1, 65, 129, 2, 1),      # one row past a query step, one key past a key block (MQA)
    (1, 300, 100, 2, 2),     # more queries than keys
    (1, 1024, 1024, 2, 1),   # many steps per unit
    (3, 130, 260, 6, 3),
])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_oracle(oracle_mod, B, Nq, Nk, H, Hk, causal):
    q, k, v, do = _inputs(B, Nq, Nk, H, Hk, 128, 1000 + Nq + Nk + causal)
    got = _gpu_grads(q, k, v, do, causal)
    ref = oracle_mod.attn_bwd_dense(I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v), I.bf16_bits(do),
                                    causal=causal)[:3]
    _assert_grads(got, ref, "B%d Nq%d Nk%d H%d Hk%d causal%d" % (B, Nq, Nk, H, Hk, causal))


@pytest.mark.parametrize("B,Nq,Nk,H,Hk", [
    (1, 256, 256, 2, 2),
    (2, 200, 333, 4, 2),
    (1, 1, 1, 1, 1),
    (1, 300, 100, 2, 2),
    (1, 1024, 1024, 2, 1),
    (3, 130, 260, 6, 3),
])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_d64_matches_oracle(oracle_mod, B, Nq, Nk, H, Hk, causal):
    """d = 64: the same kernel with one 64-feature panel per tile (K padded to
    128 features for the transposed dQ product, whose extra rows are dropped)."""
    q, k, v, do = _inputs(B, Nq, Nk, H, Hk, 64, 2000 + Nq + Nk + causal)
    got = _gpu_grads(q, k, v, do, causal)
    ref = oracle_mod.attn_bwd_dense(I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v), I.bf16_bits(do),
                                    causal=causal)[:3]
    _assert_grads(got, ref, "B%d Nq%d Nk%d H%d Hk%d causal%d" % (B, Nq, Nk, H, Hk, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_page_workload_many_heads(oracle_mod, causal):
    """The page workload (B16 N4096 H16 d128) in one call; checked in full
    against the oracle: every head of the first and the last batch, and one
    head of every other batch (head b of batch b), 46 of the 256 (batch, head)
    pairs."""
    w = I.PAGE
    q, k, v, _, _ = I.make(w)
    do = I.randn_bf16(tuple(q.shape), torch.Generator().manual_seed(77))
    got = _gpu_grads(q, k, v, do, causal)
    # Whole batches: the oracle runs their heads in parallel.
    for b in (0, w.B - 1):
        sl = lambda t: t[b:b + 1].contiguous()
        ref = oracle_mod.attn_bwd_dense(I.bf16_bits(sl(q)), I.bf16_bits(sl(k)), I.bf16_bits(sl(v)),
                                        I.bf16_bits(sl(do)), causal=causal)[:3]
        _assert_grads(tuple(g[b:b + 1] for g in got), ref, "page b%d causal%d" % (b, causal))
    # Head b of batch b, gathered as a batch of single-head problems.
    pairs = [(b, b % w.H) for b in range(1, w.B - 1)]
    pick = lambda t: torch.stack([t[b, :, h:h + 1] for b, h in pairs]).contiguous()
    ref = oracle_mod.attn_bwd_dense(I.bf16_bits(pick(q)), I.bf16_bits(pick(k)), I.bf16_bits(pick(v)),
                                    I.bf16_bits(pick(do)), causal=causal)[:3]
    mine = tuple(np.stack([g[b, :, h:h + 1] for b, h in pairs]) for g in got)
    _assert_grads(mine, ref, "page diagonal heads causal%d" % causal)


def test_key_gradients_sum_to_zero_on_gpu():
    """sum_j dK_j = 0 for every (b, head) (softmax rows annihilate constants)."""
    q, k, v, do = _inputs(2, 512, 640, 4, 4, 128, 5)
    _, gk, _ = _gpu_grads(q, k, v, do, False)
    col = np.abs(gk.sum(axis=1)).max()
    assert col <= 2e-2 * np.abs(gk).max() * np.sqrt(640), col


def test_no_queries_gives_zero_key_gradients():
    k = torch.randn(1, 200, 2, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.randn_like(k)
    q = torch.empty(1, 0, 2, 128, dtype=torch.bfloat16, device="cuda")
    o, do = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty(1, 2, 0, dtype=torch.float32, device="cuda")
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    _, gk, gv = fa.backward(q, k, v, o, lse, do, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa.check_status()[0] == fa.FA_OK
    assert torch.all(gk == 0) and torch.all(gv == 0)


def test_backward_errors():
    q = torch.randn(1, 64, 2, 32, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 64, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.backward(q, q, q, q, lse, q)  # d = 32: not built
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    q = torch.randn(1, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.backward(q, q, q, q, lse, q, workspace=ws)
    assert e.value.code == fa.FA_ERR_INVALID_ARG


def test_backward_is_repeatable():
    """dK and dV are sums in a fixed order (bit-identical reruns); dQ is
    accumulated with L2 reduce-adds whose order varies, so it is compared
    within rounding."""
    q, k, v, do = _inputs(1, 512, 512, 2, 2, 128, 9)
    a = _gpu_grads(q, k, v, do, False)
    b = _gpu_grads(q, k, v, do, False)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert np.abs(a[0] - b[0]).max() <= 1e-2 * np.abs(a[0]).max()


# ------------------------------------------------------------ variable length
def _packed(lengths, H, d, gen):
    total = int(sum(lengths))
    return I.randn_bf16((total, H, d), gen)


@pytest.mark.parametrize("lq,lk,H,Hk,d", [
    ([129, 1, 384, 77], None, 2, 1, 128),       # ragged ends, one-row sequence, MQA
    ([100, 260, 128], [300, 50, 128], 2, 2, 128),  # different query and key lengths
    ([0, 200, 0, 33], [5, 200, 7, 40], 2, 2, 128),  # empty query sequences (keys still get dk = dv = 0)
    ([129, 70, 256], None, 4, 2, 64),            # d = 64
])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_varlen_matches_oracle(oracle_mod, lq, lk, H, Hk, d, causal):
    """Packed sequences: each sequence's gradients equal the dense oracle's
    on that sequence alone (the causal mask is bottom-right per sequence)."""
    lk = lq if lk is None else lk
    g = torch.Generator().manual_seed(3000 + sum(lq) + causal)
    q = _packed(lq, H, d, g)
    k, v = _packed(lk, Hk, d, g), _packed(lk, Hk, d, g)
    do = _packed(lq, H, d, g)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lq)]), dtype=torch.int32)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lk)]), dtype=torch.int32)
    mq, mk = max(lq), max(lk)
    dq_, dk_, dv_, ddo = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.forward_qk(dq_, dk_, dv_, None, cu_q.cuda(), cu_k.cuda(), mq, mk, causal=causal)
    dk_out = torch.full_like(dk_, 7.0)
    dv_out = torch.full_like(dv_, 7.0)
    gq, gk, gv = fa.backward_varlen(dq_, dk_, dv_, o, lse, ddo, cu_q.cuda(), cu_k.cuda(), mq, mk, causal=causal,
                                    dk=dk_out, dv=dv_out)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    gq, gk, gv = (t.double().cpu().numpy() for t in (gq, gk, gv))
    for b in range(len(lq)):
        q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        what = "seq %d (lq %d lk %d) causal%d d%d" % (b, lq[b], lk[b], causal, d)
        if k1 == k0:
            continue
        if q1 == q0:
            assert np.all(gk[k0:k1] == 0) and np.all(gv[k0:k1] == 0), what
            continue
        sl = lambda t, a, z: I.bf16_bits(t[a:z].unsqueeze(0).contiguous())
        ref = oracle_mod.attn_bwd_dense(sl(q, q0, q1), sl(k, k0, k1), sl(v, k0, k1), sl(do, q0, q1),
                                        causal=causal)[:3]
        mine = (gq[None, q0:q1], gk[None, k0:k1], gv[None, k0:k1])
        _assert_grads(mine, ref, what)


def test_backward_varlen_rejects_half_given_seqlens():
    q = torch.randn(10, 2, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 10], dtype=torch.int32, device="cuda")
    lse = torch.zeros(1, 2, 10, device="cuda")
    rc = fa.fa_bwd_varlen(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), lse.data_ptr(),
                          q.data_ptr(), q.data_ptr(), q.data_ptr(), cu.data_ptr(), None, 1, 10, 10, 2, 2, 128,
                          0.1, 0, q.data_ptr(), 1 << 20, None)
    assert rc == fa.FA_ERR_INVALID_ARG


def test_backward_varlen_reports_lengths_above_the_maximum():
    """A sequence longer than the declared maximum is reported by the kernel
    (FA_ERR_BAD_SEQLENS through fa_check_status) and its units write nothing."""
    H, d = 2, 128
    g = torch.Generator().manual_seed(71)
    lens = [100, 200]
    q = _packed(lens, H, d, g).cuda()
    k, v, do = (_packed(lens, H, d, g).cuda() for _ in range(3))
    cu = torch.tensor([0, 100, 300], dtype=torch.int32, device="cuda")
    o, lse = fa.forward_qk(q, k, v, None, cu, cu, 200, 200)
    assert fa.check_status()[0] == fa.FA_OK
    fa.backward_varlen(q, k, v, o, lse[:, :, :150].contiguous(), do, cu, cu, 150, 150)
    rc, info = fa.check_status()
    assert rc == fa.FA_ERR_BAD_SEQLENS, (fa.strerror(rc), info)
    # The context stays usable.
    fa.backward_varlen(q, k, v, o, lse, do, cu, cu, 200, 200)
    assert fa.check_status()[0] == fa.FA_OK


def test_backward_tensors_above_two_to_the_31_elements(oracle_mod):
    """B128 N4096 H32 d128 (2^31 elements per tensor): the first and the last
    (batch, head) gradients against the oracle."""
    B, N, H, d = 128, 4096, 32, 128
    gen = torch.Generator(device="cuda").manual_seed(6)
    mk = lambda: torch.randn((B, N, H, d), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    q, k, v, do = mk(), mk(), mk(), mk()
    o, lse = fa.forward_qk(q, k, v)
    gq, gk, gv = fa.backward(q, k, v, o, lse, do)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    for b, h in ((0, 0), (B - 1, H - 1)):
        sl = lambda t: I.bf16_bits(t[b:b + 1, :, h:h + 1].contiguous().cpu())
        ref = oracle_mod.attn_bwd_dense(sl(q), sl(k), sl(v), sl(do))[:3]
        mine = tuple(t[b:b + 1, :, h:h + 1].double().cpu().numpy() for t in (gq, gk, gv))
        _assert_grads(mine, ref, "b%d h%d" % (b, h))
    del q, k, v, do, o, lse, gq, gk, gv
    torch.cuda.empty_cache()

"""Every output element of the full-size workloads against the fp64 oracle.

The page workload (B16 N4096 H16 d128; "Flash Attention 2 Chapter2",
introduction), dense and causal, and the 32-sequence variable-length workload
("Flash Attention实现深度解析" §3.1 packed layout), dense and causal, each in
the launch configuration the benchmark times; plus mid-size problems with
several work units per CTA of the persistent grid (512 units of 256 query
rows for 152 SMs: "GPU 内核与FlashAttention" §14.2 spreads query blocks over
the GPU), where the Q, K/V ring and O hand-offs between consecutive units of
one CTA are exercised on every element.  The oracle runs one batch at a time
to bound host memory.  Bar: max|dO| <= 2e-2, max|dLSE| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import attention_forward_fa2_gb300 as fa
from attention_forward_fa2_gb300 import inputs as I
from fa_testutil import assert_close, bits, gpu_varlen

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


def _gpu_dense_bf16(q, k, v, causal):
    """(o bf16 [B, Nq, H, d] on the CPU, lse float32 [B, H, Nq] on the CPU)."""
    o, lse = fa.forward_qk(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    return o.cpu(), lse.cpu()


def _full_dense(oracle_mod, q, k, v, causal, what):
    o, lse = _gpu_dense_bf16(q, k, v, causal)
    worst = (0.0, 0.0)
    for b in range(q.shape[0]):
        sl = slice(b, b + 1)
        o_ref, lse_ref = oracle_mod.attn_dense(bits(q[sl]), bits(k[sl]), bits(v[sl]), causal=causal)
        eo, el = assert_close(o[sl].double().numpy(), lse[sl].double().numpy(), o_ref, lse_ref,
                              "%s b%d" % (what, b))
        worst = (max(worst[0], eo), max(worst[1], el))
    return worst


@pytest.mark.parametrize("causal", [False, True])
def test_page_workload_every_element(oracle_mod, causal):
    w = I.PAGE
    q, k, v, _, _ = I.make(w)
    _full_dense(oracle_mod, q, k, v, causal, "page causal%d" % causal)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_workload_every_element(oracle_mod, causal):
    w = I.VARLEN
    q, k, v, cu_q, cu_k = I.make(w)
    maxlen = max(w.lengths)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, maxlen, maxlen, causal=causal)
    o_ref, lse_ref = oracle_mod.attn_varlen(bits(q), bits(k), bits(v), cu_q.numpy(), cu_k.numpy(), maxlen,
                                            causal=causal)
    valid = ~np.isnan(lse_ref)
    assert_close(o, lse[valid], o_ref, lse_ref[valid], "varlen causal%d" % causal)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_multi_unit_per_cta_every_element(oracle_mod, d, causal):
    """B4 N2048 H16: 512 units of 256 query rows (256 causal pairs), so each CTA
    of the 152-CTA persistent grid runs several units back to back."""
    q, k, v = I.make_dense(4, 2048, 2048, 16, d, seed=3100 + d + causal)
    _full_dense(oracle_mod, q, k, v, causal, "B4 N2048 H16 d%d causal%d" % (d, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_multi_unit_varlen_every_element(oracle_mod, causal):
    """12 packed sequences of 300..2048 tokens (tails not multiples of 128), H16 d128:
    over a thousand units, most CTAs walking several of them."""
    lens = [int(x) for x in np.random.default_rng(31).integers(300, 2048, size=12, endpoint=True)]
    q, k, v, cu_q, cu_k = I.make_varlen(lens, 16, 128, 3200 + causal)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, max(lens), max(lens), causal=causal)
    o_ref, lse_ref = oracle_mod.attn_varlen(bits(q), bits(k), bits(v), cu_q.numpy(), cu_k.numpy(), max(lens),
                                            causal=causal)
    valid = ~np.isnan(lse_ref)
    assert_close(o, lse[valid], o_ref, lse_ref[valid], "varlen 12 seqs causal%d" % causal)


# ------------------------------------------------------ the main call itself
def _call_fa_fwd(q, k, v, N, cu=None, B=None):
    """fa_fwd through the C ABI: self-attention shapes, one cu_seqlens for q and k."""
    H, d = q.shape[-2], q.shape[-1]
    B = q.shape[0] if B is None else B
    o = torch.empty_like(q)
    lse = torch.full((B, H, N), 123.0, dtype=torch.float32, device="cuda")
    rc = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, N, H, d,
                   1.0 / d ** 0.5, None if cu is None else cu.data_ptr(),
                   torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK, fa.strerror(rc)
    rc, info = fa.check_status()
    assert rc == fa.FA_OK, (fa.strerror(rc), info)
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("B,N,H,d", [(2, 300, 3, 128), (1, 1000, 2, 64), (3, 129, 1, 128)])
def test_fa_fwd_dense_through_the_c_abi(oracle_mod, B, N, H, d):
    q, k, v = I.make_dense(B, N, N, H, d, seed=3300 + N + d)
    o, lse = _call_fa_fwd(q.cuda(), k.cuda(), v.cuda(), N)
    o_ref, lse_ref = oracle_mod.attn_dense(bits(q), bits(k), bits(v))
    assert_close(o, lse, o_ref, lse_ref, "fa_fwd dense %s" % ((B, N, H, d),))


@pytest.mark.parametrize("d", [128, 64])
def test_fa_fwd_varlen_through_the_c_abi(oracle_mod, d):
    lens = [5, 128, 400, 0, 257, 1000]
    q, k, v, cu, _ = I.make_varlen(lens, 2, d, 3400 + d)
    N = max(lens)
    o, lse = _call_fa_fwd(q.cuda(), k.cuda(), v.cuda(), N, cu=cu.cuda(), B=len(lens))
    o_ref, lse_ref = oracle_mod.attn_varlen(bits(q), bits(k), bits(v), cu.numpy(), cu.numpy(), N)
    valid = ~np.isnan(lse_ref)
    assert_close(o, lse[valid], o_ref, lse_ref[valid], "fa_fwd varlen d%d" % d)
    assert np.all(lse[~valid] == 123.0)  # entries past each length untouched

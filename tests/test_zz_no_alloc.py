"""The allocation-free key-split entry point, fa_fwd_splitkv_noalloc.

It serves callers that cannot allocate device memory when attention runs (a
runtime that reserved all of its memory at start-up, a real-time path, a C
caller without a memory pool): they pass only inputs and outputs, and the
library uses a fixed scratch array of its own.  Checked here through the C ABI
against fa_fwd_splitkv with a caller-owned workspace, on two calls in a row
(the second call finds the first call's leftovers in the shared scratch), after
a larger call whose leftovers sit where a causal call's empty splits write, for
device memory left unchanged by repeated calls, for the same error codes as the
workspace entry, and for the size limit.  This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import attention_forward_fa2_gb300 as fa
from attention_forward_fa2_gb300 import build as fabuild
from attention_forward_fa2_gb300 import inputs as I
from fa_testutil import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    fabuild.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(B, Nq, Nk, H, Hk, d, seed):
    g = torch.Generator().manual_seed(seed)
    return tuple(t.cuda() for t in (I.randn_bf16((B, Nq, H, d), g), I.randn_bf16((B, Nk, Hk, d), g),
                                    I.randn_bf16((B, Nk, Hk, d), g)))


def _with_workspace(q, k, v, flags, splits):
    """The existing entry point, with a workspace the caller allocates."""
    B, Nq, H, d = q.shape
    Nk, Hk = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    n = fa.splitkv_num_splits(B, Nq, Nk, H, d, splits)
    ws = torch.empty(fa.splitkv_workspace_bytes(B, Nq, H, d, n), dtype=torch.uint8, device="cuda")
    rc = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           B, Nq, Nk, H, Hk, d, 1.0 / d ** 0.5, flags, n, ws.data_ptr(),
                           ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    assert fa.check_status()[0] == fa.FA_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def _no_alloc(q, k, v, flags, splits):
    """The allocation-free entry point: inputs and outputs only."""
    B, Nq, H, d = q.shape
    Nk, Hk = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    rc = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, Nq, Nk, H, Hk, d, 1.0 / d ** 0.5, flags,
                                   splits, torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK, fa.strerror(rc)
    assert fa.check_status()[0] == fa.FA_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("B,Nq,Nk,H,Hk,d,flags,splits", [
    (1, 64, 4096, 2, 1, 128, 0, 0),                  # the 64 x 4096 slice, chosen split count
    (1, 64, 4096, 2, 1, 128, fa.FA_FLAG_CAUSAL, 8),
    (2, 130, 1000, 4, 2, 64, 0, 5),
])
def test_matches_workspace_entry_on_two_calls(B, Nq, Nk, H, Hk, d, flags, splits):
    q, k, v = _inputs(B, Nq, Nk, H, Hk, d, 500 + Nq + splits)
    o_ref, lse_ref = _with_workspace(q, k, v, flags, splits)
    for _ in range(2):
        o, lse = _no_alloc(q, k, v, flags, splits)
        assert_close(o, lse, o_ref, lse_ref, "no-alloc vs workspace")
    # a different problem in between, then the first again: leftovers never leak
    q2, k2, v2 = _inputs(1, 200, 700, 2, 2, 128, 7)
    _no_alloc(q2, k2, v2, 0, 3)
    o, lse = _no_alloc(q, k, v, flags, splits)
    assert_close(o, lse, o_ref, lse_ref, "no-alloc after another problem")


def test_leftovers_of_a_larger_call_do_not_reach_empty_splits():
    # A large non-causal call fills much of the shared scratch; then a causal
    # call with more queries than keys, where the first query tile sees no key
    # at all and the later splits of the second tile see none either (those
    # splits write o = 0, LSE = -inf into the scratch for the merge).
    q1, k1, v1 = _inputs(2, 256, 2048, 4, 4, 128, 901)  # 8 splits: 8.5 MB of the 16 MiB
    _no_alloc(q1, k1, v1, 0, 8)
    q, k, v = _inputs(1, 512, 384, 2, 2, 128, 902)
    o_ref, lse_ref = _with_workspace(q, k, v, fa.FA_FLAG_CAUSAL, 3)
    o, lse = _no_alloc(q, k, v, fa.FA_FLAG_CAUSAL, 3)
    assert np.all(np.isneginf(lse[:, :, :128]))  # rows that see no key
    assert_close(o, lse, o_ref, lse_ref, "no-alloc causal after a larger call")


def test_allocates_nothing():
    q, k, v = _inputs(2, 64, 4096, 4, 2, 128, 903)
    o = torch.empty_like(q)
    lse = torch.empty((2, 4, 64), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        return fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), 2, 64, 4096, 4, 2, 128, 0.125, 0, 0, stream)

    assert call() == fa.FA_OK  # first call: the one-time set-up (module load, address lookup)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        assert call() == fa.FA_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "device memory changed by %d bytes" % (free0 - free1)
    assert fa.check_status()[0] == fa.FA_OK


def test_same_error_codes_as_the_workspace_entry():
    q = torch.zeros((1, 64, 2, 96), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 2, 64), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), lse.data_ptr(), 1, 64, 64, 2, 2, 96,
            0.1, 0)
    rc_ws = fa.fa_fwd_splitkv(*args, 0, None, 0, stream)
    rc_na = fa.fa_fwd_splitkv_noalloc(*args, 0, stream)
    assert rc_ws == rc_na == fa.FA_ERR_UNSUPPORTED  # d = 96
    bad_scale = args[:10] + (128, -1.0, 0)
    assert fa.fa_fwd_splitkv_noalloc(*bad_scale, 0, stream) == fa.FA_ERR_INVALID_ARG


def test_rejects_problems_beyond_the_scratch():
    # 64 x 32 heads x 1024 queries, d=128, one split: 64*32*1024*129*4 bytes >> 16 MiB.
    q = torch.zeros((64, 1024, 32, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((64, 1024, 32, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 3.0)
    lse = torch.full((64, 32, 1024), 3.0, device="cuda")
    rc = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), 64, 1024, 1024, 32, 32, 128, 0.1, 0, 1,
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_ERR_SCRATCH_LIMIT
    assert "16 MiB" in fa.strerror(rc)
    torch.cuda.synchronize()
    assert torch.all(o == 3.0) and torch.all(lse == 3.0)  # nothing was launched

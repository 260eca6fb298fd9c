"""Phase clocks of the forward kernel (the build with FA_PHASE_CLOCKS=1).

"GPU 内核与 FlashAttention" §8 profiles a kernel before tuning it; the phase
clocks say, per CTA, how many cycles each role spends waiting on each barrier
and working.  Checked on the tiny workload (B1 H2 N256 d128: two work units of
two 128-row query tiles, two key/value tiles each, on a grid of two CTAs): the event
counts are exactly those of the schedule, the cycle counts are positive, the
timer is ordered, and the outputs are bit-identical to the default build's.
The default build has no instrumentation and refuses a buffer.
"""
import math

import numpy as np
import pytest
import torch

import attention_forward_fa2_gb300 as fa
from attention_forward_fa2_gb300 import build as fabuild
from attention_forward_fa2_gb300 import inputs as I

pytestmark = pytest.mark.gpu

# Slot map of the kernel source (PhaseBase + PhaseSlot).
MMA, LOAD, SOFT0, SOFT1, EPI, TIMER = 0, 8, 16, 24, 32, 40


@pytest.fixture(scope="module")
def phase_lib():
    fabuild.build()
    fabuild.build(phase=True)
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return fa.load_library(fa.PHASE_LIB_PATH)


def _forward(L, q, k, v, B, N, H, d):
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, N, N, H, H, d,
                     1.0 / math.sqrt(d), None, None, 0, stream)
    assert rc == fa.FA_OK
    assert L.fa_check_status(stream, None) == fa.FA_OK
    return o, lse


def test_default_build_has_no_phase_clocks():
    buf = torch.zeros(1024, dtype=torch.int64, device="cuda")
    assert fa.lib().fa_set_phase_buffer(buf.data_ptr(), buf.numel()) == fa.FA_ERR_UNSUPPORTED


def test_phase_clocks_on_tiny(phase_lib):
    L = phase_lib
    w = I.TINY
    q, k, v, _, _ = I.make(w)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    buf = torch.full((4 * 48,), -1, dtype=torch.int64, device="cuda")
    assert L.fa_set_phase_buffer(buf.data_ptr(), 10) == fa.FA_ERR_INVALID_ARG   # smaller than one CTA
    words = L.fa_set_phase_buffer(buf.data_ptr(), buf.numel())
    assert words == 48
    try:
        o, lse = _forward(L, q, k, v, w.B, w.Nq, w.H, w.d)
    finally:
        assert L.fa_set_phase_buffer(None, 0) == words
    ph = buf.view(-1, words).cpu().numpy()
    # Two work items (units of 256 query rows) on a grid of two CTAs; a CTA
    # that starts first may take over the other's item, so the counts are
    # checked summed over the CTAs that ran.
    ran = [c for c in range(ph.shape[0]) if ph[c, TIMER] != -1]
    assert 1 <= len(ran) <= 2 and set(ran) <= {0, 1}
    r = ph[ran].sum(axis=0)
    assert r[MMA + 6] == 2                    # units
    assert r[MMA + 5] == 6                    # key/value steps j = 0..nkv (nkv = 2) per unit
    assert r[LOAD + 3] == 6                   # ring slots filled
    assert r[SOFT0 + 2] == 4 and r[SOFT1 + 2] == 4   # softmax steps per tile
    assert r[EPI + 4] == 4                    # epilogue tiles
    for c in ran:
        q_ = ph[c]
        assert q_[SOFT0 + 3] >= 1             # the first block of a row takes the maximum
        for base, slots in ((MMA, (0, 1, 2, 3, 4)), (LOAD, (0, 1, 2)), (SOFT0, (0, 1, 4, 5, 6)),
                            (SOFT1, (0, 1, 4, 5, 6)), (EPI, (0, 1, 2, 3))):
            assert all(q_[base + i] >= 0 for i in slots), (c, base)
        assert q_[MMA + 4] > 0 and q_[SOFT0 + 1] > 0 and q_[SOFT1 + 1] > 0 and q_[EPI + 1] > 0
        assert q_[SOFT0 + 5] > 0 and q_[SOFT0 + 6] > 0 and q_[SOFT1 + 5] > 0 and q_[SOFT1 + 6] > 0
        assert 0 < q_[TIMER] <= q_[TIMER + 1]  # %globaltimer at start and end
    assert np.all(ph[2:] == -1)               # CTAs past the grid write nothing
    # The instrumentation does not change the arithmetic.
    o_ref, lse_ref = fa.forward(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse, lse_ref)


def test_phase_buffer_too_small_for_the_grid(phase_lib):
    L = phase_lib
    q, k, v = (t.cuda() for t in I.make_dense(2, 512, 512, 4, 128, seed=5))
    buf = torch.zeros(48, dtype=torch.int64, device="cuda")       # room for one CTA only
    assert L.fa_set_phase_buffer(buf.data_ptr(), buf.numel()) == 48
    try:
        o = torch.empty_like(q)
        lse = torch.empty((2, 4, 512), dtype=torch.float32, device="cuda")
        rc = L.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 2, 512, 512, 4, 4,
                         128, 0.088, None, None, 0, torch.cuda.current_stream().cuda_stream)
        assert rc == fa.FA_ERR_INVALID_ARG     # 8 CTAs need 384 words; nothing is launched
    finally:
        L.fa_set_phase_buffer(None, 0)
    assert torch.all(buf == 0)

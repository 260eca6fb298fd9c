"""Host-side checks of the C-ABI library: it builds, loads, exports every symbol
include/fa.h declares, and rejects bad arguments before touching a device.
No call here launches GPU work."""
import os
import re

import pytest
import torch

import attention_forward_fa2_gb300 as fa
from attention_forward_fa2_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def L():
    fabuild.build()
    return fa.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_exactly_the_binding_exports():
    assert _declared() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_version_and_strerror(L):
    assert fa.version() == 100
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert fa.strerror(code) and fa.strerror(code) != "unknown error"
    assert fa.strerror(-99) == "unknown error"


def test_config_spec_roundtrip(L):
    try:
        fa.set_config("stages=3,threshold=0")
        assert fa.get_config(64, 4096) == "br=256,bc=128,stages=3,threshold=0,reduce=thread"
        assert fa.get_config(128, 4096) == "br=256,bc=128,stages=2,threshold=0,reduce=thread"  # two slots fit
        fa.set_config("threshold=8")
        assert fa.get_config(64, 512) == "br=256,bc=128,stages=4,threshold=8,reduce=thread"
        fa.set_config("br=128,bc=64,stages=4")
        assert fa.get_config(128, 4096) == "br=128,bc=64,stages=4,threshold=8,reduce=thread"
        assert fa.get_config(64, 100, True) == "br=128,bc=64,stages=4,threshold=8,reduce=thread"
        fa.set_config("reduce=quad,stages=2")
        assert fa.get_config(128, 4096) == "br=256,bc=128,stages=2,threshold=8,reduce=quad"
        assert fa.get_config(64, 4096) == "br=256,bc=128,stages=3,threshold=8,reduce=quad"
        fa.set_config("reduce=quad,bc=64")  # built for 128-key tiles only
        assert fa.get_config(64, 4096) == "br=256,bc=64,stages=4,threshold=8,reduce=thread"
        for bad in ("stages=5", "stages=1", "threshold=-1", "foo=1", "stages", "threshold=nan",
                    "bc=32", "bc=256", "br=64", "br=512", "stages=", "bc=", "br=1e3",
                    "reduce=warp", "reduce="):
            with pytest.raises(fa.FaError):
                fa.set_config(bad)
    finally:
        fa.set_config(None)
    assert fa.get_config(128, 4096) == "br=256,bc=128,stages=2,threshold=8,reduce=thread"
    assert fa.get_config(64, 4096) == "br=256,bc=128,stages=3,threshold=8,reduce=thread"


def test_timeout_setter(L):
    assert L.fa_set_timeout_ns(5_000_000) == 0
    assert L.fa_set_timeout_ns(0) == 0  # back to the default


# Fake, never-dereferenced addresses: validation fails before any CUDA call.
A = 0x10000
MIS = 0x10008  # 8-byte aligned only


def _fwd(L, q=A, k=A, v=A, o=A, lse=A, B=1, N=128, H=1, d=128, scale=0.1, cu=None):
    return L.fa_fwd(q, k, v, o, lse, B, N, H, d, scale, cu, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.5), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(B=-1), fa.FA_ERR_INVALID_ARG),
    (dict(N=-3), fa.FA_ERR_INVALID_ARG),
    (dict(H=-2), fa.FA_ERR_INVALID_ARG),
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(q=MIS), fa.FA_ERR_ALIGN),
    (dict(v=MIS), fa.FA_ERR_ALIGN),
    (dict(o=MIS), fa.FA_ERR_ALIGN),
    (dict(lse=A + 2), fa.FA_ERR_ALIGN),
    (dict(H=70000), fa.FA_ERR_INVALID_ARG),
    (dict(B=70000), fa.FA_ERR_INVALID_ARG),
    (dict(B=40000, N=65536), fa.FA_ERR_INVALID_ARG),
])
def test_argument_errors(L, kw, code):
    assert _fwd(L, **kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(N=0), dict(H=0), dict(B=0, q=0, k=0, v=0, o=0, lse=0)])
def test_empty_problems_are_noops(L, kw):
    assert _fwd(L, **kw) == fa.FA_OK


def test_qk_form_argument_errors(L):
    # exactly one cu_seqlens pointer
    assert L.fa_fwd_qk(A, A, A, A, A, 1, 8, 8, 1, 128, 0.1, A, None, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_qk(A, A, A, A, A, 1, 8, 8, 1, 128, 0.1, None, A, None) == fa.FA_ERR_INVALID_ARG
    # dense with queries but no keys
    assert L.fa_fwd_qk(A, A, A, A, A, 1, 8, 0, 1, 128, 0.1, None, None, None) == fa.FA_ERR_INVALID_ARG
    # misaligned cu_seqlens
    assert L.fa_fwd_qk(A, A, A, A, A, 1, 8, 8, 1, 128, 0.1, A + 2, A, None) == fa.FA_ERR_ALIGN


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a device")
def test_valid_call_without_device_reports_no_device(L):
    assert _fwd(L) == fa.FA_ERR_NO_DEVICE


def test_selftest_argument_range(L):
    assert L.fa_selftest_wait_timeout(0, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_selftest_wait_timeout(20_000_000_000, None) == fa.FA_ERR_INVALID_ARG


def test_torch_wrapper_rejects_cpu_tensors(L):
    q = torch.zeros(1, 8, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fa.forward(q, q, q)


def test_product_package_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "attention_forward_fa2_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "attn_ref" not in text and "liboracle" not in text, f


def test_ex_form_argument_errors(L):
    ex = L.fa_fwd_ex
    # H not a multiple of Hk, Hk = 0, unknown flag bits
    assert ex(A, A, A, A, A, 1, 8, 8, 6, 4, 128, 0.1, None, None, 0, None) == fa.FA_ERR_INVALID_ARG
    assert ex(A, A, A, A, A, 1, 8, 8, 4, 0, 128, 0.1, None, None, 0, None) == fa.FA_ERR_INVALID_ARG
    assert ex(A, A, A, A, A, 1, 8, 8, 4, 2, 128, 0.1, None, None, 4, None) == fa.FA_ERR_INVALID_ARG
    assert ex(A, A, A, A, A, 1, 8, 8, 4, -1, 128, 0.1, None, None, 0, None) == fa.FA_ERR_INVALID_ARG
    # empty problems stay no-ops with the causal flag
    assert ex(A, A, A, A, A, 0, 8, 8, 4, 2, 128, 0.1, None, None, fa.FA_FLAG_CAUSAL, None) == fa.FA_OK


def test_splitkv_workspace_arithmetic(L):
    assert L.fa_splitkv_workspace_bytes(1, 64, 1, 128, 16) == 16 * 64 * 129 * 4
    assert L.fa_splitkv_workspace_bytes(2, 300, 4, 64, 3) == 3 * 2 * 4 * 300 * 65 * 4
    assert L.fa_splitkv_workspace_bytes(1, 64, 1, 96, 4) == fa.FA_ERR_INVALID_ARG
    assert L.fa_splitkv_workspace_bytes(1, 64, 1, 128, 0) == fa.FA_ERR_INVALID_ARG
    assert L.fa_splitkv_workspace_bytes(1, 64, 1, 128, 129) == fa.FA_ERR_INVALID_ARG
    # variable-length tensors are not accepted by the key-split form
    assert L.fa_splitkv_num_splits(1, 64, 4096, 1, 96, 0) == fa.FA_ERR_INVALID_ARG


def test_backward_workspace_and_argument_errors(L):
    """Backward sizes and the checks made before any device work."""
    rows = 2 * 3 * 128  # B * H * Nq rounded up to 128-query blocks (100 -> 128)
    assert fa.bwd_workspace_bytes(2, 100, 3, 128) == rows * (128 + 2) * 4
    assert fa.bwd_workspace_bytes(2, 100, 3, 64) == rows * (64 + 2) * 4
    assert fa.bwd_workspace_bytes(1, 0, 1, 128) == 0
    with pytest.raises(fa.FaError) as e:
        fa.bwd_workspace_bytes(1, 64, 1, 32)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    with pytest.raises(fa.FaError):
        fa.bwd_workspace_bytes(-1, 64, 1, 128)
    args = dict(q=16, k=16, v=16, o=16, dout=16, lse=16, dq=16, dk=16, dv=16, B=1, Nq=64, Nk=64, H=1,
                Hk=1, d=128, scale=0.1, flags=0, workspace=16, workspace_bytes=1 << 20, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return fa.fa_bwd(*a.values())

    assert call(d=32) == fa.FA_ERR_UNSUPPORTED
    assert call(flags=4) == fa.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert call(scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert call(H=3, Hk=2) == fa.FA_ERR_INVALID_ARG
    assert call(B=-1) == fa.FA_ERR_INVALID_ARG
    assert call(B=0) == fa.FA_OK   # nothing to do
    assert call(Nk=0) == fa.FA_ERR_INVALID_ARG  # queries without keys, as in the forward
    assert call(Nk=0, Nq=0) == fa.FA_OK


def test_fp8_sizes_and_varlen_argument_errors(L):
    """FP8 buffer sizes (dense and packed) and the checks made before any device work."""
    assert fa.fp8_sizes(2, 200, 130, 4, 2, 128) == (2 * 200 * 4 * 128, 2 * 130 * 2 * 128, 2 * 2 * 128 * 144,
                                                    2 * 4 * 2, 2 * 2 * 2, 2 * 2)
    # Packed: V^T columns = 16 * ceil(total_k / 16) + 16 * B.
    assert fa.fp8_varlen_sizes(3, 500, 333, 300, 200, 4, 2, 128) == (
        500 * 4 * 128, 333 * 2 * 128, 2 * 128 * (336 + 48), 3 * 4 * 3, 3 * 2 * 2, 3 * 2)
    assert fa.fp8_varlen_sizes(2, 0, 0, 0, 0, 1, 1, 128) == (0, 0, 128 * 32, 0, 0, 2)
    for bad in ((1, 10, 10, 10, 10, 1, 1, 64), (1, -1, 10, 10, 10, 1, 1, 128), (1, 10, 10, 10, 10, 3, 2, 128),
                (1, 1 << 24, 10, 10, 10, 256, 1, 128)):
        with pytest.raises(fa.FaError):
            fa.fp8_varlen_sizes(*bad)
    args = dict(q8=A, k8=A, vt8=A, qs=A, ks=A, vs=A, o=A, lse=A, cu_q=A, cu_k=A, B=1, tq=64, tk=64, mq=64,
                mk=64, H=1, Hk=1, d=128, scale=0.1, flags=0, stream=None)

    def call(**kw):
        return fa.fa_fwd_fp8_varlen(*dict(args, **kw).values())

    assert call(d=64) == fa.FA_ERR_UNSUPPORTED
    assert call(cu_q=None) == fa.FA_ERR_INVALID_ARG
    assert call(flags=2) == fa.FA_ERR_INVALID_ARG
    assert call(tq=-1) == fa.FA_ERR_INVALID_ARG
    assert call(qs=A + 2) == fa.FA_ERR_ALIGN
    assert call(q8=MIS) == fa.FA_ERR_ALIGN
    assert call(cu_k=A + 2) == fa.FA_ERR_ALIGN
    assert call(B=0) == fa.FA_OK
    qargs = dict(q=A, k=A, v=A, cu_q=A, cu_k=A, B=1, tq=64, tk=64, mq=64, mk=64, H=1, Hk=1, d=128, q8=A, k8=A,
                 vt8=A, qs=A, ks=A, vs=A, stream=None)

    def qcall(**kw):
        return fa.fa_quantize_fp8_varlen(*dict(qargs, **kw).values())

    assert qcall(d=64) == fa.FA_ERR_UNSUPPORTED
    assert qcall(cu_k=None) == fa.FA_ERR_INVALID_ARG
    assert qcall(vt8=MIS) == fa.FA_ERR_ALIGN
    assert qcall(cu_q=A + 1) == fa.FA_ERR_ALIGN
    assert qcall(B=0) == fa.FA_OK


def test_fp8_varlen_column_ranges_fit(L):
    """The packed V^T layout: sequence b starts at c(b) = 16 ceil(cu[b] / 16) + 16 b, a multiple
    of 16; its keys rounded up to 16 end at or before c(b + 1); c(B) is the column count."""
    import numpy as np
    rng = np.random.default_rng(11)
    for _ in range(200):
        B = int(rng.integers(1, 40))
        lens = rng.integers(0, 300, size=B) * (rng.random(B) < 0.9)
        cu = np.concatenate([[0], np.cumsum(lens)])
        c = [(int(cu[b]) + 15) // 16 * 16 + 16 * b for b in range(B + 1)]
        kp = fa.fp8_varlen_sizes(B, 1, int(cu[-1]), 1, int(lens.max()), 1, 1, 128)[2] // 128
        assert kp == c[B]
        for b in range(B):
            assert c[b] % 16 == 0
            assert c[b] + (int(lens[b]) + 15) // 16 * 16 <= c[b + 1]


def test_phase_buffer_entry_without_a_device(L):
    """The default library refuses the phase-clock buffer; the instrumented one
    checks its arguments on the host (too small or misaligned buffers) and
    detaches with a null buffer, all without touching a device."""
    assert L.fa_set_phase_buffer(None, 0) == fa.FA_ERR_UNSUPPORTED
    fabuild.build(phase=True)
    P = fa.load_library(fa.PHASE_LIB_PATH)
    words = P.fa_set_phase_buffer(None, 0)
    assert words == 48  # per-CTA words (kPhaseWords of the kernel source)
    assert P.fa_set_phase_buffer(8, 47) == fa.FA_ERR_INVALID_ARG   # fewer words than one CTA's record
    assert P.fa_set_phase_buffer(12, 4096) == fa.FA_ERR_INVALID_ARG  # not 8-byte aligned
    assert P.fa_set_phase_buffer(None, 0) == words

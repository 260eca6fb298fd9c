"""Host side of the instrumented build's event trace (no GPU): the event
indices and trace shape `bench.py --phase` reads match the kernel source, and
its summary of a synthetic trace gives back the intervals built into it."""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

KERNEL = os.path.join(ROOT, "attention_forward_fa2_gb300", "csrc", "fa_fwd_kernel.cuh")


def _snake(name):
    name = re.sub(r"([A-Z]+)([A-Z][a-z])", r"\1_\2", name)
    return re.sub(r"([a-z0-9])([A-Z])", r"\1_\2", name).lower()


def _kernel_source():
    with open(KERNEL) as f:
        return f.read()


def test_trace_events_and_shape_match_the_kernel():
    src = _kernel_source()
    body = re.search(r"enum TraceEvent : int \{(.*?)\};", src, re.S).group(1)
    events = {_snake(n): int(v) for n, v in re.findall(r"kTr(\w+)\s*=\s*(\d+)", body)}
    assert events == bench.TRACE_EVENTS
    consts = {n: int(v) for n, v in re.findall(r"constexpr int kTrace(Units|Steps|Events) = (\d+);", src)}
    assert (consts["Units"], consts["Steps"], consts["Events"]) == bench.TRACE_SHAPE
    assert max(events.values()) + 1 <= consts["Events"]


def test_phase_slots_match_the_kernel():
    src = _kernel_source()
    body = re.search(r"enum PhaseBase : int \{(.*?)\};", src, re.S).group(1)
    bases = {n: int(v) for n, v in re.findall(r"kPh(\w+)\s*=\s*(\d+)", body)}
    want = {"Mma": "mma", "Load": "load", "Soft0": "softmax_tile0", "Soft1": "softmax_tile1", "Epi": "epilogue"}
    for k, role in want.items():
        assert bench.PHASE_NAMES[role][0] == bases[k]
    words = int(re.search(r"constexpr int kPhaseWords = (\d+);", src).group(1))
    assert words == 48 and bases["Timer"] + 2 <= words


def _synthetic(nkv=8):
    """Unit 0 and unit 1 of nkv key steps each on a 1000-cycle step clock.
    Per step j (both units): K/V seen at +10, tile 0's P V issued at +60, S0
    issued at +100, S0 seen by the softmax at +150, S0 loaded at +200,
    exponentials done at +350, P0 published at +450; tile 1 the same 500 later.
    The MMA thread sees P(j) at step j + 1, +20 (tile 1 +520)."""
    E = bench.TRACE_EVENTS
    tr = np.zeros(bench.TRACE_SHAPE)
    for n in (0, 1):
        base = n * 20000
        for j in range(nkv + 1):
            s = base + 1000 * j
            tr[n, j, E["mma_kv"]] = s + 10
            if j >= 1:
                tr[n, j, E["mma_p0"]] = s + 20
                tr[n, j, E["mma_p0"] + 1] = s + 520
                tr[n, j, E["mma_pv0"]] = s + 60
                tr[n, j, E["mma_pv0"] + 1] = s + 560
            if j < nkv:
                for t in (0, 1):
                    o = 500 * t
                    tr[n, j, E["mma_s0"] + t] = s + 100 + o
                    tr[n, j, E["soft_s0"] + t] = s + 150 + o
                    tr[n, j, E["soft_p0"] + t] = s + 450 + o
                tr[n, j, E["soft_load0"]] = s + 200
                tr[n, j, E["soft_exp0"]] = s + 350
    # Unit 0's epilogue and the loads and waits around the boundary.
    t0 = 1000 * nkv + 60
    tr[0, 0, E["epi_o0"]] = t0 + 300
    tr[0, 1, E["epi_o0"]] = t0 + 1300
    tr[0, 2, E["epi_o0"]] = t0 + 500
    tr[0, nkv - 1, E["mma_q_empty"]] = t0 - 1700
    tr[1, 0, E["load_q"]] = t0 - 1200
    tr[1, 0, E["mma_q"]] = 20000 - 200
    return tr, t0


def test_trace_summary_recovers_the_intervals():
    tr, t0 = _synthetic()
    r = bench.trace_summary(tr)
    assert r["tile0_S_issued_to_softmax_sees_S"] == 50 and r["tile1_S_issued_to_softmax_sees_S"] == 50
    assert r["tile0_softmax_S_to_P_published"] == 300 and r["tile1_softmax_S_to_P_published"] == 300
    assert r["tile0_P_published_to_mma_sees_P"] == 1000 + 20 - 450
    assert r["tile1_P_published_to_mma_sees_P"] == 1000 + 520 - 950
    assert r["tile0_cycle"] == 1000 and r["tile1_cycle"] == 1000
    assert r["tile0_softmax_load"] == 50 and r["tile0_softmax_exp"] == 150
    assert r["mma_pv0_issue"] == 40 and r["mma_s0_issue_after_pv0"] == 40
    b = r["boundary_0_1"]
    assert b["epi_tile0_O_final_seen"] == 300 and b["epi_tile0_O_read"] == 1300
    assert b["epi_tile0_staging_free"] == 500
    assert b["mma_Q_empty_committed"] == -1700 and b["load_next_Q_issued"] == -1200
    assert b["mma_next_Q_seen"] == 20000 - 200 - t0
    assert b["mma_next_kv0"] == 20010 - t0 and b["mma_next_S0_issued"] == 20100 - t0
    assert b["mma_next_P0_seen"] == 21020 - t0
    assert b["epi_tile1_O_read"] is None  # not recorded in this trace
    assert "boundary_1_2" not in r  # unit 2 has no events


def test_trace_summary_of_an_empty_trace():
    r = bench.trace_summary(np.zeros(bench.TRACE_SHAPE))
    assert r["tile0_cycle"] is None and r["mma_pv0_issue"] is None
    assert not any(k.startswith("boundary") for k in r)


def test_kernel_code_hash_ignores_comments_and_layout():
    """profiles/traffic.json is keyed by the hash of the kernel's code: comments
    and layout do not change it, code does, and string literals are kept."""
    a = "int f(int x) {  // twice\n  return 2 * x; /* done */ }\n"
    b = "int f(int x)\n{\n  return 2 * x;\n}\n"
    c = "int f(int x) { return 3 * x; }"
    assert bench.code_text(a) == bench.code_text(b) != bench.code_text(c)
    assert bench.code_text('s = "a // b"; t = \'/\';') == 's = "a // b"; t = \'/\';'
    assert len(bench.kernel_source_hash()) == 16

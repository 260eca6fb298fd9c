"""Numbers the pages print for a worked example, checked against the FLOP and
byte accounting used by the benchmark (attention_forward_fa2_gb300.inputs)."""
import os

from attention_forward_fa2_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = (s.strip() for s in line.split("="))
                vals[key] = float(val)
    return vals


def test_slice_arithmetic():
    g = _read("slice_arithmetic.txt")
    w = I.SLICE
    assert (w.Nq, w.Nk, w.d) == (int(g["queries"]), int(g["keys"]), int(g["d_head"]))
    mm = w.flops()  # 4 * Nq * Nk * d, the two matmuls only
    assert mm == 4 * 64 * 4096 * 128
    # The page's figure is the matmul count plus about 6 elementwise softmax
    # operations per score (scale, max, subtract, exp, sum, divide); the matmul
    # count alone is 1.2 % lower.  Both readings sit within the page's rounding.
    assert abs(mm + 6 * w.Nq * w.Nk - g["flops"]) < 0.05e6
    assert abs(mm - g["flops"]) / g["flops"] < 0.013
    # Bytes: Q, K, V read and O written once, bf16 (LSE adds 256 bytes).
    assert abs(w.hbm_bytes() - g["bytes"]) < 0.05e6
    assert abs(g["flops"] / w.hbm_bytes() - g["intensity"]) < 1.0

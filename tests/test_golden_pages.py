"""Numbers the pages print for a worked example, checked against the FLOP and
byte accounting used by the benchmark (attention_forward_fa2_gb300.inputs)."""
import os

import torch

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


def test_input_recipe_draws():
    """The seeded workloads are what the design notes state: the packed batch's
    32 lengths from default_rng(4) (81,588 tokens), the sweep seeds, the shapes."""
    w = I.VARLEN
    assert len(w.lengths) == 32 and sum(w.lengths) == 81588
    assert min(w.lengths) >= 128 and max(w.lengths) <= 4096
    assert w.lengths == I.varlen_lengths(4)
    assert (I.PAGE.B, I.PAGE.Nq, I.PAGE.H, I.PAGE.d, I.PAGE.seed) == (16, 4096, 16, 128, 2)
    seeds = {s.name: s.seed for s in I.SWEEP}
    assert seeds["sweep_d64_n512"] == 100 and seeds["sweep_d128_n8192"] == 114
    q, k, v = I.make_dense(1, 3, 3, 1, 4, seed=7)
    q2, _, _ = I.make_dense(1, 3, 3, 1, 4, seed=7)
    assert q.dtype == torch.bfloat16 and torch.equal(q, q2)  # deterministic per seed

"""Pins against figures the pages print.

The pages print no worked example of the block arithmetic (their numbers are
timings and memory sizes), so the stored fixtures here are those sizes: the
176B-layer shape the benchmarks use (hidden 14336, 112 heads, MLP 57344,
vocabulary 250880), stacked to BLOOM-176B's 70 layers, must have the printed
parameter count and bf16 footprint.
"""
import os

from bloom_decoder_token_gb300 import synth

HERE = os.path.dirname(__file__)


def load(name):
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def bloom_params(sh: synth.Shape, n_layer: int) -> int:
    """Parameters of a BLOOM stack: tied embedding + embedding LN, per layer
    LN1, fused QKV (+bias), dense (+bias), LN2, up (+bias), down (+bias), and ln_f."""
    h, F, V = sh.hidden, sh.ffn, sh.vocab
    per_layer = 2 * h + (3 * h * h + 3 * h) + (h * h + h) + 2 * h + (F * h + F) + (h * F + h)
    return V * h + 2 * h + n_layer * per_layer + 2 * h


def test_176b_shape_matches_printed_size():
    g = load("bloom176b_size.txt")
    sh = synth.PRESETS["176b14"]
    p = bloom_params(sh, 70)
    assert round(p / 1e9) == g["params_billion"]
    assert round(2 * p / 1e9) == g["bf16_gigabytes"]

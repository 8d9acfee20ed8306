"""The oracle against its pins (CPU only)."""

import json
import os

import numpy as np
import pytest

import inputs
import oracle_pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_brute_fp16_rounding_matches_numpy():
    """The brute force's exact-rational fp16 rounding agrees with numpy on
    doubles (which are exact rationals), ties and overflow included."""
    from fractions import Fraction
    from oracle import brute
    rng = np.random.default_rng(11)
    vals = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-8, 5, 3000))
    vals += [65504.0, 65520.0, 65519.0, 2.0 ** -24, 2.0 ** -25, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11]
    for v in vals:
        with np.errstate(over="ignore"):
            want = int(np.array([v]).astype(np.float16).view(np.uint16)[0])
        assert brute.fraction_to_half_bits(Fraction(v)) == want, v


def test_golden_threshold_default():
    g = json.load(open(os.path.join(GOLDEN, "pages_claims.json")))
    assert inputs.TAU_DEFAULT == g["llm_int8_threshold_default"]["value"]


def test_golden_weight_memory(orc):
    """int8 codes + one fp32 scale per output channel: N*K + 4N bytes, about
    half of fp16's 2*N*K and a quarter of fp32's 4*N*K, as the pages state."""
    g = json.load(open(os.path.join(GOLDEN, "pages_claims.json")))
    W = (np.random.default_rng(0).standard_normal((64, 4096)) * 0.02).astype(np.float16)
    Wq, sw = orc.quantize_weight(W)
    int8_bytes = Wq.nbytes + sw.nbytes
    assert int8_bytes == 64 * 4096 + 4 * 64
    assert abs(int8_bytes / W.nbytes - g["int8_weight_memory_vs_fp16"]["value"]) < 1e-3
    assert abs(Wq.nbytes / (4 * W.size) - g["int8_weight_memory_vs_fp32"]["value"]) < 1e-12
    p = g["fp16_bytes_70b_model_GB"]
    assert 2 * p["params"] / 1e9 == p["value"]


def test_sampled_rows_match_full(orc):
    """The sampled-row mode (used at full size) equals the full computation
    restricted to those rows."""
    w = inputs.random_small(20, 96, 33, n_cols=3, seed=12)
    Wq, sw = orc.quantize_weight(w.W)
    full = orc.linear(w.X, Wq, sw, w.W, w.tau)
    rows = np.array([0, 7, 19, 3])
    part = orc.linear(w.X, Wq, sw, w.W, w.tau, rows=rows)
    assert np.array_equal(part["acc"], full["acc"][rows])
    assert np.array_equal(part["Y"].view(np.uint16), full["Y"][rows].view(np.uint16))
    assert np.array_equal(part["O"], full["O"])

"""Pins of the oracle to things other than itself.

Each ``pin_*`` function takes an :class:`oracle.Oracle` and raises
``AssertionError`` when the oracle disagrees with what the pages, the
mathematics or an independent routine fix.  ``tests/test_oracle.py`` runs them
on the real oracle; ``tests/test_oracle_mutations.py`` runs them on copies of
the oracle with a planted mistake and checks that some pin fails.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import inputs
from oracle import brute


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float16).view(np.uint16)


def _rows(a):
    return _bits(a).tolist()


# ---------------------------------------------------------------------------
# fp16 conversions against numpy's independent implementation
# ---------------------------------------------------------------------------

def pin_half_roundtrip(orc):
    """fp16 -> double decodes every finite bit pattern like numpy does, and
    double -> fp16 rounds like numpy (nearest even, direct from double)."""
    allbits = np.arange(65536, dtype=np.uint16)
    vals = allbits.view(np.float16).astype(np.float64)
    finite = np.isfinite(vals)
    for b in allbits[finite][::7]:
        assert orc.half_to_double(int(b)) == float(allbits[b:b + 1].view(np.float16)[0])
    rng = np.random.default_rng(1)
    cands = np.concatenate([
        rng.standard_normal(2000) * 10.0 ** rng.integers(-9, 5, 2000),
        # exact midpoints between neighbouring fp16 values: ties
        (vals[finite][1:400:3] + np.nextafter(vals[finite][1:400:3].astype(np.float16),
                                              np.float16(np.inf)).astype(np.float64)) / 2,
        np.array([65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  0.0, -0.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11]),
    ])
    for v in cands:
        with np.errstate(over="ignore"):
            want = int(np.array([v], np.float64).astype(np.float16).view(np.uint16)[0])
        got = orc.double_to_half(float(v))
        assert got == want, (v, hex(got), hex(want))


# ---------------------------------------------------------------------------
# the fp32 code rule against exact rational rounding, exhaustively per scale
# ---------------------------------------------------------------------------

def _exact_codes(x16: np.ndarray, a16: np.ndarray) -> np.ndarray:
    """round_half_even(127*x/a) in exact integer arithmetic (vectorised).

    x = mx * 2^ex and a = ma * 2^ea with integer significands, so
    127*x/a = 127*mx*2^(ex-ea) / ma; scale both to integers and round."""
    def split(v):
        m, e = np.frexp(v.astype(np.float64))       # v = m * 2^e, m in [0.5,1)
        mi = np.rint(m * 2048).astype(np.int64)      # 11-bit significand
        return mi, e.astype(np.int64) - 11
    mx, ex = split(x16)
    ma, ea = split(a16)
    sh = ex - ea
    num = 127 * mx
    den = ma.copy()
    pos = sh >= 0
    num = np.where(pos, num << np.where(pos, sh, 0), num)
    den = np.where(~pos, den << np.where(~pos, -sh, 0), den)
    sign = np.sign(num)
    num = np.abs(num)
    q, r = np.divmod(num, den)
    twice = 2 * r
    up = (twice > den) | ((twice == den) & (q % 2 == 1))
    return (sign * (q + up)).astype(np.int64)


def pin_code_rule_exhaustive(orc, n_scales: int = 48):
    """For a spread of absmax values a (including the ones that produce exact
    ties, a = 127 * 2^s), every fp16 x with |x| <= a is coded like the exactly
    rounded rational round_half_even(127 x / a)."""
    allv = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)  # all finite >= 0
    rng = np.random.default_rng(2)
    scales = list(np.float16(127) * np.float16(2.0) ** np.arange(-8, 8, 2).astype(np.float16))
    scales += list(allv[rng.integers(1, len(allv), n_scales)])
    scales += [np.float16(1.0), np.float16(6.0), np.float16(65504.0), allv[1], allv[1023]]
    for a in scales:
        a = np.float16(a)
        if not a > 0:
            continue
        xs = allv[allv <= a]
        xs = np.concatenate([xs, -xs[1:]])
        # rows of the weight: each row holds a first, so its absmax is a
        step = 4095
        for s in range(0, len(xs), step):
            chunk = xs[s:s + step]
            W = np.empty((1, len(chunk) + 1), np.float16)
            W[0, 0] = a
            W[0, 1:] = chunk
            Wq, sw = orc.quantize_weight(W)
            assert sw[0] == np.float32(a)
            want = _exact_codes(chunk, np.full(len(chunk), a))
            got = Wq[0, 1:].astype(np.int64)
            bad = np.flatnonzero(got != want)
            assert len(bad) == 0, (float(a), chunk[bad[:3]], got[bad[:3]], want[bad[:3]])


# ---------------------------------------------------------------------------
# whole layer against the exact brute force
# ---------------------------------------------------------------------------

def _compare_with_brute(orc, X, W, tau, bias=None):
    Wq, sw = orc.quantize_weight(W)
    r = orc.linear(X, Wq, sw, W, tau, bias=bias)
    b = brute.linear(_rows(X), _rows(W), tau,
                     None if bias is None else _bits(np.asarray(bias, np.float16)).tolist())
    assert r["O"].tolist() == b["O"], (r["O"], b["O"])
    assert np.array_equal(Wq, np.array(b["Wq"], np.int8).reshape(Wq.shape))
    assert np.array_equal(sw.astype(np.float64), np.array([float(v) for v in b["sw"]]))
    assert np.array_equal(r["sx"].astype(np.float64), np.array([float(v) for v in b["sx"]]))
    assert np.array_equal(r["Xq"], np.array(b["Xq"], np.int8).reshape(r["Xq"].shape))
    assert np.array_equal(r["acc"].astype(np.int64), np.array(b["acc"], np.int64).reshape(r["acc"].shape))
    yb = np.array(b["Y"], np.uint16).reshape(r["Y"].shape)
    yo = r["Y"].view(np.uint16)
    bad = np.argwhere(yb != yo)
    assert len(bad) == 0, (bad[:3], yo[tuple(bad[0])], yb[tuple(bad[0])])


def pin_brute_tiny_config(orc):
    """The tiny workload (T16 K256 N256, columns 7 and 133 x20, tau 6)."""
    w = inputs.tiny()
    _compare_with_brute(orc, w.X, w.W, w.tau)


def pin_brute_random_small(orc):
    """Random tiny shapes and thresholds, with edge rows: an all-zero row, a
    row of only outliers, columns exactly at tau, |O| = 0 and |O| = K."""
    rng = np.random.default_rng(3)
    for i, (T, K, N) in enumerate([(1, 1, 1), (3, 5, 2), (7, 16, 9), (16, 32, 8),
                                   (5, 24, 17), (2, 48, 3), (32, 8, 32)]):
        X = (rng.standard_normal((T, K)) * 3).astype(np.float16)
        W = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
        if T > 2:
            X[1] = 0                    # an all-zero row
            X[2] = 7.5                  # a row whose every column is an outlier
        if K > 3:
            X[0, 3] = -6.0              # exactly at the threshold: an outlier (>=)
        for tau in (6.0, 1.5, 0.0, math.inf, 2.0 ** 0.5):
            _compare_with_brute(orc, X, W, tau)


def pin_bias_brute(orc):
    """An fp16 bias per output channel (the layer stands in for PyTorch's
    Linear, whose bias is added to x W^T) is added before the one rounding to
    fp16: against the exact brute force, with biases that dominate the sum,
    cancel it and sit far below its last bit."""
    rng = np.random.default_rng(11)
    for T, K, N in ((1, 1, 1), (3, 5, 4), (7, 16, 9), (4, 40, 13)):
        X = (rng.standard_normal((T, K)) * 3).astype(np.float16)
        W = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
        bias = (rng.standard_normal(N) * rng.choice([1e-4, 0.5, 300.0], N)).astype(np.float16)
        for tau in (6.0, 1.5, math.inf):
            _compare_with_brute(orc, X, W, tau, bias)


def pin_bias_integer(orc):
    """tau = inf, integer inputs with +-127 in every row and an integer bias:
    Y = fp16(X W^T + b) exactly; a zero bias gives the unbiased layer's
    values."""
    X, W = inputs.int_valued(8, 4, 24, seed=12, adversarial=True)
    bias = np.arange(-12, 12, dtype=np.float64) * 37
    Wq, sw = orc.quantize_weight(W)
    r = orc.linear(X, Wq, sw, W, math.inf, bias=bias.astype(np.float16))
    exact = X.astype(np.int64) @ W.astype(np.int64).T + bias.astype(np.int64)[None, :]
    assert np.array_equal(r["Y"].view(np.uint16), exact.astype(np.float64).astype(np.float16).view(np.uint16))
    r0 = orc.linear(X, Wq, sw, W, math.inf, bias=np.zeros(24, np.float16))
    r1 = orc.linear(X, Wq, sw, W, math.inf)
    assert np.array_equal(r0["Y"].astype(np.float64), r1["Y"].astype(np.float64))


def pin_w16_free_brute(orc):
    """Only the int8 weight kept: the outlier weights are the codes
    dequantized, Wq sw / 127.  Against the exact brute force on random tiny
    shapes and thresholds (with a bias, and with an all-zero weight row)."""
    rng = np.random.default_rng(13)
    for T, K, N in ((1, 1, 1), (3, 5, 4), (7, 16, 9), (5, 24, 6)):
        X = (rng.standard_normal((T, K)) * 3).astype(np.float16)
        W = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
        if N > 3:
            W[2] = 0
        bias = (rng.standard_normal(N) * 0.3).astype(np.float16)
        for tau in (6.0, 1.5, 0.0, math.inf):
            for b in (None, bias):
                Wq, sw = orc.quantize_weight(W)
                r = orc.linear(X, Wq, sw, None, tau, bias=b)
                bb = brute.linear(_rows(X), _rows(W), tau,
                                  None if b is None else _bits(b).tolist(), w16_free=True)
                yb = np.array(bb["Y"], np.uint16).reshape(r["Y"].shape)
                assert r["O"].tolist() == bb["O"]
                assert np.array_equal(r["Y"].view(np.uint16), yb), (T, K, N, tau)


def pin_w16_free_invariants(orc):
    """Where the dequantized codes equal the weights -- integer weights with
    +-127 in every row, so sw = 127 and Wq = W -- the int8-weight-only layer
    gives the fp16-weight layer's Y bit for bit at every threshold; with no
    outliers (tau = inf) it does so for any weight."""
    rng = np.random.default_rng(14)
    _, W = inputs.int_valued(4, 64, 24, seed=15)
    X = (rng.standard_normal((9, 64)) * 4).astype(np.float16)
    Wq, sw = orc.quantize_weight(W)
    assert np.all(sw == 127) and np.array_equal(Wq, W.astype(np.int8))
    for tau in (6.0, 3.0, 0.0):
        a = orc.linear(X, Wq, sw, W, tau)["Y"]
        b = orc.linear(X, Wq, sw, None, tau)["Y"]
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16)), tau
    W2 = (rng.standard_normal((24, 64)) * 0.05).astype(np.float16)
    Wq2, sw2 = orc.quantize_weight(W2)
    a = orc.linear(X, Wq2, sw2, W2, math.inf)["Y"]
    b = orc.linear(X, Wq2, sw2, None, math.inf)["Y"]
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


# ---------------------------------------------------------------------------
# bfloat16 inputs and output (the compute dtype)
# ---------------------------------------------------------------------------

def _f32_to_bf16_bits(x) -> np.ndarray:
    """float32 values -> bfloat16 bit patterns, nearest-even (torch's own
    conversion, independent of the oracle)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _bf16_bits_to_f64(b) -> np.ndarray:
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_bf16_roundtrip(orc):
    """bf16 -> double decodes every finite bit pattern like the binary32 with
    the same leading bits; double -> bf16 rounds like torch for values exact
    in fp32 (ties, subnormals, the overflow boundary included) and like the
    exact-rational rounding of the brute force for values that are not."""
    allbits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        vals = (allbits << 16).view(np.float32).astype(np.float64)
    finite = np.isfinite(vals)
    for b in allbits[finite][::5]:
        assert orc.bf16_to_double(int(b)) == vals[b]
    rng = np.random.default_rng(31)
    fin = vals[finite & (vals > 0)]
    f32 = np.concatenate([
        (rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000)).astype(np.float32),
        # exact midpoints of neighbouring bf16 values (exact in fp32): ties
        ((fin[:-1:97] + fin[1::97]) / 2).astype(np.float32),
        np.array([3.3895314e38, 3.3961775e38, 3.4028235e38, 2.0 ** -133, 2.0 ** -134,
                  3 * 2.0 ** -135, 2.0 ** -126, 0.0, -0.0, 1.0 + 2.0 ** -8,
                  1.0 + 3 * 2.0 ** -8], np.float32),
    ])
    f32 = f32[np.isfinite(f32)]
    want = _f32_to_bf16_bits(f32)
    for v, w in zip(f32.tolist(), want.tolist()):
        got = orc.double_to_bf16(float(v))
        assert got == w, (v, hex(got), hex(w))
    for v in (rng.standard_normal(400) * 10.0 ** rng.integers(-40, 38, 400)).tolist():
        got = orc.double_to_bf16(v)
        want = brute.fraction_to_bf16_bits(Fraction(v))
        assert got == want, (v, hex(got), hex(want))


def _exact_codes_bf16(x: np.ndarray, a: float) -> np.ndarray:
    """round_half_even(127 x / a) exactly, for bf16 values x, a (|x| <= a)."""
    def split(v):
        m, e = np.frexp(np.asarray(v, np.float64))
        return np.rint(m * 256).astype(np.int64), e.astype(np.int64) - 8  # 8-bit significand
    mx, ex = split(x)
    ma, ea = split(np.full(len(x), a))
    sh = ea - ex                                 # >= -1 since |x| <= a
    num = 127 * mx
    den = ma << np.clip(sh, 0, 40)               # past 2^40 the code is 0 either way
    num = np.where(sh < 0, num << np.clip(-sh, 0, 1), num)
    sign = np.sign(num)
    q, r = np.divmod(np.abs(num), den)
    up = (2 * r > den) | ((2 * r == den) & (q % 2 == 1))
    return (sign * (q + up)).astype(np.int64)


def pin_bf16_code_rule_exhaustive(orc, n_scales: int = 24):
    """The fp32 code rule on bf16 inputs: for a spread of bf16 absmax values
    (exact-tie scales 127 * 2^s, subnormal and huge ones), every bf16 x with
    |x| <= a is coded like round_half_even(127 x / a)."""
    pos = np.arange(0, 0x7F80, dtype=np.uint16)       # all finite >= 0
    posv = _bf16_bits_to_f64(pos)
    rng = np.random.default_rng(32)
    scales = [int(b) for b in _f32_to_bf16_bits(127 * 2.0 ** np.arange(-8, 8, 2))]
    scales += [int(b) for b in pos[rng.integers(1, len(pos), n_scales)]]
    scales += [0x0001, 0x007F, 0x0080, 0x3F80, 0x40C0, 0x7F7F]
    for ab in scales:
        a = float(_bf16_bits_to_f64([ab])[0])
        keep = posv <= a
        xb = np.concatenate([pos[keep], pos[keep][1:] | 0x8000])
        xv = _bf16_bits_to_f64(xb)
        step = 8191
        for s0 in range(0, len(xb), step):
            chunk = xb[s0:s0 + step]
            W = np.empty((1, len(chunk) + 1), np.uint16)
            W[0, 0] = ab
            W[0, 1:] = chunk
            Wq, sw = orc.quantize_weight(W, fmt="bf16")
            assert float(sw[0]) == a
            want = _exact_codes_bf16(xv[s0:s0 + step], a)
            got = Wq[0, 1:].astype(np.int64)
            bad = np.flatnonzero(got != want)
            assert len(bad) == 0, (a, xv[s0 + bad[:3]], got[bad[:3]], want[bad[:3]])


def pin_bf16_brute(orc):
    """The whole layer on bf16 bit patterns against the exact brute force:
    random tiny shapes and thresholds, with a bias, and with only the int8
    weight kept."""
    rng = np.random.default_rng(33)
    for T, K, N in ((1, 1, 1), (3, 5, 4), (7, 16, 9), (4, 24, 6)):
        X = _f32_to_bf16_bits(rng.standard_normal((T, K)) * 3)
        W = _f32_to_bf16_bits(rng.standard_normal((N, K)) * 0.05)
        bias = _f32_to_bf16_bits(rng.standard_normal(N) * 0.3)
        if T > 2:
            X[1] = 0
        for tau in (6.0, 1.5, 0.0, math.inf):
            for b, free in ((None, False), (bias, False), (bias, True)):
                Wq, sw = orc.quantize_weight(W, fmt="bf16")
                r = orc.linear(X, Wq, sw, None if free else W, tau, bias=b, fmt="bf16")
                bb = brute.linear(X.tolist(), W.tolist(), tau, None if b is None else b.tolist(),
                                  w16_free=free, fmt="bf16")
                assert r["O"].tolist() == bb["O"]
                assert np.array_equal(Wq, np.array(bb["Wq"], np.int8).reshape(Wq.shape))
                assert np.array_equal(r["acc"].astype(np.int64),
                                      np.array(bb["acc"], np.int64).reshape(r["acc"].shape))
                yb = np.array(bb["Y"], np.uint16).reshape(r["Y"].shape)
                assert np.array_equal(r["Y"], yb), (T, K, N, tau, free)


def pin_bf16_tau_inf_integer(orc):
    """tau = inf, integer bf16 inputs with +-127 in every row: the codes are
    the inputs and Y = bf16(X W^T), the exact integer product rounded once
    (torch's float32 -> bf16 rounding of a value exact in fp32)."""
    for adv, K in ((False, 256), (True, 256), (True, 16)):
        X16, W16 = inputs.int_valued(8, K, 24, seed=34, adversarial=adv)
        X = _f32_to_bf16_bits(X16.astype(np.float32))
        W = _f32_to_bf16_bits(W16.astype(np.float32))
        Wq, sw = orc.quantize_weight(W, fmt="bf16")
        r = orc.linear(X, Wq, sw, W, math.inf, fmt="bf16")
        assert np.all(sw == 127) and np.array_equal(Wq, W16.astype(np.int8))
        exact = X16.astype(np.int64) @ W16.astype(np.int64).T
        assert np.array_equal(r["Y"], _f32_to_bf16_bits(exact.astype(np.float32)))


# ---------------------------------------------------------------------------
# invariants of the method
# ---------------------------------------------------------------------------

def pin_tau_inf_integer_inputs(orc):
    """tau = inf, integer-valued inputs with +-127 in every row: scales are 127,
    codes equal the inputs, acc is the exact integer product, and
    Y = fp16(X W^T) exactly (127/127 = 1; at K = 4 every |acc| <= 4*127^2
    stays inside fp16's range, at K = 256 large values overflow to inf on
    both sides)."""
    for adv, K in ((False, 256), (True, 256), (False, 4), (True, 4)):
        X, W = inputs.int_valued(8, K, 24, seed=4, adversarial=adv)
        Wq, sw = orc.quantize_weight(W)
        r = orc.linear(X, Wq, sw, W, math.inf)
        assert len(r["O"]) == 0
        assert np.all(sw == 127) and np.all(r["sx"] == 127)
        assert np.array_equal(Wq, W.astype(np.int8)) and np.array_equal(r["Xq"], X.astype(np.int8))
        exact = X.astype(np.int64) @ W.astype(np.int64).T       # library integer matmul
        assert np.array_equal(r["acc"].astype(np.int64), exact)
        with np.errstate(over="ignore"):
            ref = exact.astype(np.float64).astype(np.float16)
        assert np.array_equal(r["Y"].view(np.uint16), ref.view(np.uint16))


def pin_tau_zero_is_fp16_matmul(orc):
    """tau = 0: every column (zero columns included) is an outlier, so the int8
    part vanishes and Y is the fp16 matmul X W^T rounded once."""
    rng = np.random.default_rng(5)
    X = rng.standard_normal((6, 40)).astype(np.float16)
    X[:, 11] = 0  # a zero column still counts: |0| >= 0
    W = (rng.standard_normal((10, 40)) * 0.1).astype(np.float16)
    Wq, sw = orc.quantize_weight(W)
    r = orc.linear(X, Wq, sw, W, 0.0)
    assert r["O"].tolist() == list(range(40))
    assert np.all(r["sx"] == 0) and not r["Xq"].any() and not r["acc"].any()
    ref = (X.astype(np.float64) @ W.astype(np.float64).T).astype(np.float16)
    assert np.array_equal(r["Y"].view(np.uint16), ref.view(np.uint16))


def pin_outliers_are_column_scan(orc):
    """The outlier set equals a direct numpy column scan of |X| >= tau."""
    w = inputs.random_small(12, 300, 4, n_cols=5, seed=6)
    for tau in (6.0, 3.0, 20.0, 0.0):
        want = np.flatnonzero((np.abs(w.X.astype(np.float32)) >= np.float32(tau)).any(axis=0))
        assert orc.outlier_columns(w.X, tau).tolist() == want.tolist()
    tiny = inputs.tiny()
    O = orc.outlier_columns(tiny.X, tiny.tau).tolist()
    assert 7 in O and 133 in O


def pin_permutation_invariance(orc):
    """Permuting the K columns of X and W jointly permutes O and leaves acc
    and Y bit-identical."""
    w = inputs.random_small(9, 64, 12, n_cols=3, seed=7)
    Wq, sw = orc.quantize_weight(w.W)
    r = orc.linear(w.X, Wq, sw, w.W, w.tau)
    perm = np.random.default_rng(8).permutation(64)
    Xp, Wp = w.X[:, perm], w.W[:, perm]
    Wqp, swp = orc.quantize_weight(Wp)
    rp = orc.linear(Xp, Wqp, swp, Wp, w.tau)
    assert sorted(perm[rp["O"]].tolist()) == r["O"].tolist()
    assert np.array_equal(r["acc"], rp["acc"])
    assert np.array_equal(r["Y"].view(np.uint16), rp["Y"].view(np.uint16))


def pin_code_extremes(orc):
    """Every row's codes reach +-127 unless its scale is zero; none is -128."""
    w = inputs.random_small(10, 128, 20, n_cols=2, seed=9)
    Wq, sw = orc.quantize_weight(w.W)
    r = orc.linear(w.X, Wq, sw, w.W, w.tau)
    for q, s in list(zip(r["Xq"], r["sx"])) + list(zip(Wq, sw)):
        if s == 0:
            assert not q.any()
        else:
            assert np.abs(q.astype(np.int32)).max() == 127
        assert q.min() >= -127


def pin_hand_example(orc):
    """A worked example, derived by hand from the definitions.

    X = [[1, -2, 8, 0.5], [3, 1, -1, 2]], W = [[0.5, 1, -1, 2], [-4, 2, 1, 0.25]],
    tau = 6.  Column 2 holds 8 >= 6: O = [2].
    sx = [max(1,2,0.5), max(3,1,2)] = [2, 3]; sw = [2, 4].
    Xq row 0: 127/2 = 63.5 -> 64 (tie, even), -127, 0 (outlier), 31.75 -> 32.
    Xq row 1: 127, 42.33 -> 42, 0, 84.67 -> 85.
    Wq row 0: 31.75 -> 32, 63.5 -> 64, -63.5 -> -64, 127.
    Wq row 1: -127, 63.5 -> 64, 31.75 -> 32, 7.9375 -> 8.
    acc = [[2048-8128+4064, -8128-8128+256], [4064+2688+10795, -16129+2688+680]]
        = [[-2016, -16000], [17547, -12761]].
    out = X[:,2] W[:,2]^T = [[-8, 8], [1, -1]].
    Y[0,0] = -2016*2*2/16129 - 8 = -8.49997 -> -8.5 (fp16 step 2^-7 there).
    Y[0,1] = 8 - 128000/16129 = 1032/16129 = 0.063984 -> 1048 * 2^-14.
    Y[1,0] = 105282/16129 + 1 = 7.527497 -> 1927 * 2^-8.
    Y[1,1] = -153132/16129 - 1 = -10.494203 -> -1343 * 2^-7.
    """
    X = np.array([[1, -2, 8, 0.5], [3, 1, -1, 2]], np.float16)
    W = np.array([[0.5, 1, -1, 2], [-4, 2, 1, 0.25]], np.float16)
    Wq, sw = orc.quantize_weight(W)
    r = orc.linear(X, Wq, sw, W, 6.0)
    assert r["O"].tolist() == [2]
    assert r["sx"].tolist() == [2.0, 3.0] and sw.tolist() == [2.0, 4.0]
    assert r["Xq"].tolist() == [[64, -127, 0, 32], [127, 42, 0, 85]]
    assert Wq.tolist() == [[32, 64, -64, 127], [-127, 64, 32, 8]]
    assert r["acc"].tolist() == [[-2016, -16000], [17547, -12761]]
    assert r["out"].tolist() == [[-8.0, 8.0], [1.0, -1.0]]
    want = [[-8.5, 1048 * 2.0 ** -14], [1927 * 2.0 ** -8, -1343 * 2.0 ** -7]]
    assert r["Y"].astype(np.float64).tolist() == want



# ---------------------------------------------------------------------------
# the blockwise 8-bit codec of optimizer states
# ---------------------------------------------------------------------------

def _bw_closed_form_blocks(rng, nblocks, B):
    """Blocks whose absmax is +-127 * 2^e; every other value is k * 2^e (code
    k, decodes to itself) or (k + 1/2) * 2^e (an exact tie: the even
    neighbour).  Returns values, codes and decoded values fixed by that."""
    xs, qs, ys = [], [], []
    for _ in range(nblocks):
        e = int(rng.integers(-30, 30))
        s = 2.0 ** e
        sign = 1 if rng.integers(0, 2) else -1
        k = rng.integers(-126, 127, size=B - 1)
        tie = rng.integers(0, 2, size=B - 1).astype(bool)
        vals = np.where(tie, (k + 0.5) * s, k * s)
        codes = np.where(tie, np.where(k % 2 == 0, k, k + 1), k)
        pos = int(rng.integers(0, B))
        xs.append(np.insert(vals, pos, sign * 127 * s))
        qs.append(np.insert(codes, pos, sign * 127))
        ys.append(np.insert(codes * s, pos, sign * 127 * s))
    return (np.concatenate(xs).astype(np.float32), np.concatenate(qs).astype(np.int64),
            np.concatenate(ys).astype(np.float32))


def pin_blockwise_closed_forms(orc):
    """Exact quotients give their integer code and decode to themselves;
    exact ties round to the even neighbour; the absmax has code +-127."""
    rng = np.random.default_rng(11)
    for B in (64, 256):
        x, q_want, y_want = _bw_closed_form_blocks(rng, 24, B)
        q, a = orc.quantize_blockwise(x, B)
        assert np.array_equal(q.astype(np.int64), q_want)
        assert np.array_equal(a, np.abs(x).reshape(-1, B).max(axis=1))
        y = orc.dequantize_blockwise(q, a, B)
        assert np.array_equal(y, y_want)


def pin_blockwise_error_bound(orc):
    """Random states with a different magnitude per block and a short last
    block: each block's scale is its absmax, codes stay within +-127 and reach
    it in every nonzero block, and every decoded value is within half a code
    step (a / 254) of the value, up to fp32 rounding."""
    rng = np.random.default_rng(12)
    B, n = 128, 128 * 37 + 45
    mag = 10.0 ** rng.uniform(-8, 3, size=(n + B - 1) // B)
    x = (rng.standard_normal(n) * np.repeat(mag, B)[:n]).astype(np.float32)
    q, a = orc.quantize_blockwise(x, B)
    y = orc.dequantize_blockwise(q, a, B)
    for b in range(a.size):
        xb = x[b * B:(b + 1) * B]
        assert a[b] == np.abs(xb).max()
        qb = q[b * B:(b + 1) * B].astype(np.int64)
        assert np.abs(qb).max() == 127
        err = np.abs(y[b * B:(b + 1) * B].astype(np.float64) - xb.astype(np.float64))
        assert err.max() <= float(a[b]) * (1 / 254 + 1e-6)


def pin_blockwise_locality(orc):
    """Each block carries its own scale, which limits what one outlier does to
    its neighbours (page "bitsandbytes", section "What it provides"): a value
    made 1000 times larger changes its own block's scale and codes only."""
    rng = np.random.default_rng(13)
    B = 256
    x = rng.standard_normal(B * 9).astype(np.float32)
    q0, a0 = orc.quantize_blockwise(x, B)
    x2 = x.copy()
    x2[4 * B + 17] *= 1000
    q1, a1 = orc.quantize_blockwise(x2, B)
    changed = {i // B for i in np.nonzero(q0 != q1)[0]} | set(np.nonzero(a0 != a1)[0].tolist())
    assert changed == {4}


def pin_blockwise_zero_and_scaling(orc):
    """An all-zero block has scale 0, codes 0 and decodes to 0; a block
    multiplied by 2^k keeps its codes and has its scale multiplied by 2^k."""
    rng = np.random.default_rng(14)
    B = 64
    x = rng.standard_normal(B * 6).astype(np.float32)
    x[2 * B:3 * B] = 0
    q, a = orc.quantize_blockwise(x, B)
    assert a[2] == 0 and not q[2 * B:3 * B].any()
    assert not orc.dequantize_blockwise(q, a, B)[2 * B:3 * B].any()
    for k in (-40, -3, 5, 60):
        q2, a2 = orc.quantize_blockwise(x * np.float32(2.0 ** k), B)
        assert np.array_equal(q2, q)
        assert np.array_equal(a2, a * np.float32(2.0 ** k))


def pin_blockwise_huge_scale(orc):
    """Blocks whose absmax is near the top of fp32's range, where 127 x and
    q a overflow fp32 if computed as written: the codes are still the integers
    nearest to 127 x / a (exact quotients, exact ties to the even neighbour,
    +-127 at the absmax, +-FLT_MAX included), and every decoded value is
    finite and within half a code step of x."""
    rng = np.random.default_rng(15)
    B = 64
    # closed forms at a = 127 * 2^e for e up to 120 (a up to 1.7e38)
    xs, qs, ys = [], [], []
    for e in (110, 113, 114, 115, 116, 117, 118, 119, 120):
        s = 2.0 ** e
        k = rng.integers(-126, 127, size=B - 1)
        tie = rng.integers(0, 2, size=B - 1).astype(bool)
        vals = np.where(tie, (k + 0.5) * s, k * s)
        codes = np.where(tie, np.where(k % 2 == 0, k, k + 1), k)
        pos = int(rng.integers(0, B))
        sign = 1 if e % 2 else -1
        xs.append(np.insert(vals, pos, sign * 127 * s))
        qs.append(np.insert(codes, pos, sign * 127))
        ys.append(np.insert(codes * s, pos, sign * 127 * s))
    x = np.concatenate(xs).astype(np.float32)
    q, a = orc.quantize_blockwise(x, B)
    assert np.array_equal(q.astype(np.int64), np.concatenate(qs))
    y = orc.dequantize_blockwise(q, a, B)
    assert np.array_equal(y, np.concatenate(ys).astype(np.float32))
    # a = 2^127 (a power of two): 127 x / a is exact in binary for x with few
    # significant bits, so the code is that quotient rounded half to even
    k = rng.integers(-2 ** 16, 2 ** 16, size=(2, B))
    xp = (k * 2.0 ** 111).astype(np.float32)
    xp[0, 5], xp[1, 9] = 2.0 ** 127, -(2.0 ** 127)
    q, a = orc.quantize_blockwise(xp.ravel(), B)
    assert np.array_equal(a, np.float32([2.0 ** 127, 2.0 ** 127]))
    want = [int(round(Fraction(127 * int(v), 2 ** 16))) for v in k.ravel()]
    want = np.array(want).reshape(2, B)
    want[0, 5], want[1, 9] = 127, -127
    assert np.array_equal(q.astype(np.int64).reshape(2, B), want)
    # +-FLT_MAX and random values below it: +-127 at the absmax, |q - 127x/a|
    # at most 1/2, decoded values finite and within a / 254 (up to fp32 rounding)
    fmax = np.finfo(np.float32).max
    xr = (rng.uniform(-1, 1, size=3 * B) * fmax).astype(np.float32)
    xr[7], xr[B + 3], xr[2 * B + 60] = fmax, -fmax, fmax
    q, a = orc.quantize_blockwise(xr, B)
    assert np.array_equal(a, np.full(3, fmax, np.float32))
    assert q[7] == 127 and q[B + 3] == -127 and q[2 * B + 60] == 127
    exact = 127 * xr.astype(np.float64) / np.float64(fmax)
    assert np.abs(q.astype(np.float64) - exact).max() <= 0.5 + 1e-6
    y = orc.dequantize_blockwise(q, a, B)
    assert np.isfinite(y).all()
    err = np.abs(y.astype(np.float64) - xr.astype(np.float64))
    assert err.max() <= float(fmax) * (1 / 254 + 1e-6)


def pin_blockwise_memory(orc):
    """8-bit codes take a quarter of the fp32 bytes (bitsandbytes GPU page,
    section "Why quantization matters for LLM deployment"), plus one fp32
    scale per block."""
    B, n = 256, 256 * 100 + 3
    q, a = orc.quantize_blockwise(np.ones(n, np.float32), B)
    assert q.nbytes == n and a.nbytes == 4 * ((n + B - 1) // B)
    assert abs((q.nbytes + a.nbytes) / (4 * n) - (0.25 + 1 / B)) < 1e-3


ALL_PINS = [
    pin_half_roundtrip,
    pin_code_rule_exhaustive,
    pin_hand_example,
    pin_brute_tiny_config,
    pin_brute_random_small,
    pin_bias_brute,
    pin_bias_integer,
    pin_w16_free_brute,
    pin_w16_free_invariants,
    pin_bf16_roundtrip,
    pin_bf16_code_rule_exhaustive,
    pin_bf16_brute,
    pin_bf16_tau_inf_integer,
    pin_tau_inf_integer_inputs,
    pin_tau_zero_is_fp16_matmul,
    pin_outliers_are_column_scan,
    pin_permutation_invariance,
    pin_code_extremes,
    pin_blockwise_closed_forms,
    pin_blockwise_error_bound,
    pin_blockwise_locality,
    pin_blockwise_zero_and_scaling,
    pin_blockwise_memory,
    pin_blockwise_huge_scale,
]

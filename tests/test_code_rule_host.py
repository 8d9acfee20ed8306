"""The kernels' division-free code rule, restated step by step on the host.

The CUDA code takes vector-wise codes without a division or a conversion
instruction: p = x r with r = fl32(127 / a); f = floor(p) from a magic-number
round; the sign of (f + 1/2) a - 127 x, which one fma gives exactly, decides
between f and f + 1 (ties to even); for bf16, x and a are first scaled by one
power of two built from a's exponent bits.  Its fast path takes rint(p)
directly whenever p lies more than 2^-15 from every half-integer (p is within
2^-16 of 127 x / a) and falls back to the rule above otherwise.  Here the same fp32 steps run in
numpy (the fma's sign from an exact float64 product) over every finite fp16
or bf16 x against a spread of scales, including both ends of bf16's range,
and must equal round_half_even(127 x / a) in exact arithmetic.  This checks
the rule's arithmetic on the CPU; the GPU parity tests check the kernels.
"""

import numpy as np

import oracle_pins

KM = np.float32(12582912.0)  # 1.5 * 2^23


def _code_byte(x: np.ndarray, a: np.float32) -> np.ndarray:
    r = np.float32(127.0) / a
    p = (x * r).astype(np.float32)
    rn = ((p + KM).astype(np.float32) - KM).astype(np.float32)
    f = np.where(rn > p, rn - np.float32(1), rn).astype(np.float32)
    s = (f.astype(np.float64) + 0.5) * float(a) - 127.0 * x.astype(np.float64)
    fb = (f + KM).astype(np.float32).view(np.uint32)
    q = fb + np.where(s < 0, 1, np.where(s == 0, fb & 1, 0)).astype(np.uint32)
    return (q & 0xFF).astype(np.uint8).view(np.int8).astype(np.int64)


def _bf16_scale(a: np.float32):
    """The two power-of-two factors of the bf16 row rule, from a's bits."""
    b = int(np.float32(a).view(np.uint32))
    E = (b >> 23) & 0xFF
    e = E - 126 if E else (b & 0x7FFFFF).bit_length() - 149
    k = 1 - e
    k1 = int(k / 2)            # C division truncates toward zero
    k2 = k - k1
    s1 = np.uint32((k1 + 127) << 23).view(np.float32)
    s2 = np.uint32((k2 + 127) << 23).view(np.float32)
    return s1, s2


def _code_byte_fast(x: np.ndarray, a: np.float32) -> np.ndarray:
    """The fast path: rint(p) by the magic-number add when p = x fl32(127/a)
    lies more than 2^-15 from every half-integer, the exact rule otherwise."""
    r = np.float32(127.0) / a
    p = (x * r).astype(np.float32)
    t = (p + KM).astype(np.float32)
    e = (p - (t - KM).astype(np.float32)).astype(np.float32)
    fast = (t.view(np.uint32) & 0xFF).astype(np.uint8).view(np.int8).astype(np.int64)
    return np.where(np.abs(e) < np.float32(0.5 - 2.0 ** -15), fast, _code_byte(x, a))


def test_fp16_rule_is_exact():
    allv = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)
    rng = np.random.default_rng(41)
    scales = list(allv[rng.integers(1, len(allv), 40)])
    scales += [np.float16(127), np.float16(1), allv[1], allv[1023], np.float16(65504)]
    for a16 in scales:
        a16 = np.float16(a16)
        xs = allv[allv.astype(np.float64) <= float(a16)]
        xs = np.concatenate([xs, -xs[1:]])
        want = oracle_pins._exact_codes(xs, np.full(len(xs), a16, dtype=np.float16))
        for rule in (_code_byte, _code_byte_fast):
            got = rule(xs.astype(np.float32), np.float32(a16))
            bad = np.flatnonzero(got != want)
            assert len(bad) == 0, (rule.__name__, float(a16), xs[bad[:3]], got[bad[:3]],
                                   want[bad[:3]])


def test_bf16_scaled_rule_is_exact():
    pos = np.arange(0, 0x7F80, dtype=np.uint16)
    posv = oracle_pins._bf16_bits_to_f64(pos)
    rng = np.random.default_rng(42)
    scales = [int(b) for b in pos[rng.integers(1, len(pos), 24)]]
    scales += [0x0001, 0x007F, 0x0080, 0x3F80, 0x42FE, 0x7F7F, 0x7F00, 0x0400]
    for ab in scales:
        a = np.float32(oracle_pins._bf16_bits_to_f64([ab])[0])
        keep = posv <= float(a)
        xb = np.concatenate([pos[keep], pos[keep][1:] | 0x8000])
        x = oracle_pins._bf16_bits_to_f64(xb).astype(np.float32)
        s1, s2 = _bf16_scale(a)
        a_s = np.float32(np.float32(a * s1) * s2)
        assert 1.0 <= a_s < 2.0, (ab, a_s)
        with np.errstate(under="ignore"):
            x_s = ((x * s1).astype(np.float32) * s2).astype(np.float32)
        want = oracle_pins._exact_codes_bf16(x.astype(np.float64), float(a))
        for rule in (_code_byte, _code_byte_fast):
            got = rule(x_s, a_s)
            bad = np.flatnonzero(got != want)
            assert len(bad) == 0, (rule.__name__, hex(ab), x[bad[:3]], got[bad[:3]],
                                   want[bad[:3]])


def _bw_code(x: np.ndarray, a: np.float32) -> np.ndarray:
    """The blockwise codec's fast path: p = fl32(127 x) * fl32(1 / a), a
    magic-number rint, and the IEEE division only where p lies within 2^-14
    of a half-integer."""
    num = (np.float32(127.0) * x).astype(np.float32)
    r = np.float32(1.0) / a
    p = (num * r).astype(np.float32)
    t = (p + KM).astype(np.float32)
    e = (p - (t - KM).astype(np.float32)).astype(np.float32)
    fast = (t.view(np.uint32) & 0xFF).astype(np.uint8).view(np.int8).astype(np.int64)
    slow = np.rint((num / a).astype(np.float32)).astype(np.int64)
    return np.where(np.abs(e) < np.float32(0.5 - 2.0 ** -14), fast, slow)


def test_blockwise_fast_path_matches_the_division():
    """The codec's reciprocal fast path gives rint(fl32(fl32(127 x) / a)) on
    random states, exact ties and values right beside them."""
    rng = np.random.default_rng(43)
    for _ in range(200):
        a = np.float32(np.abs(rng.standard_normal()) * 10.0 ** rng.integers(-20, 20) + 1e-30)
        x = (rng.uniform(-1, 1, 20000) * a).astype(np.float32)
        k = rng.integers(-127, 127, 4000)
        ties = ((k + 0.5) * (float(a) / 127.0)).astype(np.float32)
        near = np.concatenate([np.nextafter(ties, np.float32(np.inf)),
                               np.nextafter(ties, np.float32(-np.inf))])
        x = np.concatenate([x, ties, near, np.array([a, -a, 0.0], np.float32)])
        x = x[np.abs(x) <= a]
        want = np.rint(((np.float32(127.0) * x).astype(np.float32) / a).astype(np.float32))
        got = _bw_code(x, a)
        bad = np.flatnonzero(got != want.astype(np.int64))
        assert len(bad) == 0, (float(a), x[bad[:3]], got[bad[:3]], want[bad[:3]])


def test_blockwise_fast_path_at_the_top_of_the_range():
    """Blocks with absmax a >= 2^120 are coded at the scale 2^-8: the fast
    path on the scaled values equals the scaled division, which equals the
    unscaled one wherever 127 x stays finite, and gives +-127 at +-a."""
    rng = np.random.default_rng(44)
    s = np.float32(2.0 ** -8)
    fmax = np.finfo(np.float32).max
    for a in [fmax, np.float32(3e38), np.float32(2.0 ** 121), np.float32(2.0 ** 120),
              *[np.float32(v) for v in 10.0 ** rng.uniform(36.13, 38.5, 60)]]:
        a = np.float32(min(a, fmax))
        x = (rng.uniform(-1, 1, 20000) * a).astype(np.float32)
        x = np.concatenate([x, np.array([a, -a, 0.0, a / 254, -a / 254], np.float32)])
        xs, as_ = (x * s).astype(np.float32), np.float32(a * s)
        got = _bw_code(xs, as_)
        want = np.rint(((np.float32(127.0) * xs).astype(np.float32) / as_).astype(np.float32))
        assert np.array_equal(got, want.astype(np.int64))
        assert got[-5] == 127 and got[-4] == -127
        with np.errstate(over="ignore"):
            plain = (np.float32(127.0) * x).astype(np.float32)
        ok = np.isfinite(plain)
        plain_q = np.rint((plain[ok] / a).astype(np.float32)).astype(np.int64)
        assert np.array_equal(got[ok], plain_q)

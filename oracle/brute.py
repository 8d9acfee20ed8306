"""Brute-force oracle for tiny inputs: exact integers and fractions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Independent of ``oracle.c``: every step is written here again with Python
integers and :class:`fractions.Fraction`, so the C oracle can be checked
against exact arithmetic.  The method is the LLM.int8() decomposition as the
pages state it ("Hugging Face Quantization with bitsandbytes", section 2:
outlier feature dimensions in 16-bit, the rest multiplied in int8 and
converted back to 16-bit at the end; section 3: threshold).

Differences from ``oracle.c`` are deliberate and only in precision:
codes are the exactly rounded rational round_half_even(127*x/a) (the C
oracle and the kernels decide them in fp32; a test pins that the two agree),
and Y is the exact rational value rounded once to fp16.
"""

from __future__ import annotations

import math
import struct
from fractions import Fraction


def half_bits_to_fraction(bits: int) -> Fraction:
    """Exact value of an fp16 bit pattern (finite values only)."""
    (v,) = struct.unpack("<e", struct.pack("<H", bits))
    if math.isinf(v) or math.isnan(v):
        raise ValueError("non-finite fp16")
    return Fraction(v)


def bf16_bits_to_fraction(bits: int) -> Fraction:
    """Exact value of a bfloat16 bit pattern (finite values only): the high
    half of the binary32 with the same leading bits."""
    (v,) = struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))
    if math.isinf(v) or math.isnan(v):
        raise ValueError("non-finite bf16")
    return Fraction(v)


def round_half_even(q: Fraction) -> int:
    """Nearest integer to q, ties to the even one."""
    fl = math.floor(q)
    rem = q - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def fraction_to_half_bits(v: Fraction) -> int:
    """Round an exact rational to binary16, nearest-even (overflow -> inf)."""
    sign = 0x8000 if v < 0 else 0
    a = -v if v < 0 else v
    if a == 0:
        return sign
    # exponent E with 2^E <= a < 2^(E+1)
    E = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** E > a:
        E -= 1
    if E < -14:
        n = round_half_even(a * 2 ** 24)  # subnormal quantum 2^-24
        return sign | n                  # n == 1024 is the smallest normal
    n = round_half_even(a / Fraction(2) ** (E - 10))
    if n == 2048:
        n, E = 1024, E + 1
    if E > 15:
        return sign | 0x7C00
    return sign | ((E + 15) << 10) | (n - 1024)


def fraction_to_bf16_bits(v: Fraction) -> int:
    """Round an exact rational to bfloat16 (8 significand bits, exponents
    -126..127, subnormal quantum 2^-133), nearest-even, overflow -> inf."""
    sign = 0x8000 if v < 0 else 0
    a = -v if v < 0 else v
    if a == 0:
        return sign
    E = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** E > a:
        E -= 1
    if E < -126:
        n = round_half_even(a * 2 ** 133)
        return sign | n                   # n == 128 is the smallest normal
    n = round_half_even(a / Fraction(2) ** (E - 7))
    if n == 256:
        n, E = 128, E + 1
    if E > 127:
        return sign | 0x7F80
    return sign | ((E + 127) << 7) | (n - 128)


def code(x: Fraction, a: Fraction) -> int:
    """Vector-wise int8 code of x against absmax a (0 when a == 0)."""
    if a == 0:
        return 0
    return round_half_even(Fraction(127) * x / a)


def linear(X_bits, W_bits, tau: float, bias_bits=None, w16_free: bool = False,
           fmt: str = "fp16"):
    """The whole decomposition linear on tiny lists of fp16 bit patterns.

    X_bits: T lists of K ints, W_bits: N lists of K ints.  Returns a dict with
    O, Xq, sx, Wq, sw, acc and Y (fp16 bit patterns), all exact.  bias_bits:
    N fp16 bit patterns added before the final rounding (or None).
    w16_free: the outlier weights are the codes dequantized, Wq * sw / 127,
    instead of W itself.  fmt "bf16": every bit pattern (in and out) is
    bfloat16 instead of fp16.
    """
    to_frac = bf16_bits_to_fraction if fmt == "bf16" else half_bits_to_fraction
    to_bits = fraction_to_bf16_bits if fmt == "bf16" else fraction_to_half_bits
    T, K, N = len(X_bits), len(X_bits[0]) if X_bits else 0, len(W_bits)
    X = [[to_frac(b) for b in row] for row in X_bits]
    W = [[to_frac(b) for b in row] for row in W_bits]
    tau_f = Fraction(tau) if math.isfinite(tau) else None
    # outlier feature columns: any row at or above the threshold
    O = [k for k in range(K)
         if tau_f is not None and any(abs(X[t][k]) >= tau_f for t in range(T))]
    Oset = set(O)
    # per-output-channel weight scale and codes
    sw = [max((abs(w) for w in row), default=Fraction(0)) for row in W]
    Wq = [[code(w, sw[n]) for w in W[n]] for n in range(N)]
    # per-row activation scale over non-outlier columns, and codes
    sx = [max((abs(X[t][k]) for k in range(K) if k not in Oset), default=Fraction(0))
          for t in range(T)]
    Xq = [[0 if k in Oset else code(X[t][k], sx[t]) for k in range(K)] for t in range(T)]
    acc = [[sum(Xq[t][k] * Wq[n][k] for k in range(K)) for n in range(N)] for t in range(T)]
    Y = []
    for t in range(T):
        row = []
        for n in range(N):
            v = Fraction(acc[t][n]) * sx[t] * sw[n] / 16129
            if w16_free:
                v += sum((X[t][k] * Wq[n][k] * sw[n] / 127 for k in O), Fraction(0))
            else:
                v += sum((X[t][k] * W[n][k] for k in O), Fraction(0))
            if bias_bits is not None:
                v += to_frac(bias_bits[n])
            row.append(to_bits(v))
        Y.append(row)
    return {"O": O, "Xq": Xq, "sx": sx, "Wq": Wq, "sw": sw, "acc": acc, "Y": Y}

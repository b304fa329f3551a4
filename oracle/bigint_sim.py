"""ORACLE CHECK -- test infrastructure only (never on the product path).

An exact simulation of one IEEE-754 binary64 addition, rounded to nearest with
ties to even, written with Python integers only: the two operands are turned
into exact integer-over-power-of-two values, added exactly, and the exact
result is rounded to 53 significant bits (with the subnormal range and
overflow to infinity handled as IEEE-754 section 4.3.1 and 7.4 state).  It
never uses the host's floating-point adder, so it is an independent check on
the C oracle's loop (Research-1433, Question: the sum to reproduce is
``for (i = 0; i < n; i++) s += x[i];``).

The zero-sign rule follows IEEE-754 section 6.3: an exact zero sum of
operands with opposite signs (or of two opposite-signed zeros) is +0 in
round-to-nearest; the sum of two -0 is -0.
"""
from __future__ import annotations

import math

EMIN_Q = -1074          # exponent of the subnormal unit, 2^-1074
PREC = 53               # significand bits


def _is_neg_zero(x: float) -> bool:
    return x == 0.0 and math.copysign(1.0, x) < 0


def round_exact(num: int, k: int) -> float:
    """Round the exact value num / 2^k (num != 0) to the nearest binary64,
    ties to even."""
    neg = num < 0
    a = -num if neg else num
    e = a.bit_length() - 1 - k              # floor(log2(value))
    q = max(e - (PREC - 1), EMIN_Q)         # exponent of the last place
    shift = k + q                           # value / 2^q = a / 2^shift
    if shift <= 0:
        m = a << (-shift)                   # exact, no rounding
    else:
        m = a >> shift
        rem = a - (m << shift)
        half = 1 << (shift - 1)
        if rem > half or (rem == half and (m & 1)):
            m += 1
    if m == 0:
        return -0.0 if neg else 0.0
    if m.bit_length() - 1 + q >= 1024:      # rounded value >= 2^1024
        return -math.inf if neg else math.inf
    v = math.ldexp(m, q)                    # m <= 2^53: exactly representable
    return -v if neg else v


def add_rne(a: float, b: float) -> float:
    """a + b in binary64, round to nearest even, by exact integer arithmetic."""
    if math.isnan(a) or math.isnan(b):
        return math.nan
    if math.isinf(a) or math.isinf(b):
        if math.isinf(a) and math.isinf(b) and (a > 0) != (b > 0):
            return math.nan
        return a if math.isinf(a) else b
    if a == 0.0 and b == 0.0:
        return -0.0 if (_is_neg_zero(a) and _is_neg_zero(b)) else 0.0
    na, da = a.as_integer_ratio()           # da, db are powers of two
    nb, db = b.as_integer_ratio()
    ka, kb = da.bit_length() - 1, db.bit_length() - 1
    k = max(ka, kb)
    num = (na << (k - ka)) + (nb << (k - kb))
    if num == 0:
        return 0.0                          # exact cancellation: +0 under RNE
    return round_exact(num, k)


def seqsum(xs, s0: float = 0.0) -> float:
    """The sequential sum, every add simulated exactly."""
    s = float(s0)
    for v in xs:
        s = add_rne(s, float(v))
    return s


def exact_sum(xs, s0: float = 0.0):
    """The exact (unrounded) sum as (num, k): value = num / 2^k."""
    num, k = 0, 0
    for v in [float(s0)] + [float(t) for t in xs]:
        n, d = v.as_integer_ratio()
        kd = d.bit_length() - 1
        if kd > k:
            num <<= (kd - k)
            k = kd
        num += n << (k - kd)
    return num, k

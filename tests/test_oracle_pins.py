"""Pins for the oracle: it is checked against things other than itself.

* hand-built ties and special cases worked out from the rounding rule
  (tests/golden/ties.txt);
* an exact integer simulation of every binary64 add (oracle/bigint_sim.py),
  which uses no floating-point adder, on many short sequences chosen so that
  ties, binade crossings, cancellation and subnormals are dense;
* closed forms: integer-valued terms whose partial sums are all below 2^53 add
  without rounding, so the result must equal the exact integer sum;
* planted mistakes (reverse order, a dropped term, a compensated or exactly
  rounded sum, an ignored start value) must each fail at least one pin.
"""
import math
import random

import numpy as np
import pytest

from conftest import load_golden
from oracle import bigint_sim as sim


def bits(v):
    return np.float64(v).view(np.uint64).item()


def same(a, b):
    if a != a and b != b:
        return True
    return bits(a) == bits(b)


# ------------------------------------------------------------ simulator pins

def test_sim_textbook_values():
    # each value follows from the rounding rule by hand
    assert sim.add_rne(1.0, 2.0 ** -53) == 1.0
    assert sim.add_rne(1.0 + 2.0 ** -52, 2.0 ** -53) == 1.0 + 2.0 ** -51
    assert sim.add_rne(2.0 ** 53, 1.0) == 2.0 ** 53
    assert sim.add_rne(2.0 ** 53, 3.0) == 2.0 ** 53 + 4.0
    assert sim.add_rne(2.0 ** 53 + 2.0, 1.0) == 2.0 ** 53 + 4.0
    assert sim.add_rne(5e-324, 5e-324) == 1e-323
    assert math.isinf(sim.add_rne(1.7976931348623157e308, 2.0 ** 970))
    assert sim.add_rne(1.7976931348623157e308, 2.0 ** 969) == 1.7976931348623157e308
    assert bits(sim.add_rne(-0.0, -0.0)) == bits(-0.0)
    assert bits(sim.add_rne(-0.0, 0.0)) == bits(0.0)
    assert bits(sim.add_rne(1.5, -1.5)) == bits(0.0)
    assert math.isnan(sim.add_rne(math.inf, -math.inf))
    assert sim.add_rne(math.inf, 1.0) == math.inf
    assert sim.add_rne(-3.0, 1.0) == -2.0
    # 0.1 + 0.2 is the textbook 0.30000000000000004
    assert sim.add_rne(0.1, 0.2) == float.fromhex("0x1.3333333333334p-2")


@pytest.mark.parametrize("label,s0,xs,expected", load_golden("ties.txt"))
def test_sim_golden(label, s0, xs, expected):
    assert same(sim.seqsum(xs, s0), expected), label


# --------------------------------------------------------------- oracle pins

def test_oracle_env(oracle_mod):
    assert oracle_mod.lib().oracle_env_check() == 0


@pytest.mark.parametrize("label,s0,xs,expected", load_golden("ties.txt"))
def test_oracle_golden(oracle_mod, label, s0, xs, expected):
    got = oracle_mod.seqsum(np.array(xs, dtype=np.float64), s0)
    assert same(got, expected), (label, got.hex(), expected)


def _random_sequences(seed, count):
    """Short sequences with dense ties and crossings: small integer multiples
    of powers of two in a narrow exponent window, both signs, plus zeros,
    subnormals and a few huge or non-finite values."""
    rng = random.Random(seed)
    for _ in range(count):
        n = rng.randint(0, 48)
        kind = rng.randrange(6)
        base = rng.randint(-60, 60)
        xs = []
        for _ in range(n):
            r = rng.random()
            if kind == 0:      # multiples of 2^(base-53): ties every other add
                v = rng.randint(1, 7) * 2.0 ** (base - 53)
            elif kind == 1:    # random 53-bit mantissas, narrow window
                v = math.ldexp(rng.getrandbits(53) | (1 << 52), base - 52 + rng.randint(-3, 3))
            elif kind == 2:    # mixed signs: cancellation, descending crossings
                v = math.ldexp(rng.getrandbits(20) + 1, base + rng.randint(-25, 5))
                v = -v if rng.random() < 0.45 else v
            elif kind == 3:    # subnormal range
                v = rng.randint(0, 1 << 10) * 5e-324 * (1 if rng.random() < 0.8 else -1)
            elif kind == 4:    # near the top of the range
                v = math.ldexp(rng.getrandbits(53) | (1 << 52), 1023 - 52 - rng.randint(0, 3))
            else:              # wide mix
                v = math.ldexp(rng.getrandbits(53), rng.randint(-1100, 970))
                v = -v if rng.random() < 0.3 else v
            if r < 0.05:
                v = 0.0 if rng.random() < 0.5 else -0.0
            elif r < 0.06:
                v = rng.choice([math.inf, -math.inf, math.nan])
            xs.append(v)
        s0 = rng.choice([0.0, -0.0, 1.0, -1.0, xs[0] if xs else 2.5])
        yield s0, xs


def test_oracle_vs_exact_simulation(oracle_mod):
    checked = 0
    for s0, xs in _random_sequences(1433, 6000):
        want = sim.seqsum(xs, s0)
        got = oracle_mod.seqsum(np.array(xs, dtype=np.float64), s0)
        assert same(got, want), (s0, [v.hex() for v in xs], got, want)
        checked += 1
    assert checked == 6000


def test_oracle_trace_vs_simulation(oracle_mod):
    rng = random.Random(7)
    xs = [rng.randint(1, 9) * 2.0 ** -53 for _ in range(300)]
    tr = oracle_mod.seqsum_trace(np.array(xs), 1.0 - 2.0 ** -40)
    s = 1.0 - 2.0 ** -40
    for i, v in enumerate(xs):
        s = sim.add_rne(s, v)
        assert same(tr[i], s), i


def test_closed_form_integer_terms(oracle_mod):
    """c1-shaped plane with q restricted to multiples of 2^-16 inside and
    q = 1 at the edge: every term w*q is an integer, every partial sum stays
    below 2^53, so no add rounds."""
    import workloads as W
    n = 576 * 324
    u = W.draws_u64(0, 0, n)
    q = ((u >> np.uint64(48)).astype(np.float64) + 32768.0) * 2.0 ** -16   # [0.5,1)
    w = np.full(n, 65536.0)
    edge = W.edge_mask(576, 324)
    w[edge] = W.uniform_int(W.draws_u64(0, 1, n), 1, 65535)[edge]
    q[edge] = 1.0
    x = w * q
    assert np.all(x == np.floor(x))
    exact = sum(int(v) for v in x)
    assert exact < 2 ** 53
    assert oracle_mod.seqsum(x, 0.0) == float(exact)
    # and from a start value that keeps the sum integral
    assert oracle_mod.seqsum(x, 12345.0) == float(exact + 12345)


def test_closed_form_dyadic_terms(oracle_mod):
    """Multiples of 2^-53 with a total below 2 stay exact in [1, 2) only if the
    sum never needs more than 53 bits; with terms that are multiples of 2^-52
    and s0 = 1 every partial sum is a multiple of 2^-52 below 2: exact."""
    rng = np.random.default_rng(5)
    k = rng.integers(0, 64, size=4000)
    x = k.astype(np.float64) * 2.0 ** -52
    exact = 2 ** 52 + int(k.sum())
    assert exact < 2 ** 53
    assert oracle_mod.seqsum(x, 1.0) == exact * 2.0 ** -52


def test_batched_vs_simulation(oracle_mod):
    rng = random.Random(11)
    seqs = list(_random_sequences(99, 40))
    x = np.array([v for _, xs in seqs for v in xs], dtype=np.float64)
    offs = np.zeros(len(seqs) + 1, dtype=np.int64)
    offs[1:] = np.cumsum([len(xs) for _, xs in seqs])
    s0s = np.array([s0 for s0, _ in seqs])
    out = oracle_mod.seqsum_batched(x, offs, s0s)
    for k, (s0, xs) in enumerate(seqs):
        assert same(out[k], sim.seqsum(xs, s0)), k
    del rng


def test_strided_vs_simulation(oracle_mod):
    """Interleaved sums (ADR-1464, Decision: the lcs variant's four sums per
    window, one accumulator each): every sum is pinned to the exact
    simulation of its own subsequence, and every mean to the division
    rounded to the nearest double by exact rational arithmetic, then to the
    nearest float (the host's (float)(sum / windows))."""
    from fractions import Fraction
    rng = random.Random(21)
    for stride in [1, 2, 4, 7]:
        for n in [1, 2, 5, 33, 200]:
            xs = []
            for _ in range(n * stride):
                e = rng.randint(-60, 8)
                xs.append(rng.choice([1.0, -1.0, 1.0]) * rng.randint(1, 2 ** 20) * 2.0 ** e)
            s0s = [rng.choice([0.0, 1.0, -0.5, 3.0]) for _ in range(stride)]
            sums, means = oracle_mod.seqsum_strided(np.array(xs), stride, np.array(s0s))
            for k in range(stride):
                want = sim.seqsum(xs[k::stride], s0s[k])
                assert same(sums[k], want), (stride, n, k)
                q = float(Fraction(want) / n)          # correctly rounded double quotient
                assert np.float32(q).view(np.uint32) == means[k].view(np.uint32), (stride, n, k)


def test_strided_closed_forms(oracle_mod):
    """Integer terms: each interleaved sum is the exact integer total; with
    n a power of two the mean is that total scaled exactly; 1/3 as a float
    is 0x3EAAAAAB."""
    n, stride = 1024, 4
    x = np.arange(n * stride, dtype=np.float64)
    sums, means = oracle_mod.seqsum_strided(x, stride, np.zeros(stride))
    for k in range(stride):
        exact = sum(i * stride + k for i in range(n))
        assert sums[k] == float(exact)
        assert means[k] == np.float32(exact / 1024.0)
    sums, means = oracle_mod.seqsum_strided(np.array([1.0, 0.0, 0.0]), 1, np.zeros(1))
    assert sums[0] == 1.0 and means[0].view(np.uint32) == 0x3EAAAAAB


# ------------------------------------------------------- planted mistakes

def _pin_suite_passes(fn):
    """True when `fn(xs, s0)` passes every pin above (golden, simulation,
    closed form).  Used to show that each planted mistake is caught."""
    for label, s0, xs, expected in load_golden("ties.txt"):
        if not same(fn(xs, s0), expected):
            return False
    for s0, xs in _random_sequences(2024, 600):
        if not same(fn(xs, s0), sim.seqsum(xs, s0)):
            return False
    return True


@pytest.mark.parametrize("mutant", ["reverse", "drop_last", "exact_rounding", "kahan", "ignore_s0",
                                    "pairwise"])
def test_planted_mistakes_are_caught(oracle_mod, mutant):
    def reverse(xs, s0):
        return oracle_mod.seqsum(np.array(xs[::-1], dtype=np.float64), s0)

    def drop_last(xs, s0):
        return oracle_mod.seqsum(np.array(xs[:-1], dtype=np.float64), s0)

    def exact_rounding(xs, s0):
        return math.fsum([s0] + list(xs)) if all(map(math.isfinite, [s0] + xs)) else sim.seqsum(xs, s0)

    def kahan(xs, s0):
        s, c = s0, 0.0
        for v in xs:
            y = v - c
            t = s + y
            c = (t - s) - y
            s = t
        return s

    def ignore_s0(xs, s0):
        return oracle_mod.seqsum(np.array(xs, dtype=np.float64), 0.0)

    def pairwise(xs, s0):
        vals = [s0] + list(xs)
        while len(vals) > 1:
            vals = [vals[i] + vals[i + 1] if i + 1 < len(vals) else vals[i]
                    for i in range(0, len(vals), 2)]
        return vals[0]

    fn = dict(reverse=reverse, drop_last=drop_last, exact_rounding=exact_rounding,
              kahan=kahan, ignore_s0=ignore_s0, pairwise=pairwise)[mutant]
    assert not _pin_suite_passes(fn), f"pins did not catch the '{mutant}' mistake"
    # and the real oracle passes the same suite
    assert _pin_suite_passes(lambda xs, s0: oracle_mod.seqsum(np.array(xs, dtype=np.float64), s0))

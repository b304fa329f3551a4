"""Seeded synthetic term planes shaped like the workloads the pages measure.

This module only draws inputs. It holds none of the summation method: no
binade, no increment, no rounding rule. Both the oracle (under ``oracle/``)
and the CUDA path are fed the same arrays from here, so the two sides can be
compared bit for bit.

The random source is splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used as a counter-based
generator: draw ``i`` of a stream is ``mix(base + (i + 1) * GAMMA)``, which is
what the sequential generator started from state ``base`` returns at its
``i``-th call. Every float step below is a single IEEE-754 binary64 operation
(numpy applies one ufunc at a time and does not contract), so the same seed
gives the same bytes on x86-64 and on aarch64.

Workloads (the pages' fixtures are not available, so these stand in for them):

* ``c1`` -- 576x324 plane of integer_ssim-style terms ``w * q``
  (Research-1424, section 1 "The sum is the only difference": the per-pixel
  term carries the window weight ``m.w``; ADR-1443, "Three shortcuts, each
  exact": interior windows have weight 2^16, edge windows a smaller one).
* ``c2`` -- 1920x1080 ssimulacra2-style ``d = 1 - q`` with ``q`` a multiple of
  2^-53 in [0.5, 1) (Research-1433, finding 3 "Ties need the parity of the
  running integer": such terms tie every second add while the sum is in [1, 2)).
* ``c3`` -- 3840x2160 non-negative terms spanning 41 binades after 64 zero rows
  (Research-1424, section 3: the 4K sum crosses a dozen binades in its first
  row; Research-1433, finding 4: one fallback chunk per binade crossed).
* ``c4`` -- the 108 sums of one ssimulacra2 frame, 6 scales x 3 channels x 6
  sums (ADR-1391, Decision item 3: one 864-byte copy of the per-scale sums).
* ``c5`` -- 3840x2160 signed integer_ssim-style terms ``w * s``
  (Research-1424, section 3: signed terms need the smallest and largest prefix).
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function (uint64 in, uint64 out, wrapping)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def mix_scalar(v: int) -> int:
    """splitmix64 output function on one Python int (mod 2^64)."""
    z = v & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_base(seed: int, stream: int) -> int:
    """Starting state of sub-stream ``stream`` of ``seed`` (independent draws
    for independent purposes: values, weights, zero masks ...)."""
    return mix_scalar(mix_scalar(seed) ^ ((stream + 1) * 0xD1B54A32D192ED03))


def draws_u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Draws ``start .. start+n-1`` of a splitmix64 sub-stream, as uint64."""
    base = np.uint64(stream_base(seed, stream))
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + idx * GAMMA)


def uniform53(u: np.ndarray) -> np.ndarray:
    """Random 53-bit double in [0, 1): (u >> 11) * 2^-53 (exact)."""
    return (u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def half_open_q(u: np.ndarray) -> np.ndarray:
    """Random 53-bit double in [0.5, 1): (2^52 + (u >> 12)) * 2^-53 (exact)."""
    return ((u >> np.uint64(12)) + np.uint64(1 << 52)).astype(np.float64) * (2.0 ** -53)


def mantissa_1_2(u: np.ndarray) -> np.ndarray:
    """Random 53-bit double in [1, 2): 1 + (u >> 12) * 2^-52 (exact)."""
    return ((u >> np.uint64(12)) + np.uint64(1 << 52)).astype(np.float64) * (2.0 ** -52)


def uniform_int(u: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """Integer uniform in [lo, hi] (inclusive) from the top bits, as int64.
    Uses the multiply-shift map of the top 32 bits; the bias is below 2^-15
    for ranges up to 2^17, which is irrelevant for synthetic inputs."""
    span = np.uint64(hi - lo + 1)
    top = u >> np.uint64(32)
    return ((top * span) >> np.uint64(32)).astype(np.int64) + np.int64(lo)


def edge_mask(width: int, height: int, border: int = 5) -> np.ndarray:
    """True for windows within ``border`` pixels of the frame edge (raster order)."""
    y = np.arange(height)[:, None]
    x = np.arange(width)[None, :]
    m = (y < border) | (y >= height - border) | (x < border) | (x >= width - border)
    return m.reshape(-1)


def approx_normal(seed: int, stream: int, n: int) -> np.ndarray:
    """Approximately N(0, 1): the Irwin-Hall sum of twelve U[0,1) minus 6.

    Box-Muller would need log and cos, whose last bit is library-dependent;
    this form uses only exact-order IEEE adds, so both machines draw the same
    bytes. Mean 0, variance 1, support [-6, 6]."""
    acc = np.zeros(n, dtype=np.float64)
    for j in range(12):
        acc = acc + uniform53(draws_u64(seed, stream + j, n))
    return acc - 6.0


# ---------------------------------------------------------------- configs

@dataclass
class Workload:
    """One or more sums over a concatenated fp64 plane."""
    name: str
    x: np.ndarray                 # float64, all sums concatenated in order
    offsets: np.ndarray           # int64, nsums + 1 entries
    s0: np.ndarray                # float64, one start value per sum
    shape: list = field(default_factory=list)   # (width, height) per sum
    recipe: str = ""

    @property
    def nsums(self) -> int:
        return len(self.offsets) - 1

    def sum_slice(self, k: int) -> np.ndarray:
        return self.x[self.offsets[k]:self.offsets[k + 1]]

    def checksum(self) -> str:
        h = hashlib.blake2b(digest_size=16)
        h.update(np.ascontiguousarray(self.x).view(np.uint8))
        h.update(np.ascontiguousarray(self.offsets).view(np.uint8))
        h.update(np.ascontiguousarray(self.s0).view(np.uint8))
        return h.hexdigest()


def _single(name, x, w, h, recipe, s0=0.0):
    return Workload(name, np.ascontiguousarray(x, dtype=np.float64),
                    np.array([0, len(x)], dtype=np.int64),
                    np.array([s0], dtype=np.float64), [(w, h)], recipe)


def plane_c1(width=576, height=324, seed=0):
    """w * q: q uniform 53-bit in [0.5, 1); w = 65536 inside, w in [1, 65535]
    within 5 px of the edge."""
    n = width * height
    q = half_open_q(draws_u64(seed, 0, n))
    w = np.full(n, 65536.0)
    edge = edge_mask(width, height)
    w[edge] = uniform_int(draws_u64(seed, 1, n), 1, 65535)[edge].astype(np.float64)
    return w * q


def plane_c2(width=1920, height=1080, seed=2, zero_frac=0.10):
    """d = 1 - k * 2^-53, k uniform in [2^52, 2^53); a fraction of exact zeros."""
    n = width * height
    k = (draws_u64(seed, 0, n) >> np.uint64(12)) + np.uint64(1 << 52)
    q = k.astype(np.float64) * (2.0 ** -53)
    d = 1.0 - q
    z = uniform53(draws_u64(seed, 1, n)) < zero_frac
    d[z] = 0.0
    return d


def plane_pow2(n, seed, u_lo, u_hi, stream=0):
    """2^U * mantissa with U uniform integer in [u_lo, u_hi], mantissa in [1, 2)."""
    U = uniform_int(draws_u64(seed, stream, n), u_lo, u_hi)
    m = mantissa_1_2(draws_u64(seed, stream + 1, n))
    return np.ldexp(m, U.astype(np.int32))


def plane_c3(width=3840, height=2160, seed=3, zero_rows=64, zero_frac=0.01):
    """64 zero rows, then 2^U * mant, U in [-40, 0]; 1% exact zeros."""
    n = width * height
    x = plane_pow2(n, seed, -40, 0)
    z = uniform53(draws_u64(seed, 2, n)) < zero_frac
    x[z] = 0.0
    x[: zero_rows * width] = 0.0
    return x


def plane_c5(width=3840, height=2160, seed=5):
    """w * s: s = 0.95 + 0.05 * N(0,1) clipped to [-0.2, 1.0]; 2% of windows
    s uniform in [-0.2, 0.2]; w = 65536 inside, [1, 65535] near the edge."""
    n = width * height
    s = 0.95 + 0.05 * approx_normal(seed, 10, n)
    s = np.clip(s, -0.2, 1.0)
    lowsel = uniform53(draws_u64(seed, 2, n)) < 0.02
    s_low = -0.2 + 0.4 * uniform53(draws_u64(seed, 3, n))
    s[lowsel] = s_low[lowsel]
    w = np.full(n, 65536.0)
    edge = edge_mask(width, height)
    w[edge] = uniform_int(draws_u64(seed, 1, n), 1, 65535)[edge].astype(np.float64)
    return w * s


C4_SCALES = [(3840, 2160), (1920, 1080), (960, 540), (480, 270), (240, 135), (120, 68)]


def c4_seed(scale: int, channel: int, which: int) -> int:
    return mix_scalar((4 << 32) | (scale << 16) | (channel << 8) | which)


def plane_c4_sum(width, height, seed):
    """Half c2-style terms, half 2^U * mant with U in [-30, 2] (per-term choice)."""
    n = width * height
    a = plane_c2(width, height, seed=seed)
    b = plane_pow2(n, seed, -30, 2, stream=5)
    pick = uniform53(draws_u64(seed, 7, n)) < 0.5
    return np.where(pick, a, b)


def config(name: str, scale_div: int = 1, height_mult: int = 1) -> Workload:
    """The five workloads. ``scale_div`` > 1 shrinks width and height (for
    quick tests); ``height_mult`` > 1 makes a single-sum plane that many times
    taller (larger than L2, for profiling); the recipe is otherwise unchanged."""
    d = scale_div
    if height_mult > 1 and name != "c4":
        base = config(name, scale_div)
        w, h = base.shape[0]
        planes = {"c1": plane_c1, "c2": plane_c2, "c3": plane_c3, "c5": plane_c5}
        big = planes[name](w, h * height_mult)
        return _single(name, big, w, h * height_mult, base.recipe + f", {height_mult}x taller")
    if name == "c1":
        w, h = 576 // d, 324 // d
        return _single("c1", plane_c1(w, h), w, h,
                       "w*q, q in [0.5,1) 53-bit, w=65536 inside / [1,65535] edge, seed 0")
    if name == "c2":
        w, h = 1920 // d, 1080 // d
        return _single("c2", plane_c2(w, h), w, h,
                       "1 - k*2^-53, k in [2^52,2^53), 10% zeros, seed 2")
    if name == "c3":
        w, h = 3840 // d, 2160 // d
        return _single("c3", plane_c3(w, h, zero_rows=max(1, 64 // d)), w, h,
                       "64 zero rows, then 2^U*mant, U in [-40,0], 1% zeros, seed 3")
    if name == "c5":
        w, h = 3840 // d, 2160 // d
        return _single("c5", plane_c5(w, h), w, h,
                       "w*s, s=0.95+0.05*N(0,1) clip [-0.2,1], 2% s in [-0.2,0.2], seed 5")
    if name == "c4":
        xs, shapes = [], []
        for si, (w, h) in enumerate(C4_SCALES):
            w2, h2 = max(1, w // d), max(1, h // d)
            for ch in range(3):
                for k in range(6):
                    xs.append(plane_c4_sum(w2, h2, c4_seed(si, ch, k)))
                    shapes.append((w2, h2))
        offs = np.zeros(len(xs) + 1, dtype=np.int64)
        offs[1:] = np.cumsum([len(v) for v in xs])
        return Workload("c4", np.concatenate(xs), offs, np.zeros(len(xs)), shapes,
                        "108 sums: 6 scales x 3 channels x 6 sums; half c2-style, "
                        "half 2^U*mant U in [-30,2]; seed per (scale, channel, sum)")
    raise KeyError(name)


CONFIG_NAMES = ["c1", "c2", "c3", "c4", "c5"]

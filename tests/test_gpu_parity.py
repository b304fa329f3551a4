"""Parity of the CUDA path with the oracle, bit for bit (tolerance: 0 ULP;
NaN results compare as "both NaN", the one case the oracle leaves unpinned).

Every input comes from the seeded generators in ``workloads``; every expected
value comes from ``oracle`` on the same bytes.  All calls go through the
C-ABI library, in the same launch configuration the benchmark times.
"""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import parity_binade_chunked_gb300 as sq
    sq.lib()
    return sq


def bits(v):
    return np.float64(v).view(np.uint64).item()


def assert_same(got, want, what=""):
    got, want = float(got), float(want)
    if got != got and want != want:
        return
    assert bits(got) == bits(want), f"{what}: got {got!r} ({got.hex()}) want {want!r} ({want.hex()})"


def gpu_sum(sq, x, s0=0.0, offset=0):
    """One call through the C ABI.  offset > 0 shifts the data by that many
    doubles inside a larger buffer (misaligned starts)."""
    buf = torch.zeros(len(x) + offset, dtype=torch.float64, device="cuda")
    if len(x):
        buf[offset:] = torch.from_numpy(np.ascontiguousarray(x))
    xv = buf[offset:]
    out = sq.seqsum_f64(xv, s0)
    torch.cuda.synchronize()
    return out.item()


def check(sq, x, s0=0.0, what="", offset=0):
    want = oracle.seqsum(x, s0)
    sq.get_stats()   # counters of earlier calls out of the way
    got = gpu_sum(sq, x, s0, offset)
    assert_same(got, want, what)
    st = sq.get_stats()
    assert st["device_status"] == 0, st
    return st


# ------------------------------------------------------------ the workloads

@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c5"])
@pytest.mark.parametrize("div", [8, 3])
def test_config_reduced(sq, name, div):
    wl = W.config(name, scale_div=div)
    check(sq, wl.x, float(wl.s0[0]), f"{name}/{div}")


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c5"])
def test_config_full_size(sq, name):
    wl = W.config(name)
    st = check(sq, wl.x, float(wl.s0[0]), name)
    assert st["tiles"] == (len(wl.x) + 4095) // 4096


def _batched(sq, wl, sized):
    x = torch.from_numpy(wl.x).cuda()
    offs = torch.from_numpy(wl.offsets).cuda()
    s0s = torch.from_numpy(wl.s0).cuda()
    outs = sq.seqsum_f64_batched_sized(x, offs, s0s) if sized else sq.seqsum_f64_batched(x, offs, s0s)
    torch.cuda.synchronize()
    return outs.cpu().numpy()


@pytest.mark.parametrize("sized", [False, True])
def test_config_c4_reduced(sq, sized):
    wl = W.config("c4", scale_div=8)
    got = _batched(sq, wl, sized)
    want = oracle.seqsum_batched(wl.x, wl.offsets, wl.s0)
    for k in range(wl.nsums):
        assert_same(got[k], want[k], f"c4/8 sum {k}")
    assert sq.get_stats()["device_status"] == 0


def test_config_c4_full_size(sq):
    wl = W.config("c4")
    got = _batched(sq, wl, True)
    want = oracle.seqsum_batched(wl.x, wl.offsets, wl.s0)
    for k in range(wl.nsums):
        assert_same(got[k], want[k], f"c4 sum {k}")
    st = sq.get_stats()
    assert st["device_status"] == 0
    got2 = _batched(sq, wl, False)
    assert np.array_equal(got.view(np.uint64), got2.view(np.uint64))


@pytest.mark.parametrize("name", ["c3", "c5"])
@pytest.mark.parametrize("mult", [2, 4])
def test_single_sums_above_the_wave(sq, name, mult):
    """One sum of 2x and 4x the plane's height: more tiles than the wave the
    plan units run ahead of the run units (2048), so plan and run units mix
    and the walk takes ranges while tiles are still being formed."""
    wl = W.config(name, height_mult=mult)
    st = check(sq, wl.x, float(wl.s0[0]), f"{name} x{mult}")
    assert st["tiles"] == (len(wl.x) + 4095) // 4096


def test_single_sum_one_term_past_2048_tiles(sq):
    """2048 * 4096 + 1 terms: the last tile holds one term, one past the wave."""
    x = W.plane_c2(2048 * 4096 + 1, 1, seed=31)
    st = check(sq, x, 0.125, "2048 tiles + 1 term")
    assert st["tiles"] == 2049


# ------------------------------------------------------------ bounded waits

def test_withheld_header_times_out_then_recovers(sq):
    """A tile header that never comes (the fault hook withholds it): the
    walk's bounded wait gives up, the call writes NaN and reports
    SEQSUM_ETIMEOUT at site 3 (a walk header), and the next call -- on the
    same workspace -- is exact again."""
    x = W.plane_c2(4096 * 40 + 5, 1, seed=3)
    sq.debug_set_fault(1, 17, 3_000_000)   # tile 17's header withheld; every wait gives up after 3 ms
    try:
        got = gpu_sum(sq, x, 0.0)
        st = sq.get_stats()
    finally:
        sq.debug_set_fault(0, 0, 0)
    assert got != got, got
    assert st["device_status"] == -3, st
    assert st["timeout_site"] == 3, st
    check(sq, x, 0.0, "the call after a timeout")
    check(sq, W.config("c1").x, 0.0, "c1 after a timeout")


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("n", [1, 2, 15, 16, 17, 31, 511, 512, 513, 4095, 4096, 4097, 8191, 12289, 65537])
def test_sizes_ragged(sq, n):
    x = W.plane_c2(n, 1, seed=n)
    check(sq, x, 0.5, f"n={n}")
    check(sq, x, 0.5, f"n={n} misaligned", offset=1)


def test_empty_returns_s0_bits(sq):
    for s0 in [0.0, -0.0, 1.5, -3.25e300, float("inf"), 5e-324]:
        assert_same(gpu_sum(sq, np.zeros(0), s0), s0, f"n=0 s0={s0}")


def test_signed_zero_rules(sq):
    for n in [1, 100, 5000, 9000]:
        check(sq, np.full(n, -0.0), -0.0, f"all -0 n={n}")
        x = np.full(n, -0.0)
        x[n // 2] = 0.0
        check(sq, x, -0.0, f"one +0 n={n}")
        check(sq, np.full(n, -0.0), 0.0, f"+0 start n={n}")
    x = np.zeros(20000)
    x[12345] = 1.0
    x[12346] = -1.0
    check(sq, x, 0.0, "cancel to +0")


def test_ties_dense(sq):
    rng = np.random.default_rng(1)
    for e in [-53, -52, -30, 0, 40]:
        k = rng.integers(0, 8, size=30000).astype(np.float64)
        x = np.ldexp(k, e)
        check(sq, x, 1.0 if e < 0 else float(2.0 ** (e + 52)), f"ties e={e}")


def test_subnormal_and_tiny(sq):
    rng = np.random.default_rng(2)
    x = rng.integers(0, 1 << 20, size=50000).astype(np.float64) * 5e-324
    check(sq, x, 0.0, "subnormal terms")
    x = x * np.where(rng.random(50000) < 0.3, -1.0, 1.0)
    check(sq, x, 0.0, "signed subnormal terms")
    check(sq, x, 2.0 ** -1022, "from the smallest normal")


def test_near_overflow(sq):
    rng = np.random.default_rng(3)
    x = np.ldexp(1.0 + rng.random(20000), 1000 + rng.integers(0, 20, 20000))
    check(sq, x, 0.0, "toward overflow (ends at inf)")
    x2 = np.ldexp(1.0 + rng.random(20000), 990)
    check(sq, x2, 1.5e308, "overflow mid-way")
    x3 = -x2
    check(sq, x3, -1.5e308, "negative overflow")


def test_non_finite(sq):
    x = W.plane_c2(9000, 1, seed=9)
    for pos, v in [(0, np.inf), (4000, -np.inf), (8999, np.nan), (100, np.inf)]:
        y = x.copy()
        y[pos] = v
        check(sq, y, 0.0, f"{v} at {pos}")
    y = x.copy()
    y[10] = np.inf
    y[7000] = -np.inf
    check(sq, y, 0.0, "inf then -inf")
    check(sq, x, np.inf, "inf start")
    check(sq, x, np.nan, "nan start")


def test_negative_and_cancelling_sums(sq):
    rng = np.random.default_rng(4)
    x = -W.plane_c3(256, 64, zero_rows=2)
    check(sq, x, 0.0, "negated c3")
    y = rng.standard_normal(200000) * np.ldexp(1.0, rng.integers(-10, 10, 200000))
    check(sq, y, 0.0, "random walk")
    z = np.concatenate([np.full(10000, 1.0), np.full(10000, -1.0), rng.random(10000)])
    check(sq, z, 0.0, "up, down, up")


def test_walk_ranges_full_of_items(sq):
    """A signed random walk crosses zero again and again, so most tiles carry
    item lists and a walk range can hold more steps than its slot (the range
    is then read from x).  Prefixes of several lengths, ragged tails and a
    partial last range included."""
    rng = np.random.default_rng(4)
    y = rng.standard_normal(200000) * np.ldexp(1.0, rng.integers(-10, 10, 200000))
    for n in [188284, 188285, 150000, 200000, 4096 * 40, 4096 * 40 + 1]:
        check(sq, y[:n], 0.0, f"random walk prefix {n}")


def test_wide_exponent_mix(sq):
    rng = np.random.default_rng(5)
    x = np.ldexp(rng.random(100000), rng.integers(-1074, 1000, 100000)) * np.where(
        rng.random(100000) < 0.5, -1.0, 1.0)
    check(sq, x, 0.0, "wide mix")


def test_stream_and_repeats(sq):
    """Many calls on a side stream, across the tag wrap (255 calls)."""
    s = torch.cuda.Stream()
    rng = np.random.default_rng(6)
    planes = [W.plane_c2(int(n), 1, seed=int(n)) for n in rng.integers(1, 40000, 12)]
    dev = [torch.from_numpy(p).cuda() for p in planes]
    wants = [oracle.seqsum(p, 0.25) for p in planes]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        outs = []
        for it in range(300):
            k = it % len(planes)
            outs.append((k, sq.seqsum_f64(dev[k], 0.25, stream=s)))
    s.synchronize()
    for k, o in outs:
        assert_same(o.item(), wants[k], f"repeat plane {k}")


def test_crossing_at_every_term_reads_the_range_from_x(sq):
    """A running sum that crosses a power of two at every term (1.0, 0.5,
    1.0, ...): every row's plan range spans a power of two, so every row is
    a raw item and a walk range holds more steps than its slot -- the walk
    reads that range's terms from x itself, and the bits still match the
    loop's."""
    n = 32 * 4096 * 2
    x = np.empty(n)
    x[0] = 1.0
    x[1::2] = -0.5
    x[2::2] = 0.5
    st = check(sq, x, 0.0, "alternating crossings")
    assert st["ranges_from_x"] > 0, st


# ------------------------------------------------------------ plan independence

@pytest.mark.parametrize("mode", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("name", ["c2", "c3", "c5"])
def test_forced_plans_give_the_same_bits(sq, mode, name):
    """Research-1433, finding 5: plans one binade too high, "all zero", one
    fixed binade, every chunk term by term, and random neighbours must all
    give the oracle's bits."""
    wl = W.config(name, scale_div=12)
    old = sq.debug_set_plan(mode)
    try:
        check(sq, wl.x, 0.0, f"{name} plan {mode}")
    finally:
        sq.debug_set_plan(old)


# ------------------------------------------------------------ batched edge cases

def test_batched_ragged_and_empty(sq):
    rng = np.random.default_rng(7)
    lens = [0, 1, 17, 0, 4096, 4097, 5, 0, 12000, 1, 33333, 0]
    parts = [W.plane_c2(max(n, 1), 1, seed=i)[:n] for i, n in enumerate(lens)]
    x = np.concatenate(parts)
    offs = np.zeros(len(lens) + 1, dtype=np.int64)
    offs[1:] = np.cumsum(lens)
    s0s = rng.standard_normal(len(lens))
    s0s[3] = -0.0
    wl = W.Workload("ragged", x, offs, s0s)
    want = oracle.seqsum_batched(x, offs, s0s)
    for sized in [False, True]:
        got = _batched(sq, wl, sized)
        for k in range(len(lens)):
            assert_same(got[k], want[k], f"ragged sum {k} (len {lens[k]})")


def many_sums(seed=11, nsums=700):
    """nsums sums whose lengths cover tile counts from 0 to 40 and one of
    about 300 tiles, in shuffled order, over a 2^U * mant plane (every sum
    crosses binades from its own start)."""
    rng = np.random.default_rng(seed)
    kinds = [0, 1, 15, 16, 17, 4095, 4096, 4097, 8195, 20000, 70000, 163839]
    lens = [int(v) for v in rng.choice(kinds, size=nsums - 1)] + [300 * 4096 + 5]
    rng.shuffle(lens)
    offs = np.zeros(nsums + 1, dtype=np.int64)
    offs[1:] = np.cumsum(lens)
    x = W.plane_c3(int(offs[-1]), 1, seed=seed, zero_rows=0)
    s0s = rng.standard_normal(nsums)
    s0s[::50] = 0.0
    s0s[7] = -0.0
    return W.Workload("many", x, offs, s0s), lens


def test_batched_many_sums_in_mixed_size_order(sq):
    """The sums are streamed and walked in size order, smaller first (the
    set-up kernel sorts them 256 at a time); every result must still land at
    its own index with the oracle's bits."""
    wl, lens = many_sums()
    want = oracle.seqsum_batched(wl.x, wl.offsets, wl.s0)
    for sized in [False, True]:
        got = _batched(sq, wl, sized)
        for k in range(len(lens)):
            assert_same(got[k], want[k], f"sum {k} of {len(lens)} (len {lens[k]}, sized {sized})")
    assert sq.get_stats()["device_status"] == 0


def test_batched_offset_start(sq):
    x = W.plane_c3(200, 100, zero_rows=3)
    offs = np.array([1000, 1000, 5003, 9000, 20000], dtype=np.int64)
    s0s = np.array([1.0, 2.0, -3.0, 0.0])
    wl = W.Workload("offset", x, offs, s0s)
    want = oracle.seqsum_batched(x, offs, s0s)
    got = _batched(sq, wl, True)
    for k in range(4):
        assert_same(got[k], want[k], f"offset sum {k}")


def test_batched_bad_offsets_are_reported(sq):
    x = torch.zeros(100, dtype=torch.float64, device="cuda")
    offs = torch.tensor([0, 50, 40, 100], dtype=torch.int64, device="cuda")
    s0s = torch.zeros(3, dtype=torch.float64, device="cuda")
    outs = sq.seqsum_f64_batched_sized(x, offs, s0s)
    torch.cuda.synchronize()
    assert torch.isnan(outs).all()
    st = sq.get_stats()
    assert st["device_status"] == -6
    # the library stays usable
    check(sq, W.plane_c2(1000, 1, seed=1), 0.0, "after bad offsets")


def test_negative_start_crossing_zero(sq):
    """Sums that start negative and cross zero: the running value changes
    sign and runs through many binades (random sub-ranges of a c3 plane)."""
    x = W.plane_c3(200, 100, zero_rows=3)
    rng = np.random.default_rng(11)
    for _ in range(120):
        n = int(rng.integers(1, 6000))
        a = int(rng.integers(0, len(x) - n))
        s0 = float(rng.choice([-3.0, -1.0, -0.25, -7.5, -10.0, 2.0]))
        check(sq, x[a:a + n], s0, f"[{a}:{a + n}] s0={s0}")

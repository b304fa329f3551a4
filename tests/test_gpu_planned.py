"""Parity of the planned calls (a plan kept from one frame to the next) with
the oracle, bit for bit, whatever the frames hold: the same frame again, a
frame close to the one before, an unrelated frame, every binade moved, a
size change, forced wrong plans, and more calls than the 8-bit call tag has
values.  Research-1433, Open questions (throughput): keep the previous
frame's plan and form again only the chunks whose plan changed; finding 5:
the plan can only cost time, never bits.
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


def frame(sq, plan, x, s0=0.0, what="", offset=0):
    """One planned call on x (shifted by `offset` doubles in its buffer),
    checked against the oracle; returns the call's counters."""
    want = oracle.seqsum(x, s0)
    sq.get_stats()
    buf = torch.zeros(len(x) + offset, dtype=torch.float64, device="cuda")
    if len(x):
        buf[offset:] = torch.from_numpy(np.ascontiguousarray(x))
    out = plan(buf[offset:], s0)
    torch.cuda.synchronize()
    assert_same(out.item(), want, what)
    st = sq.get_stats()
    assert st["device_status"] == 0, st
    return st


def noisy(x, seed, rel):
    """x with every term scaled by its own factor in [1 - rel, 1 + rel]
    (a next frame close to this one)."""
    u = W.uniform53(W.draws_u64(seed, 7, len(x)))
    return x * (1.0 + rel * (2.0 * u - 1.0))


def test_same_frame_again_reforms_nothing(sq):
    wl = W.config("c3")
    x, s0 = wl.x, float(wl.s0[0])
    ntiles = (len(x) + 4095) // 4096
    with sq.SeqsumPlan() as plan:
        st = frame(sq, plan, x, s0, "first frame")
        assert st["tiles"] == ntiles and st["tiles_redone"] == 0
        for k in range(3):
            st = frame(sq, plan, x, s0, f"same frame {k}")
            # one unit a tile, none formed again: the stored plan is the new one
            assert st["tiles"] == ntiles and st["tiles_redone"] == 0, st


@pytest.mark.parametrize("name", ["c3", "c5", "c2"])
def test_close_frames_reform_few_tiles(sq, name):
    wl = W.config(name)
    x, s0 = wl.x, float(wl.s0[0])
    ntiles = (len(x) + 4095) // 4096
    with sq.SeqsumPlan() as plan:
        frame(sq, plan, x, s0, "first")
        for k in range(3):
            xk = noisy(x, 100 + k, 2.0 ** -7)
            st = frame(sq, plan, xk, s0, f"{name} noisy frame {k}")
            assert st["tiles_redone"] <= ntiles // 4, st


def test_frames_unlike_the_one_before(sq):
    """An unrelated frame, then every term doubled (every binade moves up
    one, so no tile's stored plan holds), then scaled by 1 + 2^-10 (the
    crossings move a little), then the first frame again."""
    a = W.config("c3")
    x, s0 = a.x, float(a.s0[0])
    xb = W.plane_c3(seed=33)   # the same recipe, other draws
    ntiles = (len(x) + 4095) // 4096
    with sq.SeqsumPlan() as plan:
        frame(sq, plan, x, s0, "first")
        frame(sq, plan, xb, s0, "unrelated")
        frame(sq, plan, x, s0, "first again")
        st = frame(sq, plan, 2.0 * x, 2.0 * s0, "doubled")
        assert st["tiles_redone"] > ntiles // 2, st
        frame(sq, plan, x * (1.0 + 2.0 ** -10), s0, "scaled")
        frame(sq, plan, x, s0, "first once more")


def test_size_changes_and_small_frames(sq):
    """A plan follows n: a new size forms its plan first, then reuses it;
    sizes below one row (no TMA), one tile, a ragged tail, an empty frame,
    and a start that is not 16-byte aligned."""
    x3 = W.config("c1").x
    with sq.SeqsumPlan() as plan:
        for n in [0, 0, 1, 15, 16, 17, 4095, 4096, 4097, 50000, 50000, 12345, len(x3), len(x3)]:
            xs = x3[:n].copy()
            frame(sq, plan, xs, 0.25, f"n={n}")
            frame(sq, plan, noisy(xs, n, 2.0 ** -6), 0.25, f"n={n} noisy")
        frame(sq, plan, x3, -1.5, "misaligned", offset=1)
        frame(sq, plan, x3, -1.5, "misaligned again", offset=1)


def test_signed_and_special_frames(sq):
    """Signed frames whose sum changes sign, a frame with an infinity, and
    with a NaN, between ordinary ones."""
    wl = W.config("c5", scale_div=4)
    x = wl.x.copy()
    with sq.SeqsumPlan() as plan:
        frame(sq, plan, x, 0.0, "signed")
        frame(sq, plan, -x, 0.0, "negated")
        frame(sq, plan, x - np.float64(x.mean()), 0.0, "centred")
        y = x.copy()
        y[len(y) // 3] = np.inf
        frame(sq, plan, y, 0.0, "inf")
        y[len(y) // 2] = np.nan
        frame(sq, plan, y, 0.0, "nan")
        frame(sq, plan, x, 0.0, "signed again")


@pytest.mark.parametrize("mode", [1, 5])
def test_forced_wrong_plans_stay_exact(sq, mode):
    """Forced plans (one binade too high; random neighbouring binades) on
    the tiles formed on the stored plan and on those formed again."""
    wl = W.config("c3", scale_div=16)
    x, s0 = wl.x, float(wl.s0[0])
    old = sq.debug_set_plan(mode)
    try:
        with sq.SeqsumPlan() as plan:
            frame(sq, plan, x, s0, f"mode {mode} first")
            frame(sq, plan, x, s0, f"mode {mode} same")
            frame(sq, plan, noisy(x, 9, 2.0 ** -5), s0, f"mode {mode} noisy")
    finally:
        sq.debug_set_plan(old)


def test_more_calls_than_tags(sq):
    """300 planned calls (the call tag wraps past 255) alternating between
    two frames and a third close to the first, with plain calls between."""
    wl = W.config("c1")
    x = wl.x[:60000].copy()
    frames = [x, noisy(x, 1, 2.0 ** -8), 1.5 * x]
    want = [oracle.seqsum(f, 0.5) for f in frames]
    dev = [torch.from_numpy(f).cuda() for f in frames]
    outs = torch.empty(300, dtype=torch.float64, device="cuda")
    with sq.SeqsumPlan() as plan:
        sq.get_stats()
        for i in range(300):
            plan(dev[i % 3], 0.5, out=outs[i:i + 1])
            if i % 37 == 0:
                sq.seqsum_f64(dev[0], 0.5)
        torch.cuda.synchronize()
        st = sq.get_stats()
    assert st["device_status"] == 0, st
    got = outs.cpu().numpy()
    for i in range(300):
        assert_same(got[i], want[i % 3], f"call {i}")


def test_two_plans_on_one_stream(sq):
    """Two plans used in turn keep their own stored plans."""
    a = W.config("c2").x
    b = W.config("c1").x
    with sq.SeqsumPlan() as pa, sq.SeqsumPlan() as pb:
        for k in range(3):
            frame(sq, pa, a, 0.0, f"a {k}")
            frame(sq, pb, b, 0.0, f"b {k}")
            frame(sq, pa, noisy(a, k, 2.0 ** -8), 0.0, f"a noisy {k}")

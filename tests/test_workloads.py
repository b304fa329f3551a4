"""The seeded generators: fixed bytes, the configured shapes and value ranges."""
import numpy as np
import pytest

import workloads as W


def test_splitmix64_reference_values():
    # splitmix64 started from state 0 (Vigna's reference implementation):
    # the first outputs are these published constants.
    z = np.array([0], dtype=np.uint64)
    outs = []
    state = np.uint64(0)
    for _ in range(3):
        with np.errstate(over="ignore"):
            state = state + W.GAMMA
        outs.append(int(W._mix(np.array([state], dtype=np.uint64))[0]))
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert W.mix_scalar(int(W.GAMMA)) == 0xE220A8397B1DCDAF
    del z


def test_draws_are_deterministic_and_counter_based():
    a = W.draws_u64(7, 3, 1000)
    b = W.draws_u64(7, 3, 600, start=400)
    assert np.array_equal(a[400:], b)
    assert not np.array_equal(W.draws_u64(7, 4, 10), a[:10])


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c5"])
def test_small_configs_shapes(name):
    wl = W.config(name, scale_div=8)
    w, h = wl.shape[0]
    assert len(wl.x) == w * h and wl.nsums == 1
    assert wl.x.dtype == np.float64 and np.all(np.isfinite(wl.x))
    assert wl.checksum() == W.config(name, scale_div=8).checksum()


def test_c1_ranges():
    x = W.plane_c1()
    assert len(x) == 186624
    edge = W.edge_mask(576, 324)
    assert np.all((x[~edge] >= 32768.0) & (x[~edge] < 65536.0))
    assert np.all((x[edge] > 0) & (x[edge] < 65535.0))


def test_c2_multiples_of_2m53():
    x = W.plane_c2(192, 108)
    nz = x[x != 0]
    assert np.all((nz > 0) & (nz <= 0.5))
    k = nz * 2.0 ** 53
    assert np.all(k == np.floor(k))
    frac0 = np.mean(x == 0)
    assert 0.07 < frac0 < 0.13


def test_c3_structure():
    x = W.plane_c3(384, 216, zero_rows=6)
    assert np.all(x[: 6 * 384] == 0)
    rest = x[6 * 384:]
    nz = rest[rest != 0]
    assert nz.min() >= 2.0 ** -40 and nz.max() < 2.0
    assert 0.005 < np.mean(rest == 0) < 0.02


def test_c5_signed():
    x = W.plane_c5(384, 216)
    assert (x < 0).any() and (x > 0).any()
    assert np.all(np.abs(x) <= 65536.0)


def test_c4_layout():
    wl = W.config("c4", scale_div=16)
    assert wl.nsums == 108
    sizes = np.diff(wl.offsets)
    assert np.all(sizes > 0)
    assert len(wl.x) == wl.offsets[-1]
    full = sum(w * h for (w, h) in W.C4_SCALES) * 18
    assert full == 199_018_080

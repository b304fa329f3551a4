"""Interleaved sums (seqsum_f64_strided) against the oracle, bit for bit: the
lcs variant's four sums per window (ADR-1464, Decision) over a 1920x1080
plane, other strides, ragged and empty sums, and the float means."""
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


def u64(a):
    return np.asarray(a, dtype=np.float64).view(np.uint64)


def u32(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def check(sq, x, stride, s0s):
    want, want_means = oracle.seqsum_strided(x, stride, s0s)
    outs, means = sq.seqsum_f64_strided(torch.from_numpy(x).cuda(), stride, torch.from_numpy(s0s).cuda(),
                                        means=True)
    torch.cuda.synchronize()
    got, gm = outs.cpu().numpy(), means.cpu().numpy()
    for k in range(stride):
        if not (got[k] != got[k] and want[k] != want[k]):
            assert u64(got[k]) == u64(want[k]), (stride, k, got[k], want[k])
        if not (gm[k] != gm[k] and want_means[k] != want_means[k]):
            assert u32(gm[k]) == u32(want_means[k]), (stride, k, gm[k], want_means[k])
    st = sq.get_stats()
    assert st["device_status"] == 0, st


def test_lcs_four_sums_per_window(sq):
    """1920x1080 windows, four interleaved sums each: the value (c2-style
    terms, ties in [1, 2)), and three factors of the 2^U style."""
    n = 1920 * 1080
    x = np.empty(4 * n)
    x[0::4] = W.plane_c2(1920, 1080, seed=41)
    x[1::4] = W.plane_pow2(n, 42, -30, 2, stream=5)
    x[2::4] = W.plane_pow2(n, 43, -20, 0, stream=5)
    x[3::4] = -W.plane_pow2(n, 44, -40, 0, stream=5)
    check(sq, x, 4, np.array([0.0, 1.0, 0.0, -0.5]))


@pytest.mark.parametrize("stride", [1, 3, 16, 64])
@pytest.mark.parametrize("n", [0, 1, 17, 4097, 50000])
def test_strides_and_ragged(sq, stride, n):
    x = W.plane_c2(max(n * stride, 1), 1, seed=stride * 1000 + n)[:n * stride]
    s0s = np.linspace(-1.0, 1.0, stride)
    check(sq, x, stride, s0s)


def test_strided_rejects_bad_arguments(sq):
    import ctypes
    L = sq.lib()
    assert L.seqsum_f64_strided(None, 4, 0, ctypes.c_void_p(256), ctypes.c_void_p(256), None, None) == -1
    assert L.seqsum_f64_strided(ctypes.c_void_p(256), 4, 65, ctypes.c_void_p(256), ctypes.c_void_p(256), None,
                                None) == -1
    assert L.seqsum_f64_strided(ctypes.c_void_p(256), -1, 4, ctypes.c_void_p(256), ctypes.c_void_p(256), None,
                                None) == -1

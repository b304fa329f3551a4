"""seqsum_f64_static, the entry point that allocates nothing: it must give the
bits of seqsum_f64 (and of the oracle) call after call, and refuse sizes
above its maximum before any CUDA call.  This file is collected last, so the
GPU test runs both alone and after every other test in the session."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")


def bits(v):
    return np.float64(v).view(np.uint64).item()


def test_static_refuses_sizes_above_its_maximum():
    import parity_binade_chunked_gb300 as sq
    L = sq.lib()
    too_many = sq.STATIC_MAX_TERMS + 1
    # a non-null x that is never read: the size is refused first
    assert L.seqsum_f64_static(ctypes.c_void_p(256), too_many, 0.0, ctypes.c_void_p(256), None) == -5
    assert L.seqsum_f64_static(None, -1, 0.0, ctypes.c_void_p(256), None) == -1
    assert L.seqsum_f64_static(None, 3, 0.0, ctypes.c_void_p(256), None) == -1


@pytest.mark.gpu
def test_static_matches_seqsum_f64_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import parity_binade_chunked_gb300 as sq
    cases = [
        (W.plane_c2(1920, 1080, seed=21), 0.0),                      # 2,073,600 terms, under the maximum
        (W.plane_c3(640, 480, seed=22, zero_rows=8), -3.0),          # crosses zero, many binades
        (W.plane_c2(sq.STATIC_MAX_TERMS, 1, seed=23), 1.5),          # exactly the maximum
        (W.plane_c2(4097, 1, seed=24), 0.25),                        # a ragged tail
    ]
    for x, s0 in cases:
        want = oracle.seqsum(x, s0)
        xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        ref = sq.seqsum_f64(xd, s0)
        a = sq.seqsum_f64_static(xd, s0)
        b = sq.seqsum_f64_static(xd, s0)                               # a second call in a row
        torch.cuda.synchronize()
        got = [bits(v.item()) for v in (ref, a, b)]
        assert got == [bits(want)] * 3, (len(x), s0, got, bits(want))

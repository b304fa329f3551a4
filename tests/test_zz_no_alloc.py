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


@pytest.mark.gpu
def test_static_many_calls_misaligned_and_no_device_allocation():
    """130 calls in a row (past the 255-call tag cycle when the session's
    other calls are counted), a plane that starts one double past an aligned
    address (no tensor map: the rows are read with plain loads), and the
    device's free memory unchanged across all of them."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import parity_binade_chunked_gb300 as sq
    x = W.plane_c3(512, 300, seed=25, zero_rows=4)
    buf = torch.zeros(len(x) + 1, dtype=torch.float64, device="cuda")
    buf[1:] = torch.from_numpy(x)
    xv = buf[1:]                                       # 8 bytes past a 256-byte aligned start
    assert xv.data_ptr() % 16 == 8
    want = bits(oracle.seqsum(x, 0.5))
    outs = torch.empty(130, dtype=torch.float64, device="cuda")
    sq.seqsum_f64_static(xv, 0.5, out=outs[0:1])      # the first call sets the scratch up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for i in range(130):
        sq.seqsum_f64_static(xv, 0.5, out=outs[i:i + 1])
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    got = outs.cpu().numpy().view(np.uint64)
    assert all(int(g) == want for g in got), [hex(int(g)) for g in got[:4]]
    assert free1 == free0, (free0, free1)

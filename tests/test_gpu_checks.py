"""The self-checking build (-DSEQSUM_CHECKS): every bound the kernel relies
on is tested on the device, and the first that fails is recorded.  A fresh
interpreter loads that build (the library is chosen when the package is
first imported) and runs workloads, a batched call and a forced plan; no
check may fail and every result must be the oracle's."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import numpy as np, torch
import oracle, workloads as W
import parity_binade_chunked_gb300 as sq
assert "check" in sq.lib_path(), sq.lib_path()
def bits(v): return np.float64(v).view(np.uint64).item()
cases = [(W.config("c1").x, 0.0), (W.config("c3", scale_div=2).x, 0.0), (W.config("c5", scale_div=2).x, 0.0),
         (W.plane_c2(4097, 1, seed=5), 0.5), (W.plane_c3(256, 64, zero_rows=2) * -1.0, 0.0)]
for x, s0 in cases:
    got = sq.seqsum_f64(torch.from_numpy(x).cuda(), s0).item()
    assert bits(got) == bits(oracle.seqsum(x, s0)), len(x)
    st = sq.get_stats()
    assert st["device_status"] == 0 and st["check_site"] == 0, st
wl = W.config("c4", scale_div=8)
outs = sq.seqsum_f64_batched_sized(torch.from_numpy(wl.x).cuda(), torch.from_numpy(wl.offsets).cuda(),
                                   torch.from_numpy(wl.s0).cuda()).cpu().numpy()
want = oracle.seqsum_batched(wl.x, wl.offsets, wl.s0)
assert [bits(v) for v in outs] == [bits(v) for v in want]
st = sq.get_stats()
assert st["device_status"] == 0 and st["check_site"] == 0, st
sq.debug_set_plan(5)
x = W.config("c2", scale_div=12).x
got = sq.seqsum_f64(torch.from_numpy(x).cuda(), 0.0).item()
assert bits(got) == bits(oracle.seqsum(x, 0.0))
st = sq.get_stats()
assert st["check_site"] == 0, st
print("checks ok")
"""


def test_self_checking_build_passes_its_checks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, SEQSUM_CHECKS="1")
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "checks ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])

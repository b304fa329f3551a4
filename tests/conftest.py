import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: longer CPU test")


def load_golden(name):
    """Parse a `name | s0 | terms | expected` fixture under tests/golden/."""
    path = os.path.join(ROOT, "tests", "golden", name)
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [p.strip() for p in line.split("|")]
            label, s0, terms, expected = parts[:4]
            xs = [float.fromhex(t) if "0x" in t else float(t)
                  for t in terms.split(",") if t.strip()] if terms else []
            s0v = float.fromhex(s0) if "0x" in s0 else float(s0)
            ev = float.fromhex(expected) if "0x" in expected else float(expected)
            rows.append((label, s0v, xs, ev))
    return rows


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()
    return oracle


# With SEQSUM_WATCHDOG=<seconds>, a GPU test still running after that long
# prints the library's device counters (read without waiting for the call)
# and ends the process, instead of leaving a call stuck.
@pytest.fixture(autouse=True)
def _watchdog(request):
    limit = float(os.environ.get("SEQSUM_WATCHDOG", "0") or 0)
    if limit <= 0 or request.node.get_closest_marker("gpu") is None:
        yield
        return
    import threading

    def fire():
        try:
            import parity_binade_chunked_gb300 as sq
            print(f"\nWATCHDOG {request.node.nodeid}: counters {sq.debug_counters()}", flush=True)
        except Exception as e:          # diagnostics only
            print("WATCHDOG failed:", e, flush=True)
        os._exit(3)

    timer = threading.Timer(limit, fire)
    timer.daemon = True
    timer.start()
    yield
    timer.cancel()

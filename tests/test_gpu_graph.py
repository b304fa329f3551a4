"""Calls captured into a CUDA graph and replayed over new inputs.  Each
launch takes its call tag from a device counter that the kernel advances
itself, so a replay never mistakes the words of the replay before for its
own; every replay must give the oracle's bits for the data then in the
buffer.
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


def frames(n):
    """Three planes of n terms: c2's recipe, the same scaled per term, and c3's."""
    a = W.config("c2").x[:n].copy()
    u = W.uniform53(W.draws_u64(77, 7, n))
    b = a * (1.0 + 2.0 ** -6 * (2.0 * u - 1.0))
    c = W.config("c3").x[:n].copy()
    return [a, b, c, b, a]


def replay_check(call, xb, out, fr, s0s):
    for k, f in enumerate(fr):
        xb.copy_(torch.from_numpy(f))
        torch.cuda.synchronize()
        call()
        torch.cuda.synchronize()
        got = out.cpu().numpy().reshape(-1)
        for j, s0 in enumerate(s0s):
            want = oracle.seqsum(f if len(s0s) == 1 else f[j * (len(f) // len(s0s)):(j + 1) * (len(f) // len(s0s))],
                                 s0)
            assert bits(got[j]) == bits(want), f"replay {k}, sum {j}: {got[j]!r} vs {want!r}"


@pytest.mark.parametrize("entry", ["seqsum_f64", "seqsum_f64_static"])
def test_single_sum_graph_replays(sq, entry):
    n = 1 << 20 if entry == "seqsum_f64_static" else 1920 * 1080
    fr = frames(n)
    s = torch.cuda.Stream()
    xb = torch.empty(n, dtype=torch.float64, device="cuda")
    out = torch.empty(1, dtype=torch.float64, device="cuda")
    fn = getattr(sq, entry)
    with torch.cuda.stream(s):
        xb.copy_(torch.from_numpy(fr[0]))
        fn(xb, 0.5, out=out, stream=s)   # the workspace and the tensor map exist before the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(xb, 0.5, out=out, stream=s)
    replay_check(g.replay, xb, out, fr, [0.5])


def test_batched_graph_replays(sq):
    n, k = 4 * 200000, 4
    fr = frames(n)
    s = torch.cuda.Stream()
    xb = torch.empty(n, dtype=torch.float64, device="cuda")
    offs = torch.tensor([j * (n // k) for j in range(k + 1)], dtype=torch.int64, device="cuda")
    s0s = [0.0, -1.0, 2.5, 1e-3]
    s0d = torch.tensor(s0s, dtype=torch.float64, device="cuda")
    outs = torch.empty(k, dtype=torch.float64, device="cuda")
    with torch.cuda.stream(s):
        xb.copy_(torch.from_numpy(fr[0]))
        sq.seqsum_f64_batched_sized(xb, offs, s0d, outs=outs, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sq.seqsum_f64_batched_sized(xb, offs, s0d, outs=outs, stream=s)
    replay_check(g.replay, xb, outs, fr, s0s)


def test_many_replays_cross_the_tag_wrap(sq):
    """300 replays (the 8-bit call tag wraps) alternating two planes."""
    n = 150000
    fr = frames(n)[:2]
    want = [oracle.seqsum(f, 0.0) for f in fr]
    s = torch.cuda.Stream()
    xa = torch.from_numpy(fr[0]).cuda()
    xbb = torch.from_numpy(fr[1]).cuda()
    xb = torch.empty(n, dtype=torch.float64, device="cuda")
    out = torch.empty(1, dtype=torch.float64, device="cuda")
    with torch.cuda.stream(s):
        xb.copy_(xa)
        sq.seqsum_f64(xb, 0.0, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sq.seqsum_f64(xb, 0.0, out=out, stream=s)
    res = torch.empty(300, dtype=torch.float64, device="cuda")
    with torch.cuda.stream(s):
        for i in range(300):
            xb.copy_(xa if i % 2 == 0 else xbb)
            g.replay()
            res[i:i + 1].copy_(out)
    s.synchronize()
    got = res.cpu().numpy()
    for i in range(300):
        assert bits(got[i]) == bits(want[i % 2]), f"replay {i}"

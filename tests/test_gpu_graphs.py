"""The library's calls inside CUDA graphs: a chain of calls captured once on a
stream (each op warmed up first, so every one-time attribute is already set)
replays with new input data each time and gives the oracle's results bit for
bit; ap_check, which synchronises, runs after the replay."""

import numpy as np
import pytest

import synth
from gpu_util import assert_bits, device, lib, reset_debug, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture
def ap():
    ap = lib()
    reset_debug(ap)
    yield ap
    reset_debug(ap)


def test_graph_of_every_op(ap, orc):
    import torch

    dev = device()
    n = 1 << 20
    rows, cols = 64, 4
    x = torch.empty(n, device=dev)
    A = torch.empty(rows * cols, device=dev)
    y1, y2, y3, y4, y5 = (torch.empty(n, device=dev) for _ in range(5))
    B = torch.empty_like(A)
    c = synth.coeffs_np(8).tolist()
    s = torch.cuda.Stream()

    def chain():
        ap.ap_row_roll(A, B, rows, cols, 1, s)                  # one CTA, cp.async.cg
        ap.ap_scale(x, y1, n // 256, 256, 2.0, 2, s)           # ring
        ap.ap_poly(y1, y2, n, c, 8, 3, s)                      # ring, reads the scale's output
        ap.ap_cluster_exchange(y2, y3, n, 4, 16384, s)          # cluster hand-off
        ap.ap_cluster_all_to_all(y3, y4, n, 8, 32768, s)        # cluster all-to-all
        ap.ap_row_roll(y4, y5, n // 4, 4, -3, s)                # ring row shift

    with torch.cuda.stream(s):
        x.copy_(synth.uniform_pm1_torch(1, n, dev))
        A.copy_(torch.arange(rows * cols, dtype=torch.float32, device=dev))
        chain()  # warm-up outside capture
    s.synchronize()
    assert ap.ap_check(s) == ap.AP_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    for rep in range(3):
        with torch.cuda.stream(s):
            x.copy_(synth.uniform_pm1_torch(100 + rep, n, dev))
            A.copy_(synth.uniform_pm1_torch(200 + rep, rows * cols, dev))
        s.synchronize()
        g.replay()
        s.synchronize()
        assert ap.ap_check(s) == ap.AP_OK
        xh = to_np(x)
        want = orc.row_roll(orc.cluster_all_to_all(orc.cluster_exchange(orc.poly(orc.scale(xh, 2.0),
                                                                                  np.array(c, dtype=np.float32)),
                                                                         4, 16384), 8, 32768).reshape(-1, 4), -3)
        assert_bits(to_np(y5), want.ravel(), f"graph replay {rep}")
        assert_bits(to_np(B), orc.row_roll(to_np(A).reshape(rows, cols), 1).ravel(), f"64x4 roll in graph, {rep}")


def test_graph_of_many_small_rolls(ap, orc):
    """The latency-bound 64 x 4 worked example, 100 calls per graph."""
    import torch

    dev = device()
    A = synth.uniform_pm1_torch(7, 256, dev).reshape(64, 4)
    bufs = [torch.empty_like(A) for _ in range(100)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ap.ap_row_roll(A, bufs[0], 64, 4, 1, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for k, b in enumerate(bufs):
            ap.ap_row_roll(A, b, 64, 4, k, s)
    g.replay()
    s.synchronize()
    assert ap.ap_check(s) == ap.AP_OK
    Ah = to_np(A)
    for k, b in enumerate(bufs):
        assert_bits(to_np(b), orc.row_roll(Ah, k), f"roll by {k} in graph")


def test_graph_of_polynomial_shapes_and_masked_copy(ap, orc):
    """Polynomial launches of every consumer form in one graph (one group at
    depth 3, two groups taking alternate stages at depths 4 and 6, eight
    warps for degree 8 at depth 6) and a masked copy, replayed with new input
    data each time."""
    import torch

    dev = device()
    n = 1 << 20
    x = torch.empty(n, device=dev)
    ys = [torch.empty(n, device=dev) for _ in range(4)]
    m = torch.empty(n, device=dev)
    codes = torch.from_numpy(np.random.default_rng(7).integers(-2, 17, n // 4).astype(np.int8)).to(dev)
    calls = [(32, 3), (32, 4), (128, 6), (8, 6)]
    coeffs = {k: synth.coeffs_np(k) for k, _ in calls}
    s = torch.cuda.Stream()

    def chain():
        for (k, stages), y in zip(calls, ys):
            ap.ap_poly(x, y, n, coeffs[k].tolist(), k, stages, s)
        ap.ap_masked_copy(x, m, n // 4, codes, 3, s)

    with torch.cuda.stream(s):
        x.copy_(synth.uniform_pm1_torch(11, n, dev))
        m.zero_()
        chain()  # warm-up outside capture
    s.synchronize()
    assert ap.ap_check(s) == ap.AP_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    for rep in range(2):
        with torch.cuda.stream(s):
            x.copy_(synth.uniform_pm1_torch(300 + rep, n, dev))
        s.synchronize()
        before = to_np(m).copy()
        g.replay()
        s.synchronize()
        assert ap.ap_check(s) == ap.AP_OK
        xh = to_np(x)
        for (k, stages), y in zip(calls, ys):
            assert_bits(to_np(y), orc.poly(xh, coeffs[k]), f"graph poly K={k} S={stages}, replay {rep}")
        assert_bits(to_np(m), orc.masked_copy(xh, before, to_np(codes)), f"graph masked copy, replay {rep}")

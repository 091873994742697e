"""Stream semantics: calls are ordered on their stream, independent streams
run side by side, and chains of calls on one buffer give the composed result."""

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


def test_chain_on_one_stream(ap, orc):
    """scale -> poly -> roll on a side stream, each reading the previous
    output with no synchronisation in between."""
    import torch

    dev = device()
    rows, cols = 1 << 18, 4
    n = rows * cols
    x = synth.uniform_pm1_torch(21, n, dev)
    a = torch.empty_like(x)
    b = torch.empty_like(x)
    s = torch.cuda.Stream()
    c = synth.coeffs_np(8)
    s.wait_stream(torch.cuda.current_stream())
    ap.ap_scale(x, a, n // 256, 256, 0.5, 3, s)
    ap.ap_poly(a, a, n, c.tolist(), 8, 2, s)  # in place
    ap.ap_row_roll(a, b, rows, cols, 7, s)
    assert ap.ap_check(s) == ap.AP_OK
    want = orc.row_roll(orc.poly(orc.scale(to_np(x), 0.5), c).reshape(rows, cols), 7)
    assert_bits(to_np(b), want, "chained on one stream")


def test_independent_streams(ap, orc):
    import torch

    dev = device()
    n = 1 << 22
    streams = [torch.cuda.Stream() for _ in range(4)]
    xs = [synth.uniform_pm1_torch(100 + i, n, dev) for i in range(4)]
    ys = [torch.empty_like(x) for x in xs]
    torch.cuda.synchronize()
    for i, (st, x, y) in enumerate(zip(streams, xs, ys)):
        if i % 2 == 0:
            ap.ap_scale(x, y, n, 1, float(i + 1), 2 + i, st)
        else:
            ap.ap_cluster_exchange(x, y, n, 4, 16384, st)
    torch.cuda.synchronize()
    assert ap.ap_check() == ap.AP_OK
    for i, (x, y) in enumerate(zip(xs, ys)):
        want = orc.scale(to_np(x), float(i + 1)) if i % 2 == 0 else orc.cluster_exchange(to_np(x), 4, 16384)
        assert_bits(to_np(y), want, f"stream {i}")


def test_many_small_calls(ap, orc):
    """Back-to-back small launches (the 64 x 4 worked example and tiny rings)
    stay correct and report no device error."""
    import torch

    dev = device()
    A = torch.arange(256, dtype=torch.float32, device=dev).reshape(64, 4)
    B = torch.empty_like(A)
    y = torch.empty(1000, device=dev)
    x = synth.uniform_pm1_torch(5, 1000, dev)
    for i in range(200):
        ap.ap_row_roll(A, B, 64, 4, i)
        ap.ap_scale(x, y, 1000, 1, 2.0, 2 + i % 5)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(B), orc.row_roll(to_np(A), 199), "last roll")
    assert_bits(to_np(y), orc.scale(to_np(x), 2.0), "last scale")


def test_binding_follows_torch_current_stream():
    """Calls without a stream argument go to torch's current stream: the
    default one, and the one a `torch.cuda.stream` block selects."""
    import torch

    from async_global_shared_gb300 import _lib

    assert _lib._stream(None) == torch.cuda.current_stream().cuda_stream
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert _lib._stream(None) == side.cuda_stream
    assert _lib._stream(None) == torch.cuda.current_stream().cuda_stream

"""The calls on pinned host buffers: the kernels read and write host memory
over the host link directly (no staging copies), with the same results as on
device memory."""

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


def _pinned(values):
    import torch

    t = torch.empty(values.size, dtype=torch.float32, pin_memory=True)
    t.copy_(torch.from_numpy(values))
    return t


def test_every_op_on_pinned_host_buffers(ap, orc):
    import torch

    n = 1 << 20
    xh = synth.uniform_pm1_np(31, n)
    x = _pinned(xh)
    y = torch.empty(n, dtype=torch.float32, pin_memory=True)
    c = synth.coeffs_np(8)
    cases = [
        ("scale", lambda: ap.ap_scale(x, y, n // 256, 256, 2.0, 2), lambda: orc.scale(xh, 2.0)),
        ("scale S=5", lambda: ap.ap_scale(x, y, n, 1, -0.5, 5), lambda: orc.scale(xh, -0.5)),
        ("roll", lambda: ap.ap_row_roll(x, y, n // 4, 4, 7), lambda: orc.row_roll(xh.reshape(-1, 4), 7).ravel()),
        ("poly", lambda: ap.ap_poly(x, y, n, c.tolist(), 8, 3), lambda: orc.poly(xh, c)),
        ("exchange", lambda: ap.ap_cluster_exchange(x, y, n, 4, 16384), lambda: orc.cluster_exchange(xh, 4, 16384)),
        ("exchange, 256-byte chunks", lambda: ap.ap_cluster_exchange(x, y, n, 4, 256),
         lambda: orc.cluster_exchange(xh, 4, 256)),
        ("all-to-all", lambda: ap.ap_cluster_all_to_all(x, y, n, 8, 32768),
         lambda: orc.cluster_all_to_all(xh, 8, 32768)),
    ]
    for what, call, want in cases:
        y.fill_(float("nan"))
        call()
        assert ap.ap_check() == ap.AP_OK, what
        assert_bits(y.numpy(), want(), f"{what} on pinned host buffers")


def test_host_input_device_output_and_back(ap, orc):
    import torch

    dev = device()
    n = 1 << 22
    xh = synth.uniform_pm1_np(32, n)
    x = _pinned(xh)
    yd = torch.empty(n, device=dev)
    zh = torch.empty(n, dtype=torch.float32, pin_memory=True)
    ap.ap_scale(x, yd, n, 1, 3.0, 2)           # host -> device
    ap.ap_row_roll(yd, zh, n // 4, 4, 1)        # device -> host
    assert ap.ap_check() == ap.AP_OK
    assert_bits(zh.numpy(), orc.row_roll(orc.scale(xh, 3.0).reshape(-1, 4), 1).ravel(), "host -> device -> host")

"""The device-checked ring (AP_DBG_DEVICE_CHECKS): every copy and every
shared/global range the kernels touch is verified in the kernel before use.
Random geometries and every producer/consumer mode run clean (AP_OK) and
still give the oracle's bits."""

import numpy as np
import pytest

import synth
from gpu_util import Guarded, assert_bits, device, lib, reset_debug, to_np
from test_gpu_fuzz import _knobs, _run_op

pytestmark = pytest.mark.gpu


@pytest.fixture
def ap():
    ap = lib()
    reset_debug(ap)
    yield ap
    reset_debug(ap)


@pytest.mark.parametrize("seed", range(4))
def test_checked_ring_random(ap, orc, seed):
    dev = device()
    rng = np.random.default_rng(3000 + seed)
    for case in range(40):
        op = str(rng.choice(["scale", "poly", "roll"]))
        n = int(rng.integers(1, 1 << int(rng.integers(1, 18))))
        in_shift, out_shift = (int(v) for v in rng.integers(0, 4, 2))
        stages = int(rng.integers(2, 7))
        _knobs(ap, rng)
        ap.ap_debug_set(ap.AP_DBG_DEVICE_CHECKS, 1)
        src = Guarded(n, in_shift, dev, fill=synth.uniform_pm1_torch(seed * 77 + case, n, dev))
        out = Guarded(n, out_shift, dev)
        what = f"seed={seed} case={case} op={op} n={n} in+{in_shift} out+{out_shift} S={stages}"
        try:
            want = _run_op(ap, orc, rng, op, src, out, to_np(src.view), n, stages)
        except ap.APError as e:
            assert e.status == ap.AP_ERR_SMEM, what
            reset_debug(ap)
            continue
        st = ap.ap_check()
        assert st == ap.AP_OK, f"{what}: {ap.ap_status_string(st)} at site {ap.ap_debug_get(ap.AP_DBG_LAST_SITE)}"
        assert_bits(to_np(out.view), want, what)
        assert out.intact() and src.intact(), what
        reset_debug(ap)


@pytest.mark.parametrize("variant", ["aligned", "A+4", "B+4", "tensor"])
def test_checked_ring_full_size_roll(ap, orc, variant):
    import torch

    dev = device()
    rows, cols = 1 << 24, 4
    n = rows * cols
    a_shift = 1 if variant == "A+4" else 0
    b_shift = 1 if variant == "B+4" else 0
    abuf = torch.empty(n + 4, dtype=torch.float32, device=dev)
    bbuf = torch.empty(n + 4, dtype=torch.float32, device=dev)
    A = abuf[a_shift:a_shift + n]
    B = bbuf[b_shift:b_shift + n]
    synth.uniform_pm1_torch(9, n, dev, out=A)
    ap.ap_debug_set(ap.AP_DBG_DEVICE_CHECKS, 1)
    if variant == "tensor":
        ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    ap.ap_row_roll(A, B, rows, cols, 3)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(B), orc.row_roll(to_np(A).reshape(rows, cols), 3), f"checked roll {variant}")


def test_checked_scale_and_poly_full_size(ap, orc):
    import torch

    dev = device()
    n = 1 << 26
    x = synth.uniform_pm1_torch(10, n, dev)
    y = torch.empty_like(x)
    ap.ap_debug_set(ap.AP_DBG_DEVICE_CHECKS, 1)
    for stages in (2, 3, 4, 5, 6):
        ap.ap_scale(x, y, n // 256, 256, 2.0, stages)
        assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.scale(to_np(x), 2.0), "checked scale")
    c = synth.coeffs_np(32)
    idx = np.random.default_rng(0).integers(0, n, 1 << 16)
    for stages in (3, 4):  # one consumer group, then two groups taking alternate stages
        y.zero_()
        ap.ap_poly(x, y, n, c.tolist(), 32, stages)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(y)[idx], orc.poly(to_np(x)[idx], c), f"checked poly S={stages} (sampled)")

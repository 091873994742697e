"""ap_autotune: the chosen shape is installed for later calls (and still
gives the oracle's bits); ap_autotune_reset restores the defaults."""

import pytest

import synth
from gpu_util import assert_bits, device, lib, reset_debug, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture
def ap():
    ap = lib()
    reset_debug(ap)
    ap.ap_autotune_reset()
    yield ap
    ap.ap_autotune_reset()
    reset_debug(ap)


def test_autotune_scale_installs_choice(ap, orc):
    import torch

    dev = device()
    n = 1 << 26
    x = synth.uniform_pm1_torch(synth.SEED_SCALE, n, dev)
    scratch = torch.empty_like(x)
    shape = ap.ap_autotune(ap.AP_TUNE_SCALE, x, scratch, n, 2)
    assert shape["gbs"] > 0 and shape["stage_bytes"] >= 8192 and 1 <= shape["ctas_per_sm"] <= 4
    assert shape["stages_per_cta"] in (0, 2, 4, 8)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    y = torch.empty_like(x)
    ap.ap_scale(x, y, n // 256, 256, 2.0, 2)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_RUN) == shape["stages_per_cta"]
    if shape["stages_per_cta"] == 0:
        assert ap.ap_debug_get(ap.AP_DBG_LAST_GRID) == sms * shape["ctas_per_sm"]
    assert ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS) == shape["stage_bytes"] // 4
    assert_bits(to_np(y), orc.scale(to_np(x), 2.0), "scale with the tuned shape")
    ap.ap_autotune_reset()
    ap.ap_scale(x, y, n // 256, 256, 2.0, 2)
    assert ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS) == 16384 // 4  # the built-in default again


def test_autotune_poly_and_roll(ap, orc):
    import torch

    dev = device()
    n = 1 << 26
    x = synth.uniform_pm1_torch(synth.SEED_POLY, n, dev)
    scratch = torch.empty_like(x)
    shape = ap.ap_autotune(ap.AP_TUNE_POLY, x, scratch, n, 3, degree=32)
    assert shape["consumer_warps"] in (8, 12, 16)
    c = synth.coeffs_np(32)
    m = 1 << 20
    y = torch.empty(m, device=dev)
    ap.ap_poly(x[:m], y, m, c.tolist(), 32, 3)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.poly(to_np(x[:m]), c), "poly with the tuned shape")
    shape = ap.ap_autotune(ap.AP_TUNE_ROW_ROLL, x, scratch, n, 3)
    rows = m // 4
    ap.ap_row_roll(x[:m], y, rows, 4, 5)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.row_roll(to_np(x[:m]).reshape(rows, 4), 5).ravel(), "roll with the tuned shape")

"""Bounded waits: a barrier whose expected byte count is inflated never
completes (every real copy still lands), so the kernel's waits give up after
a short limit, record AP_ERR_DEVICE_TIMEOUT for ap_check and return. The
context stays usable: the next normal call is correct. No fault, trap or
hang is involved."""

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


def _inject(ap):
    ap.ap_debug_set(ap.AP_DBG_TIMEOUT_NS, 20_000_000)  # 20 ms
    ap.ap_debug_set(ap.AP_DBG_EXPECT_TX_EXTRA, 16)


def test_ring_wait_times_out_and_recovers(ap, orc):
    import torch

    dev = device()
    assert ap.ap_check() == ap.AP_OK
    n_tiles, tile = 512, 256
    x = synth.uniform_pm1_torch(3, n_tiles * tile, dev)
    y = torch.empty_like(x)
    _inject(ap)
    ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, 4096)
    ap.ap_scale(x, y, n_tiles, tile, 2.0, 3)
    assert ap.ap_check() == ap.AP_ERR_DEVICE_TIMEOUT
    assert ap.ap_check() == ap.AP_OK  # the check cleared the status word
    reset_debug(ap)
    ap.ap_scale(x, y, n_tiles, tile, 2.0, 3)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.scale(to_np(x), 2.0), "after recovery")


@pytest.mark.parametrize("stages", [3, 4])
def test_poly_wait_times_out_and_recovers(ap, orc, stages):
    """The polynomial's 16 consumer warps, as one group (depth 3) and as two
    groups taking alternate stages (depth 4)."""
    import torch

    dev = device()
    assert ap.ap_check() == ap.AP_OK
    n = 64 * 8192
    x = synth.uniform_pm1_torch(5, n, dev)
    y = torch.empty_like(x)
    c = synth.coeffs_np(32)
    _inject(ap)
    ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, 16 * 1024)
    ap.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, 16)
    ap.ap_poly(x, y, n, c.tolist(), 32, stages)
    assert ap.ap_check() == ap.AP_ERR_DEVICE_TIMEOUT
    assert ap.ap_check() == ap.AP_OK
    reset_debug(ap)
    ap.ap_poly(x, y, n, c.tolist(), 32, stages)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.poly(to_np(x), c), f"poly S={stages} after recovery")


@pytest.mark.parametrize("send", [1, 4])
@pytest.mark.parametrize("store,group", [(1, 0), (2, 8), (2, 4), (2, 1)])
def test_exchange_wait_times_out_and_recovers(ap, orc, store, group, send):
    import torch

    dev = device()
    assert ap.ap_check() == ap.AP_OK
    n = 4 * 4096 * 16 // 4
    x = synth.uniform_pm1_torch(4, n, dev)
    y = torch.empty_like(x)
    _inject(ap)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_STORE, store)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, group)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_SEND_SLOTS, send)
    ap.ap_cluster_exchange(x, y, n, 4, 4096)
    assert ap.ap_check() == ap.AP_ERR_DEVICE_TIMEOUT
    reset_debug(ap)
    ap.ap_cluster_exchange(x, y, n, 4, 4096)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.cluster_exchange(to_np(x), 4, 4096), "exchange after recovery")


@pytest.mark.parametrize("send", [0, 1, 4])
@pytest.mark.parametrize("store,group,lanes", [(1, 0, 1), (2, 1, 2), (2, 4, 4)])
def test_all_to_all_wait_times_out_and_recovers(ap, orc, store, group, lanes, send):
    """The all-to-all's bounded waits: no piece is ever loaded (the loader's
    barrier expects bytes that never come), so nothing is pushed between CTAs,
    every wait gives up (receiver warps of a group agree before leaving), and
    the next call runs normally."""
    import torch

    dev = device()
    assert ap.ap_check() == ap.AP_OK
    n = 4 * 4096 * 16 // 4
    x = synth.uniform_pm1_torch(5, n, dev)
    y = torch.empty_like(x)
    _inject(ap)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_STORE, store)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, group)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, lanes)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_SEND_SLOTS, send)
    ap.ap_cluster_all_to_all(x, y, n, 4, 4096)
    assert ap.ap_check() == ap.AP_ERR_DEVICE_TIMEOUT
    reset_debug(ap)
    ap.ap_cluster_all_to_all(x, y, n, 4, 4096)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.cluster_all_to_all(to_np(x), 4, 4096), "all-to-all after recovery")


def test_all_to_all_three_ctas_wait_times_out_and_recovers(ap, orc):
    """The same for clusters of 8 with 4 KiB sub-blocks, which run the
    register-capped three-CTAs-per-SM instantiation."""
    import torch

    dev = device()
    assert ap.ap_check() == ap.AP_OK
    n = 8 * 32768 * 6 // 4
    x = synth.uniform_pm1_torch(6, n, dev)
    y = torch.empty_like(x)
    _inject(ap)
    ap.ap_cluster_all_to_all(x, y, n, 8, 32768)
    assert ap.ap_check() == ap.AP_ERR_DEVICE_TIMEOUT
    reset_debug(ap)
    ap.ap_cluster_all_to_all(x, y, n, 8, 32768)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_STAGES) == 8
    assert_bits(to_np(y), orc.cluster_all_to_all(to_np(x), 8, 32768), "all-to-all after recovery")


def test_batched_exchange_wait_times_out_and_recovers(ap, orc):
    """The batched form's bounded waits (its loader barrier never completes)."""
    import torch

    dev = device()
    assert ap.ap_check() == ap.AP_OK
    n = 4 * 256 * 64 // 4
    x = synth.uniform_pm1_torch(6, n, dev)
    y = torch.empty_like(x)
    _inject(ap)
    ap.ap_cluster_exchange(x, y, n, 4, 256)
    assert ap.ap_check() == ap.AP_ERR_DEVICE_TIMEOUT
    reset_debug(ap)
    ap.ap_cluster_exchange(x, y, n, 4, 256)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 4
    assert_bits(to_np(y), orc.cluster_exchange(to_np(x), 4, 256), "batched exchange after recovery")


def test_bad_arguments_raise(ap):
    import torch

    dev = device()
    x = torch.zeros(1024, device=dev)
    with pytest.raises(ap.APError):
        ap.ap_scale(x, x[4:], 1, 1000, 2.0, 2)  # partial overlap
    with pytest.raises(ap.APError):
        ap.ap_row_roll(x, x, 256, 4, 1)  # roll never in place
    with pytest.raises(TypeError):
        ap.ap_scale(x.double(), x, 1, 1024, 2.0, 2)
    with pytest.raises(TypeError):
        ap.ap_scale(x.cpu(), x, 1, 1024, 2.0, 2)


def test_tensor_map_ring_wait_times_out_and_recovers(ap, orc):
    """The same bounded wait behind the tensor-map producer."""
    import torch

    dev = device()
    assert ap.ap_check() == ap.AP_OK
    rows, cols = 20000, 4
    A = synth.uniform_pm1_torch(6, rows * cols, dev)
    B = torch.empty_like(A)
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    _inject(ap)
    ap.ap_row_roll(A, B, rows, cols, 1)
    assert ap.ap_check() == ap.AP_ERR_DEVICE_TIMEOUT
    reset_debug(ap)
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    ap.ap_row_roll(A, B, rows, cols, 1)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(B), orc.row_roll(to_np(A).reshape(rows, cols), 1), "tensor roll after recovery")


@pytest.mark.parametrize("call", ["ring", "exchange", "all_to_all"])
def test_failed_wait_ends_the_launch_promptly(ap, call):
    """Once one wait gives up, every other role stops: the drains do not wait
    out the limit again for each copy still owed, so a faulted launch ends a
    small multiple of the limit after it starts (0.2 s here; the ring's seven
    stages in flight, or four pusher lanes with several pieces each, would
    otherwise add seconds)."""
    import time

    import torch

    dev = device()
    assert ap.ap_check() == ap.AP_OK
    n = 4 * 4096 * 64 // 4
    x = synth.uniform_pm1_torch(7, n, dev)
    y = torch.empty_like(x)
    ap.ap_debug_set(ap.AP_DBG_TIMEOUT_NS, 200_000_000)
    ap.ap_debug_set(ap.AP_DBG_EXPECT_TX_EXTRA, 16)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    if call == "ring":
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, 4096)
        ap.ap_scale(x, y, n, 1, 2.0, 6)
    elif call == "exchange":
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, 4)
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, 1024)
        ap.ap_debug_set(ap.AP_DBG_CTAS_PER_SM, 3)
        ap.ap_cluster_exchange(x, y, n, 4, 4096)
    else:
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, 4)
        ap.ap_cluster_all_to_all(x, y, n, 4, 4096)
    assert ap.ap_check() == ap.AP_ERR_DEVICE_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert elapsed < 1.5, f"{call}: the faulted launch took {elapsed:.2f} s with a 0.2 s wait limit"
    reset_debug(ap)

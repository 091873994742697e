"""ap_masked_copy against the oracle, bit for bit: per-chunk predicate,
source size (prefix + zero fill) and ignored source."""

import numpy as np
import pytest

import synth
from gpu_util import Guarded, assert_bits, device, lib, reset_debug, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture
def ap():
    ap = lib()
    reset_debug(ap)
    yield ap
    reset_debug(ap)


def _codes(rng, n_chunks, dev):
    import torch

    c = rng.integers(-2, 17, n_chunks).astype(np.int8)
    return c, torch.from_numpy(c).to(dev)


@pytest.mark.parametrize("stages", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("n_chunks", [1, 3, 255, 1024, 1025, 100003])
def test_masked_copy_random_codes(ap, orc, stages, n_chunks):
    dev = device()
    rng = np.random.default_rng(n_chunks + stages)
    x = synth.uniform_pm1_torch(n_chunks, 4 * n_chunks, dev)
    before = synth.uniform_pm1_torch(n_chunks + 1, 4 * n_chunks, dev)
    c_h, c_d = _codes(rng, n_chunks, dev)
    out = Guarded(4 * n_chunks, 0, dev, fill=before)
    ap.ap_masked_copy(x, out.view, n_chunks, c_d, stages)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_PATH) == 5
    assert_bits(to_np(out.view), orc.masked_copy(to_np(x), to_np(before), c_h), f"masked n={n_chunks} S={stages}")
    assert out.intact()


@pytest.mark.parametrize("stages", [2, 3, 6])
@pytest.mark.parametrize("run", [1, 2, 3, 7, 12])
@pytest.mark.parametrize("n_chunks", [1, 1025, 100003])
def test_masked_copy_stage_runs(ap, orc, stages, run, n_chunks):
    """Both schedules: the persistent grid (run 1) and CTAs that each take a
    run of consecutive stages of 1024 chunks, with a short last run, runs
    shorter and longer than the pipeline's depth, and random codes."""
    dev = device()
    rng = np.random.default_rng(7 * n_chunks + run)
    x = synth.uniform_pm1_torch(n_chunks + run, 4 * n_chunks, dev)
    before = synth.uniform_pm1_torch(n_chunks + 2, 4 * n_chunks, dev)
    c_h, c_d = _codes(rng, n_chunks, dev)
    ap.ap_debug_set(ap.AP_DBG_RING_RUN, run)
    out = Guarded(4 * n_chunks, 0, dev, fill=before)
    ap.ap_masked_copy(x, out.view, n_chunks, c_d, stages)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_RUN) == (0 if run == 1 else run)
    assert_bits(to_np(out.view), orc.masked_copy(to_np(x), to_np(before), c_h),
                f"masked n={n_chunks} S={stages} run={run}")
    assert out.intact()


def test_masked_copy_worked_example(ap):
    import torch

    dev = device()
    x = torch.arange(1, 25, dtype=torch.float32, device=dev)
    out = torch.full((24,), -1.0, device=dev)
    codes = torch.tensor([16, -1, 8, 0, -2, 4], dtype=torch.int8, device=dev)
    ap.ap_masked_copy(x, out, 6, codes, 2)
    assert ap.ap_check() == ap.AP_OK
    assert to_np(out).tolist() == [1, 2, 3, 4, -1, -1, -1, -1, 9, 10, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 21, 0, 0, 0]


def test_masked_copy_in_place_and_bad_codes(ap, orc):
    import torch

    dev = device()
    n_chunks = 5000
    rng = np.random.default_rng(3)
    x = synth.uniform_pm1_torch(11, 4 * n_chunks, dev)
    x_h = to_np(x)
    c_h, c_d = _codes(rng, n_chunks, dev)
    ap.ap_masked_copy(x, x, n_chunks, c_d, 3)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(x), orc.masked_copy(x_h, x_h, c_h), "in place")
    # an out-of-range code leaves its chunk unchanged and is reported
    bad = c_d.clone()
    bad[17] = 40
    y = torch.zeros_like(x)
    ap.ap_masked_copy(x, y, n_chunks, bad, 2)
    assert ap.ap_check() == ap.AP_ERR_ARG
    assert ap.ap_check() == ap.AP_OK
    assert bool((y[68:72] == 0).all())


def test_masked_copy_full_size(ap, orc):
    """2**26 chunks (1 GiB): every 8th chunk predicated off, every 8th + 1 a
    half chunk, every 8th + 2 zeroed, the rest plain copies."""
    import torch

    dev = device()
    n_chunks = 1 << 26
    x = synth.uniform_pm1_torch(synth.SEED_SCALE, 4 * n_chunks, dev)
    pattern = np.array([-1, 8, -2, 16, 16, 16, 16, 16], dtype=np.int8)
    c_h = np.tile(pattern, n_chunks // 8)
    c_d = torch.from_numpy(c_h).to(dev)
    y = torch.full_like(x, 7.0)
    ap.ap_masked_copy(x, y, n_chunks, c_d, 4)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.masked_copy(to_np(x), np.full(4 * n_chunks, 7.0, np.float32), c_h), "full masked")


@pytest.mark.parametrize("stages", [3, 6])
def test_masked_copy_beyond_2p32_bytes(ap, orc, stages):
    """2^28 + 1029 chunks (4 GiB + 16 KiB in and out, random codes), so byte
    offsets pass 2^32, under the run schedule (depth 3) and the persistent grid
    (depth 6); checked against the oracle over the first and last 1 Mi chunks
    and 4096 random windows of 64 chunks."""
    import torch

    dev = device()
    n_chunks = (1 << 28) + 1029
    g = torch.Generator(device=dev)
    g.manual_seed(0xA5A7 + stages)
    x = torch.empty(4 * n_chunks, dtype=torch.float32, device=dev).uniform_(-1.0, 1.0, generator=g)
    codes = torch.randint(-2, 17, (n_chunks,), dtype=torch.int8, device=dev, generator=g)
    y = torch.full_like(x, 7.0)
    ap.ap_masked_copy(x, y, n_chunks, codes, stages)
    assert ap.ap_check() == ap.AP_OK
    rng = np.random.default_rng(stages)
    windows = [(0, 1 << 20), (n_chunks - (1 << 20), n_chunks)]
    windows += [(int(s), int(s) + 64) for s in rng.integers(0, n_chunks - 64, 4096)]
    for lo, hi in windows:
        xs = to_np(x[4 * lo:4 * hi])
        want = orc.masked_copy(xs, np.full(xs.size, 7.0, np.float32), to_np(codes[lo:hi]))
        assert_bits(to_np(y[4 * lo:4 * hi]), want, f"masked beyond 2^32 bytes, chunks {lo}..{hi} S={stages}")

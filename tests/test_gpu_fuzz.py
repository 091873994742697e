"""Randomised parity of the ring and the cluster exchange against the oracle:
random sizes, 4-byte offsets of input and output, ring depths, stage sizes,
grid caps, CTAs per SM and consumer-warp counts, bit for bit, with sentinels
around every output. AP_FUZZ_SEEDS (default 3) sets how many seeds each test
runs (the ring test at least 6), for longer stress runs."""

import os

import numpy as np
import pytest

import synth
from gpu_util import Guarded, assert_bits, device, lib, reset_debug, to_np

pytestmark = pytest.mark.gpu

SEEDS = range(int(os.environ.get("AP_FUZZ_SEEDS", "3")))
RING_SEEDS = range(max(6, len(SEEDS)))


@pytest.fixture
def ap():
    ap = lib()
    reset_debug(ap)
    yield ap
    reset_debug(ap)


def _knobs(ap, rng):
    ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, int(rng.choice([0, 16, 48, 256, 4096, 24576, 65536])))
    ap.ap_debug_set(ap.AP_DBG_GRID, int(rng.choice([0, 0, 1, 2, 5, 37])))
    ap.ap_debug_set(ap.AP_DBG_CTAS_PER_SM, int(rng.choice([0, 1, 2, 3])))
    ap.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, int(rng.choice([0, 8, 12, 16])))
    ap.ap_debug_set(ap.AP_DBG_RING_RUN, int(rng.choice([0, 0, 1, 2, 3, 7, 12])))


@pytest.mark.parametrize("seed", RING_SEEDS)
def test_ring_fuzz(ap, orc, seed):
    dev = device()
    rng = np.random.default_rng(1000 + seed)
    for case in range(40):
        op = str(rng.choice(["scale", "poly", "roll"]))
        n = int(rng.integers(1, 1 << int(rng.integers(1, 18))))
        in_shift, out_shift = (int(v) for v in rng.integers(0, 4, 2))
        stages = int(rng.integers(2, 7))
        _knobs(ap, rng)
        src = Guarded(n, in_shift, dev, fill=synth.uniform_pm1_torch(seed * 100 + case, n, dev))
        x = to_np(src.view)
        out = Guarded(n, out_shift, dev)
        what = f"seed={seed} case={case} op={op} n={n} in+{in_shift} out+{out_shift} S={stages}"
        try:
            want = _run_op(ap, orc, rng, op, src, out, x, n, stages)
        except ap.APError as e:
            # only a stage size whose ring cannot fit in shared memory may be refused
            assert e.status == ap.AP_ERR_SMEM, what
            assert ap.ap_debug_get(ap.AP_DBG_STAGE_BYTES) * stages > 200 * 1024, what
            assert out.intact(), what
            reset_debug(ap)
            continue
        assert ap.ap_check() == ap.AP_OK, what
        assert_bits(to_np(out.view), want, what)
        assert out.intact(), what
        assert src.intact(), what
        reset_debug(ap)


def _run_op(ap, orc, rng, op, src, out, x, n, stages):
    """Run one random operation; returns the oracle's expected output."""
    if op == "scale":
        alpha = float(np.float32(rng.uniform(-4, 4)))
        ap.ap_scale(src.view, out.view, n, 1, alpha, stages)
        want = orc.scale(x, alpha)
    elif op == "poly":
        # low degrees, and degrees from 64 where whole six-group stages take 24 chains
        degree = int(rng.integers(0, 40)) if rng.random() < 0.7 else int(rng.integers(60, 140))
        c = synth.coeffs_np(degree)
        ap.ap_poly(src.view, out.view, n, c.tolist(), degree, stages)
        want = orc.poly(x, c)
    else:
        divisors = [d for d in range(1, 9) if n % d == 0]
        cols = int(rng.choice(divisors))
        rows = n // cols
        shift = int(rng.integers(-3 * rows, 3 * rows + 1))
        ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, int(rng.choice([0, 1])))
        ap.ap_debug_set(ap.AP_DBG_ROLL_STAGES, stages)
        ap.ap_row_roll(src.view, out.view, rows, cols, shift)
        want = orc.row_roll(x.reshape(rows, cols), shift).ravel()
    return want


@pytest.mark.parametrize("seed", SEEDS)
def test_exchange_fuzz(ap, orc, seed):
    dev = device()
    rng = np.random.default_rng(2000 + seed)
    for case in range(25):
        cs = int(rng.choice([1, 2, 4, 8]))
        chunk = 16 * int(rng.integers(1, 2049))
        groups = int(rng.integers(1, 40))
        n = groups * cs * chunk // 4
        x = synth.uniform_pm1_torch(seed * 100 + case, n, dev)
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, int(rng.choice([0, 16, 1024, 8192, 16384])))
        ap.ap_debug_set(ap.AP_DBG_GRID, int(rng.choice([0, 0, cs, 3 * cs])))
        ap.ap_debug_set(ap.AP_DBG_CTAS_PER_SM, int(rng.choice([0, 1, 2, 3])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_STORE, int(rng.choice([0, 1, 2])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, int(rng.choice([0, 1, 2, 4, 8])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, int(rng.choice([0, 1, 2, 4])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, int(rng.choice([0, 0, 1, 2, 8, 100])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_SEND_SLOTS, int(rng.choice([0, 0, 1, 2, 4, 8, 16])))
        out = Guarded(n, 0, dev)
        ap.ap_cluster_exchange(x, out.view, n, cs, chunk)
        what = f"seed={seed} case={case} cs={cs} chunk={chunk} groups={groups}"
        assert ap.ap_check() == ap.AP_OK, what
        assert_bits(to_np(out.view), orc.cluster_exchange(to_np(x), cs, chunk), what)
        assert out.intact(), what
        reset_debug(ap)


@pytest.mark.parametrize("seed", SEEDS)
def test_all_to_all_fuzz(ap, orc, seed):
    """Random cluster sizes 1-16, sub-block sizes, group counts and every
    exchange setting (receiver form, warps per piece, lanes, batch, pieces,
    grid, CTAs per SM) against the oracle."""
    dev = device()
    rng = np.random.default_rng(3000 + seed)
    for case in range(25):
        cs = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16]))
        sub = 16 * int(rng.choice([int(rng.integers(1, 257)), 256, 512]))  # up to 8 KiB: the three-CTA form too
        chunk = cs * sub
        groups = int(rng.integers(1, 60))
        n = groups * cs * chunk // 4
        x = synth.uniform_pm1_torch(seed * 1000 + case, n, dev)
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, int(rng.choice([0, 0, 512, 2048, 8192])))
        ap.ap_debug_set(ap.AP_DBG_GRID, int(rng.choice([0, 0, cs, 2 * cs])))
        ap.ap_debug_set(ap.AP_DBG_CTAS_PER_SM, int(rng.choice([0, 1, 2, 3])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_STORE, int(rng.choice([0, 1, 2])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, int(rng.choice([0, 1, 2, 4, 8])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, int(rng.choice([0, 1, 2, 4])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, int(rng.choice([0, 0, 1, 2, 8, 100])))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_SEND_SLOTS, int(rng.choice([0, 0, 1, 2, 4, 8, 16])))
        out = Guarded(n, 0, dev)
        what = f"seed={seed} case={case} cs={cs} sub={sub} groups={groups}"
        try:
            ap.ap_cluster_all_to_all(x, out.view, n, cs, chunk)
        except ap.APError as e:  # a shape the settings cannot fit in shared memory
            assert e.status == ap.AP_ERR_SMEM, what
            reset_debug(ap)
            continue
        assert ap.ap_check() == ap.AP_OK, what
        assert_bits(to_np(out.view), orc.cluster_all_to_all(to_np(x), cs, chunk), what)
        assert out.intact(), what
        reset_debug(ap)

"""ap_poly against the oracle: Horner with fmaf on both sides in the same
order, so the tolerance is 0 ULP (bit-exact)."""

import numpy as np
import pytest

import synth
from gpu_util import oracle_poly_threads, Guarded, assert_bits, device, lib, reset_debug, tensor_flags, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture
def ap():
    ap = lib()
    reset_debug(ap)
    yield ap
    reset_debug(ap)


@pytest.mark.parametrize("degree", [0, 1, 2, 3, 4, 5, 7, 8, 32, 127, 128, 1023])
@pytest.mark.parametrize("stages", [2, 3, 4, 6])
def test_poly_small(ap, orc, degree, stages):
    dev = device()
    n = 20011
    x = synth.uniform_pm1_torch(n + degree, n, dev)
    c = synth.coeffs_np(degree)
    want = orc.poly(to_np(x), c)
    for stage_bytes, grid, warps in ((256, 2, 8), (0, 0, 0), (1024, 3, 16), (0, 0, 16), (2048, 2, 12), (0, 0, 12)):
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        ap.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, warps)
        out = Guarded(n, 0, dev)
        ap.ap_poly(x, out.view, n, c.tolist(), degree, stages)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), want, f"poly K={degree} S={stages} stage={stage_bytes} warps={warps}")
        assert out.intact()


@pytest.mark.parametrize("degree", [6, 9, 12, 13, 15, 16, 17, 31, 33, 124, 125, 126, 129, 130, 131, 132, 133, 255, 511])
def test_poly_degree_boundaries(ap, orc, degree):
    """Degrees on both sides of the coefficient loop's four-step words (a
    scalar lead-in until k + 1 is a multiple of four, then four steps per
    16-byte word with the next word loaded ahead), in rounds of 8 to 32
    chains a thread: element by element against the oracle, under 8, 12 and
    16 consumer warps and stages that do and do not take six groups a round."""
    dev = device()
    n = 3 * 96 * 1024 // 4 + 4099
    x = synth.uniform_pm1_torch(n + degree + 11, n, dev)
    c = synth.coeffs_np(degree)
    want = orc.poly(to_np(x), c)
    for stage_bytes, warps in ((0, 0), (48 * 1024, 16), (64 * 1024, 16), (32 * 1024, 8), (16 * 1024, 12)):
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        ap.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, warps)
        out = Guarded(n, 0, dev)
        ap.ap_poly(x, out.view, n, c.tolist(), degree, 2)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), want, f"poly K={degree} stage={stage_bytes} warps={warps}")
        assert out.intact()


@pytest.mark.parametrize("warps,groups,stages", [(12, 2, 2), (12, 2, 4), (12, 2, 6), (12, 3, 3), (12, 3, 6),
                                                  (16, 2, 2), (16, 1, 4), (12, 1, 5)])
@pytest.mark.parametrize("degree", [0, 8, 33, 128])
def test_poly_consumer_groups(ap, orc, degree, warps, groups, stages):
    """Explicit consumer groups (group g takes stages g, g + groups, ...; the
    count divides the warps and the ring depth), persistent and in runs of
    consecutive stages, with ragged ends; element by element."""
    dev = device()
    c = synth.coeffs_np(degree)
    ap.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, warps)
    ap.ap_debug_set(ap.AP_DBG_CONSUMER_GROUPS, groups)
    for stage_bytes, run in ((16 * 1024, 1), (8 * 1024, 0), (12 * 1024, 2 * stages), (4096, 7)):
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        ap.ap_debug_set(ap.AP_DBG_RING_RUN, run)
        n = 37 * stage_bytes // 4 + 1237
        x = synth.uniform_pm1_torch(n + degree + 5, n, dev)
        want = orc.poly(to_np(x), c)
        out = Guarded(n, 1, dev)
        ap.ap_poly(x, out.view, n, c.tolist(), degree, stages)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), want, f"poly K={degree} warps={warps} groups={groups} S={stages} run={run}")
        assert out.intact()


def test_poly_consumer_groups_rejected(ap):
    """A group count that does not divide the warps or the ring depth."""
    import torch

    dev = device()
    x = torch.zeros(4096, device=dev)
    y = torch.empty_like(x)
    for warps, groups, stages in ((16, 3, 3), (12, 2, 3), (12, 3, 4), (8, 2, 4), (8, 3, 6)):
        ap.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, warps)
        ap.ap_debug_set(ap.AP_DBG_CONSUMER_GROUPS, groups)
        with pytest.raises(ap.APError) as e:
            ap.ap_poly(x, y, 4096, [1.0, 2.0], 1, stages)
        assert e.value.status == ap.AP_ERR_ARG


@pytest.mark.parametrize("stages", [4, 6])
@pytest.mark.parametrize("degree", [7, 9, 32, 64, 128])
def test_poly_two_consumer_groups(ap, orc, degree, stages):
    """16 consumer warps at even depths of 4 or more split into two groups of
    8 that take alternate stages (group g: stages g, g + 2, ...). Two CTAs
    of about 20 stages each run many laps of the ring, with an odd stage
    count on one CTA and a ragged last stage; element by element."""
    dev = device()
    c = synth.coeffs_np(degree)
    for stage_bytes in (32 * 1024, 16 * 1024):
        per = stage_bytes // 4
        n = 41 * per + 1237
        x = synth.uniform_pm1_torch(n + degree + 3, n, dev)
        want = orc.poly(to_np(x), c)
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        ap.ap_debug_set(ap.AP_DBG_GRID, 2)
        ap.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, 16)
        out = Guarded(n, 0, dev)
        ap.ap_poly(x, out.view, n, c.tolist(), degree, stages)
        assert ap.ap_check() == ap.AP_OK
        assert ap.ap_debug_get(ap.AP_DBG_LAST_GRID) == 2
        assert_bits(to_np(out.view), want, f"poly K={degree} S={stages} stage={stage_bytes} two groups")
        assert out.intact()


@pytest.mark.parametrize("degree", [31, 32, 43, 44, 48, 63, 64, 127, 128, 200])
def test_poly_six_group_rounds(ap, orc, degree):
    """Stages that are whole rounds of six 16-byte groups per consumer thread
    (16 consumer warps in one group: 48 KiB and 96 KiB) take 24 Horner chains
    a thread from degree 44 on, 16 below; the automatic stage (96 KiB, or
    64 KiB at degrees 27-31) and both whole-round sizes; five whole stages
    and a ragged sixth, element by element."""
    dev = device()
    c = synth.coeffs_np(degree)
    for stage_bytes in (0, 48 * 1024, 96 * 1024):
        per = (stage_bytes or _auto_shape(degree, 2)[0] * 1024) // 4
        n = 5 * per + 1234
        x = synth.uniform_pm1_torch(n + degree + 7, n, dev)
        want = orc.poly(to_np(x), c)
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        for grid in (0, 2):
            ap.ap_debug_set(ap.AP_DBG_GRID, grid)
            out = Guarded(n, 0, dev)
            ap.ap_poly(x, out.view, n, c.tolist(), degree, 2)
            assert ap.ap_check() == ap.AP_OK
            assert ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS) == per
            assert_bits(to_np(out.view), want, f"poly K={degree} stage={stage_bytes} grid={grid}")
            assert out.intact()


def _auto_shape(degree: int, stages: int) -> tuple:
    """The documented automatic shapes of ap_poly, band by band: (stage KiB,
    stages per CTA (0: persistent grid), consumer warps, consumer groups)."""
    if stages == 2:
        if degree <= 15:
            return (64, 4, 16, 1)
        if degree <= 26:
            return (96, 4, 16, 1)
        return (64, 0, 16, 1) if degree <= 31 else (96, 0, 16, 1)
    if stages == 3:
        if degree <= 1:
            return (32, 6, 16, 1)
        if degree <= 14:
            return (48, 6, 16, 1)
        if degree <= 26:
            return (64, 6, 16, 1)
        if degree <= 29:
            return (48, 0, 16, 1)
        return (64, 0, 16, 1) if degree < 64 else (48, 0, 16, 1)
    if stages == 4:
        if degree <= 16:
            return (32, 8, 16, 2)
        if degree <= 26:
            return (48, 8, 16, 2)
        return (32, 0, 16, 2) if degree <= 31 else (48, 0, 16, 2)
    if stages == 5:
        if degree <= 18:
            return (32, 10, 16, 1)
        if degree <= 22:
            return (32, 0, 12, 1)
        return (40, 0, 16, 1) if degree <= 25 else (32, 0, 16, 1)
    if degree <= 12:
        return (24, 12, 16, 2)
    if degree <= 26:
        return (32, 12, 16, 2)
    return (24, 0, 16, 2) if degree <= 30 else (32, 0, 12, 3)


def test_poly_automatic_stage_sizes(ap, orc):
    """Automatic shapes across the degree bands at every depth: runs of
    stages where memory bounds the kernel, the persistent grid where the fma
    work does (stage size, schedule, consumer warps and groups as documented)."""
    dev = device()
    n = 3 * 24576 + 5
    x = synth.uniform_pm1_torch(n, n, dev)
    for degree in (0, 1, 2, 3, 4, 8, 12, 13, 14, 15, 16, 17, 18, 19, 22, 23, 25, 26, 27, 29, 30, 31, 32, 63, 64, 128):
        c = synth.coeffs_np(degree)
        want = orc.poly(to_np(x), c)
        for stages in (2, 3, 4, 5, 6):
            out = Guarded(n, 0, dev)
            ap.ap_poly(x, out.view, n, c.tolist(), degree, stages)
            assert ap.ap_check() == ap.AP_OK
            kib, run, warps, groups = _auto_shape(degree, stages)
            got = (ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS), ap.ap_debug_get(ap.AP_DBG_LAST_RUN),
                   ap.ap_debug_get(ap.AP_DBG_LAST_WARPS), ap.ap_debug_get(ap.AP_DBG_LAST_GROUPS))
            assert got == (kib * 256, run, warps, groups), f"K={degree} S={stages}: {got}"
            assert_bits(to_np(out.view), want, f"poly K={degree} S={stages} automatic shape")
            assert out.intact()


@pytest.mark.parametrize("stages", [2, 3, 4, 5, 6])
def test_poly_every_degree_automatic(ap, orc, stages):
    """Every degree 0-66 and a few about 128 under the automatic shape of each
    depth (every band edge and both chain counts), over several stages and
    CTAs with a ragged end, element by element against the oracle."""
    dev = device()
    n = 5 * 24576 + 4099  # at least two CTAs under every run schedule, several stages each
    x = synth.uniform_pm1_torch(n + 17 * stages, n, dev)
    xh = to_np(x)
    for degree in list(range(0, 67)) + [79, 80, 126, 127, 128]:
        c = synth.coeffs_np(degree)
        out = Guarded(n, 0, dev)
        ap.ap_poly(x, out.view, n, c.tolist(), degree, stages)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), orc.poly(xh, c), f"poly K={degree} S={stages} automatic")
        assert out.intact()


@pytest.mark.parametrize("degree", [0, 3, 8, 128])
def test_poly_tensor_map_producer(ap, orc, degree):
    """Horner over the tensor-map producer's boxes, ragged lengths; three whole
    automatic stages and a ragged fourth at depth 2 (degree 128: 96 KiB stages
    in rounds of six groups, 24 chains a thread)."""
    dev = device()
    c = synth.coeffs_np(degree)
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    for n, stages in ((1, 2), (7, 3), (256, 4), (20011, 2), (20011, 6), (1 << 18, 3), (3 * 24576 + 17, 2)):
        x = synth.uniform_pm1_torch(n + degree, n, dev)
        out = Guarded(n, 0, dev)
        ap.ap_poly(x, out.view, n, c.tolist(), degree, stages)
        assert ap.ap_check() == ap.AP_OK
        assert ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 12 == tensor_flags(ap, n, 0)
        assert_bits(to_np(out.view), orc.poly(to_np(x), c), f"tensor poly K={degree} n={n} S={stages}")
        assert out.intact()


@pytest.mark.parametrize("in_shift,out_shift", [(1, 0), (0, 3), (2, 2)])
def test_poly_misaligned_and_edges(ap, orc, in_shift, out_shift):
    import torch

    dev = device()
    c = synth.coeffs_np(8)
    for n in (1, 2, 3, 5, 17, 4099):
        src = Guarded(n, in_shift, dev, fill=synth.uniform_pm1_torch(n, n, dev))
        out = Guarded(n, out_shift, dev)
        ap.ap_poly(src.view, out.view, n, c.tolist(), 8, 2)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), orc.poly(to_np(src.view), c), f"poly n={n} in+{in_shift} out+{out_shift}")
        assert out.intact()


def test_poly_special_values(ap, orc):
    """Zeros of both signs, infinities, NaN, a subnormal and a large finite
    value; 9 * 5000 elements, so that the wide rounds (16 and 24 chains a
    thread) see them as well as the one-group rounds and the tails."""
    import torch

    dev = device()
    vals = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 1e-40, 65504.0], dtype=np.float32)
    x = torch.from_numpy(np.tile(vals, 5000)).to(dev)
    for degree in (0, 1, 3, 16, 128, 130):
        c = synth.coeffs_np(degree)
        y = torch.empty_like(x)
        ap.ap_poly(x, y, x.numel(), c.tolist(), degree, 2)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(y), orc.poly(to_np(x), c), f"special K={degree}", nan_equal=True)


def test_poly_full_size_sweep(ap, orc):
    """2**30 floats (4 GiB), stages {2,3,4,6} x degree {0,8,32,128}, every
    element compared bit for bit with the oracle. The oracle's output for a
    degree is computed once (its loop split over the host cores) and compared
    with each depth's output on the device (torch.equal of the bit patterns;
    the seeded inputs hold no NaN)."""
    import torch

    dev = device()
    n = 1 << 30
    x = synth.uniform_pm1_torch(synth.SEED_POLY, n, dev)
    x_host = to_np(x)
    y = torch.empty_like(x)
    for degree in (0, 8, 32, 128):
        c = synth.coeffs_np(degree)
        want = torch.from_numpy(oracle_poly_threads(orc, x_host, c)).to(dev).view(torch.int32)
        for stages in (2, 3, 4, 6):
            y.fill_(float("nan"))
            ap.ap_poly(x, y, n, c.tolist(), degree, stages)
            assert ap.ap_check() == ap.AP_OK
            got = y.view(torch.int32)
            if not torch.equal(got, want):
                bad = torch.nonzero(got != want)[:8].flatten().tolist()
                raise AssertionError(f"full poly K={degree} S={stages}: {int((got != want).sum())} elements differ "
                                     f"from the oracle, first at {bad}")
        del want


def test_fma_probes_cover_their_threads(ap):
    """Both FP32 probes write one finite float per launched thread (whole
    CTAs of 512, at most 1024 a SM for the register-only form and 512 for the
    Horner form) and nothing past them; bad sizes are refused."""
    import torch

    dev = device()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for fn, per_sm in ((ap.ap_debug_fma_probe, 1024), (ap.ap_debug_fma_probe_horner, 512)):
        for elems in (sms * 1024 + 7, 3 * 512 + 100):
            out = torch.full((elems,), float("nan"), dtype=torch.float32, device=dev)
            fn(out, elems, 8)
            assert ap.ap_check() == ap.AP_OK
            launched = min(elems, sms * per_sm) // 512 * 512
            o = to_np(out)
            assert np.isfinite(o[:launched]).all(), fn.__name__
            assert np.isnan(o[launched:]).all(), fn.__name__
        for elems, iters in ((100, 8), (512, 0)):
            with pytest.raises(ap.APError):
                fn(out, elems, iters)


# (degree, depth) -> (run, consumer warps, groups, chains) of the automatic shape
AUTO_SHAPES = {
    (0, 2): (4, 16, 1, 16), (8, 2): (4, 16, 1, 16), (32, 2): (0, 16, 1, 16), (128, 2): (0, 16, 1, 24),
    (0, 3): (6, 16, 1, 16), (8, 3): (6, 16, 1, 16), (32, 3): (0, 16, 1, 16), (128, 3): (0, 16, 1, 24),
    (0, 4): (8, 16, 2, 16), (8, 4): (8, 16, 2, 16), (32, 4): (0, 16, 2, 16), (128, 4): (0, 16, 2, 24),
    (0, 6): (12, 16, 2, 16), (8, 6): (12, 16, 2, 16), (32, 6): (0, 12, 3, 32), (128, 6): (0, 12, 3, 32),
    # where 24 chains start: degree 44 in one group (depth 2), 34 in two (depth 4)
    (43, 2): (0, 16, 1, 16), (44, 2): (0, 16, 1, 24), (33, 4): (0, 16, 2, 16), (34, 4): (0, 16, 2, 24),
}


@pytest.mark.parametrize("degree,stages", sorted(AUTO_SHAPES))
def test_poly_automatic_shapes(ap, orc, degree, stages):
    """The automatic shape of each cell of the degree x depth sweep (runs of
    stages where memory bounds the kernel, the persistent grid where the fma
    work does, 24 chains a round with 16 warps from degree 44 in one group or
    34 in two, 12 warps in three groups at depth 6 from degree 31) is the one
    that runs, and its
    output matches the oracle element by element."""
    dev = device()
    n = (1 << 20) + 4099
    x = synth.uniform_pm1_torch(n + degree + stages, n, dev)
    c = synth.coeffs_np(degree)
    out = Guarded(n, 0, dev)
    ap.ap_poly(x, out.view, n, c.tolist(), degree, stages)
    assert ap.ap_check() == ap.AP_OK
    got = tuple(ap.ap_debug_get(k) for k in (ap.AP_DBG_LAST_RUN, ap.AP_DBG_LAST_WARPS, ap.AP_DBG_LAST_GROUPS,
                                             ap.AP_DBG_LAST_CHAINS))
    assert got == AUTO_SHAPES[(degree, stages)], f"K={degree} S={stages}: {got}"
    assert_bits(to_np(out.view), orc.poly(to_np(x), c), f"automatic shape K={degree} S={stages}")
    assert out.intact()

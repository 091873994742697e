"""ap_scale (pipelined ring) and ap_scale_sync (synchronous baseline) against
the oracle, bit for bit (one correctly rounded fp32 multiply per element)."""

import numpy as np
import pytest

import synth
from gpu_util import Guarded, assert_bits, device, lib, reset_debug, tensor_flags, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture
def ap():
    ap = lib()
    reset_debug(ap)
    yield ap
    reset_debug(ap)


@pytest.mark.parametrize("stages", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("n_tiles,tile", [(1, 1), (1, 3), (3, 5), (37, 256), (101, 7), (64, 256)])
def test_scale_small_many_stages(ap, orc, stages, n_tiles, tile):
    import torch

    dev = device()
    n = n_tiles * tile
    x = synth.uniform_pm1_torch(n + 17, n, dev)
    want = orc.scale(to_np(x), 2.0)
    # tiny stages and few CTAs: every ring slot goes through many phases
    for stage_bytes, grid, warps, cps in ((64, 1, 8, 0), (256, 3, 16, 0), (1024, 0, 0, 3), (0, 0, 0, 0)):
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        ap.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, warps)
        ap.ap_debug_set(ap.AP_DBG_CTAS_PER_SM, cps)
        out = Guarded(n, 0, dev)
        ap.ap_scale(x, out.view, n_tiles, tile, 2.0, stages)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), want, f"scale S={stages} n={n} stage={stage_bytes} grid={grid}")
        assert out.intact(), "wrote outside the output"
        assert ap.ap_debug_get(ap.AP_DBG_LAST_PATH) == 1


@pytest.mark.parametrize("stages", [2, 3, 5, 6])
@pytest.mark.parametrize("n", [5, 4099, 65536 + 3, 1000003])
@pytest.mark.parametrize("run", [1, 2, 3, 7, 12])
def test_scale_stage_runs(ap, orc, stages, n, run):
    """Both schedules: a persistent grid (run 1) and CTAs that each take a run
    of consecutive stages, including a short last run and runs shorter than,
    equal to and longer than the ring, over misaligned buffers too."""
    dev = device()
    x = synth.uniform_pm1_torch(n + 5, n + 1, dev)
    ap.ap_debug_set(ap.AP_DBG_RING_RUN, run)
    for stage_bytes, in_shift, out_shift in ((256, 0, 0), (4096, 1, 0), (0, 0, 3)):
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        src = Guarded(n, in_shift, dev, fill=x[:n])
        want = orc.scale(to_np(src.view), 2.0)
        out = Guarded(n, out_shift, dev)
        ap.ap_scale(src.view, out.view, n, 1, 2.0, stages)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), want, f"run={run} S={stages} n={n} stage={stage_bytes}")
        assert out.intact(), "wrote outside the output"
        stage_elems = ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS)
        n_stages = max(1, -(-(n - (-out_shift % 4)) // stage_elems))
        if run > 1:
            assert ap.ap_debug_get(ap.AP_DBG_LAST_GRID) >= -(-(n_stages - 1) // run)


@pytest.mark.parametrize("in_shift,out_shift", [(0, 1), (1, 0), (1, 1), (2, 3), (3, 2), (3, 3)])
def test_scale_misaligned(ap, orc, in_shift, out_shift):
    dev = device()
    n = 10007
    src = Guarded(n, in_shift, dev, fill=synth.uniform_pm1_torch(99, n, dev))
    want = orc.scale(to_np(src.view), -1.5)
    for stage_bytes in (0, 512):
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        ap.ap_debug_set(ap.AP_DBG_GRID, 4 if stage_bytes else 0)
        out = Guarded(n, out_shift, dev)
        ap.ap_scale(src.view, out.view, n, 1, -1.5, 3)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), want, f"misaligned in+{in_shift} out+{out_shift}")
        assert out.intact()
        assert src.intact()


@pytest.mark.parametrize("stages", [2, 3, 6])
@pytest.mark.parametrize("n", [1, 3, 4, 255, 256, 257, 1000, 4099, 65536 + 5, 300001])
def test_scale_tensor_map_producer(ap, orc, stages, n):
    """The tensor-map producer (whole stages as 2-D boxes of 1 KiB lines, the
    ragged end as 1-D boxes of 256 floats with zeros past it) carries the
    scale stream bit for bit."""
    dev = device()
    x = synth.uniform_pm1_torch(n + 31, n, dev)
    want = orc.scale(to_np(x), -3.0)
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    for stage_bytes, grid in ((0, 0), (1024, 2), (8192, 5)):
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        out = Guarded(n, 0, dev)
        ap.ap_scale(x, out.view, n, 1, -3.0, stages)
        assert ap.ap_check() == ap.AP_OK
        assert ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 12 == tensor_flags(ap, n, 0), "tensor map did not run"
        assert_bits(to_np(out.view), want, f"tensor scale n={n} S={stages} stage={stage_bytes}")
        assert out.intact()
    # in place, and a misaligned output (the bulk producer takes over)
    y = x.clone()
    ap.ap_scale(y, y, n, 1, -3.0, stages)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), want, "tensor scale in place")
    out = Guarded(n, 1, dev)
    ap.ap_scale(x, out.view, n, 1, -3.0, stages)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 4 == 0
    assert_bits(to_np(out.view), want, "misaligned output falls back")
    assert out.intact()


def test_scale_tensor_map_full_size(ap, orc):
    """2**20 tiles x 256 floats through the tensor maps, 2 stages."""
    import torch

    dev = device()
    n = 1 << 28
    x = synth.uniform_pm1_torch(synth.SEED_SCALE, n, dev)
    y = torch.empty_like(x)
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    ap.ap_scale(x, y, n >> 8, 256, 2.0, 2)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 12 == 12
    assert_bits(to_np(y), orc.scale(to_np(x), 2.0), "full-size tensor scale")


def test_scale_in_place(ap, orc):
    import torch

    dev = device()
    n_tiles, tile = 300, 256
    x = synth.uniform_pm1_torch(5, n_tiles * tile, dev)
    want = orc.scale(to_np(x), 0.375)
    ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, 2048)
    ap.ap_scale(x, x, n_tiles, tile, 0.375, 4)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(x), want, "in place")


def test_scale_special_values(ap, orc):
    import torch

    dev = device()
    vals = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 1.1754942e-38, 3.4e38, -3.4e38, 1.0, -2.5],
                    dtype=np.float32)
    x_np = np.tile(vals, 100)
    x = torch.from_numpy(x_np).to(dev)
    for alpha in (2.0, 0.5, -3.0, 1e-10):
        y = torch.empty_like(x)
        ap.ap_scale(x, y, len(x_np), 1, alpha, 2)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(y), orc.scale(x_np, alpha), f"special alpha={alpha}", nan_equal=True)
        ys = torch.empty_like(x)
        ap.ap_scale_sync(x, ys, len(x_np), 1, alpha)
        assert_bits(to_np(ys), orc.scale(x_np, alpha), f"sync special alpha={alpha}", nan_equal=True)


@pytest.mark.parametrize("n_tiles,tile", [(1, 1), (5, 3), (37, 256), (4, 2000), (2, 20000)])
def test_scale_sync_small(ap, orc, n_tiles, tile):
    dev = device()
    n = n_tiles * tile
    x = synth.uniform_pm1_torch(n, n, dev)
    out = Guarded(n, 0, dev)
    ap.ap_scale_sync(x, out.view, n_tiles, tile, 2.0)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(out.view), orc.scale(to_np(x), 2.0), "sync")
    assert out.intact()


def test_scale_full_size_ring_vs_sync_vs_oracle(ap, orc):
    """The benchmark's workload: 2**20 tiles x 256 floats, alpha 2, 2 stages."""
    import torch

    dev = device()
    n_tiles, tile = 1 << 20, 256
    n = n_tiles * tile
    x = synth.uniform_pm1_torch(synth.SEED_SCALE, n, dev)
    y = torch.empty_like(x)
    ap.ap_scale(x, y, n_tiles, tile, 2.0, 2)
    assert ap.ap_check() == ap.AP_OK
    x_h = to_np(x)
    assert_bits(to_np(y), orc.scale(x_h, 2.0), "full-size ring")
    ys = torch.empty_like(x)
    ap.ap_scale_sync(x, ys, n_tiles, tile, 2.0)
    assert ap.ap_check() == ap.AP_OK
    assert torch.equal(ys.view(torch.int32), y.view(torch.int32)), "sync baseline and ring differ"
    for stages in (3, 4, 6):
        ap.ap_scale(x, ys, n_tiles, tile, 2.0, stages)
        assert ap.ap_check() == ap.AP_OK
        assert torch.equal(ys.view(torch.int32), y.view(torch.int32)), f"stages={stages} differs"


def test_device_generator_matches_host(ap):
    import torch

    dev = device()
    n = 1 << 22
    t = synth.uniform_pm1_torch(synth.SEED_POLY, n, dev)
    idx = np.random.default_rng(0).integers(0, n, 4096)
    got = to_np(t[torch.from_numpy(idx).to(dev)])
    assert_bits(got, synth.uniform_pm1_np(synth.SEED_POLY, n)[idx], "device generator")


@pytest.mark.parametrize("n_tiles,tile", [(1, 1), (5, 3), (37, 256), (1000, 1024), (1 << 20, 256)])
def test_scale_pages_async_baseline(ap, orc, n_tiles, tile):
    """The pages' two-stage, per-thread cp.async version gives the same bits."""
    dev = device()
    n = n_tiles * tile
    x = synth.uniform_pm1_torch(n + 3, n, dev)
    out = Guarded(n, 0, dev)
    ap.ap_debug_scale_pages_async(x, out.view, n_tiles, tile, 2.0)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_PATH) == 6
    assert_bits(to_np(out.view), orc.scale(to_np(x), 2.0), f"pages async {n_tiles}x{tile}")
    assert out.intact()


@pytest.mark.parametrize("op", ["scale", "roll", "poly"])
def test_beyond_2p32_elements(ap, orc, op):
    """The largest buffers exercised: 2^32 + 1028 floats (16 GiB in and 16 GiB
    out, an input 4 bytes past a 16-byte boundary), so element indices and
    byte offsets pass 2^32 and 2^34 inside the planner, the regular-stage
    shortcut and the consumers. Checked against the oracle at the first and
    last 1 Mi elements and 1 Mi random positions (each computed one by one by
    the oracle); the row shift wraps its last stage to row 0."""
    import torch

    dev = device()
    n = (1 << 32) + 1028
    base = torch.empty(n + 1, dtype=torch.float32, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(0xA5A5)
    base.uniform_(-1.0, 1.0, generator=g)
    x = base[1:]  # 4 bytes past the allocation's 16-byte boundary
    y = torch.empty(n, dtype=torch.float32, device=dev)
    rng = np.random.default_rng(3)
    idx_h = np.unique(np.concatenate([np.arange(1 << 20), np.arange(n - (1 << 20), n),
                                      rng.integers(0, n, 1 << 20)]))
    idx = torch.from_numpy(idx_h).to(dev)
    if op == "scale":
        ap.ap_scale(x, y, n, 1, -3.0, 4)
        want = orc.scale(to_np(x[idx]), -3.0)
    elif op == "roll":
        rows, cols = n // 4, 4
        shift = 7
        ap.ap_row_roll(x, y, rows, cols, shift)
        assert ap.ap_check() == ap.AP_OK
        # Output rows [r0, r0 + k) need input rows r0 .. r0 + k + shift - 1
        # (mod rows): the oracle shifts that window, and its first k rows are
        # the expected output rows. Windows at the start, across the wrap at
        # the end, and at random rows.
        starts = [0, rows - 4096] + [int(r) for r in rng.integers(0, rows - 16, 256)]
        for r0 in starts:
            k = 4096 if r0 in (0, rows - 4096) else 16
            src_rows = torch.remainder(torch.arange(r0, r0 + k + shift, device=dev), rows)
            window = to_np(x.view(rows, cols)[src_rows])
            want = orc.row_roll(window, shift)[:k]
            assert_bits(to_np(y.view(rows, cols)[r0:r0 + k]), want, f"roll beyond 2^32, rows {r0}..{r0 + k}")
        return
    else:
        c = synth.coeffs_np(8)
        ap.ap_poly(x, y, n, c.tolist(), 8, 3)
        want = orc.poly(to_np(x[idx]), c)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y[idx]), want, f"{op} over 2^32 + 1028 elements")

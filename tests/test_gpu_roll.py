"""ap_row_roll against the oracle, bit for bit: the 64 x 4 worked example
(one CTA, cp.async.cg), the ring path with halo rows across tiles and CTAs,
misaligned bases, and the full 2**26 x 4 matrix."""

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


def test_worked_example_64x4(ap, orc):
    import torch

    dev = device()
    A = torch.arange(256, dtype=torch.float32, device=dev).reshape(64, 4)
    B = torch.empty_like(A)
    ap.ap_row_roll(A, B, 64, 4, 1)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_PATH) == 2  # one CTA, cp.async.cg
    assert ap.ap_debug_get(ap.AP_DBG_LAST_GRID) == 1
    assert torch.equal(B, torch.roll(A, shifts=-1, dims=0))  # the page's own check
    assert_bits(to_np(B), orc.row_roll(to_np(A), 1), "64x4 arange")
    U = synth.uniform_pm1_torch(synth.SEED_ROLL_SMALL, 256, dev).reshape(64, 4)
    ap.ap_row_roll(U, B, 64, 4, 1)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(B), orc.row_roll(to_np(U), 1), "64x4 uniform")


@pytest.mark.parametrize("force", [0, 1])
@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 7), (2, 4), (3, 3), (64, 4), (100, 1), (257, 5), (1000, 4), (33, 8)])
def test_roll_shapes_and_shifts(ap, orc, force, rows, cols):
    dev = device()
    n = rows * cols
    A = synth.uniform_pm1_torch(rows * 1000 + cols, n, dev)
    A_h = to_np(A).reshape(rows, cols)
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, force)
    if force:
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, 128)
        ap.ap_debug_set(ap.AP_DBG_GRID, 3)
    for shift in (0, 1, -1, 2, rows - 1, rows, 7 * rows + 3, -(10**12) - 5):
        out = Guarded(n, 0, dev)
        ap.ap_row_roll(A, out.view, rows, cols, shift)
        assert ap.ap_check() == ap.AP_OK
        assert ap.ap_debug_get(ap.AP_DBG_LAST_PATH) == (1 if force else 2)
        assert_bits(to_np(out.view), orc.row_roll(A_h, shift), f"roll {rows}x{cols} shift={shift} force={force}")
        assert out.intact()


@pytest.mark.parametrize("stages", [2, 3, 4, 6])
def test_roll_ring_many_tiles(ap, orc, stages):
    dev = device()
    rows, cols = 50000, 4
    A = synth.uniform_pm1_torch(77, rows * cols, dev)
    A_h = to_np(A).reshape(rows, cols)
    ap.ap_debug_set(ap.AP_DBG_ROLL_STAGES, stages)
    for stage_bytes, grid in ((256, 5), (4096, 0), (0, 0)):
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        for shift in (1, 12345, rows - 1):
            out = Guarded(rows * cols, 0, dev)
            ap.ap_row_roll(A, out.view, rows, cols, shift)
            assert ap.ap_check() == ap.AP_OK
            assert ap.ap_debug_get(ap.AP_DBG_LAST_PATH) == 1
            assert_bits(to_np(out.view), orc.row_roll(A_h, shift), f"ring roll S={stages} stage={stage_bytes}")
            assert out.intact()


@pytest.mark.parametrize("a_shift,b_shift", [(1, 0), (0, 1), (1, 1), (2, 0), (3, 1)])
@pytest.mark.parametrize("rows,cols", [(64, 4), (20000, 4), (999, 3)])
def test_roll_misaligned(ap, orc, a_shift, b_shift, rows, cols):
    dev = device()
    n = rows * cols
    src = Guarded(n, a_shift, dev, fill=synth.uniform_pm1_torch(n + a_shift, n, dev))
    A_h = to_np(src.view).reshape(rows, cols)
    for force in (0, 1):
        ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, force)
        out = Guarded(n, b_shift, dev)
        ap.ap_row_roll(src.view, out.view, rows, cols, 1)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), orc.row_roll(A_h, 1), f"misaligned A+{a_shift} B+{b_shift} force={force}")
        assert out.intact() and src.intact()
        if a_shift % 4 and ap.ap_debug_get(ap.AP_DBG_LAST_PATH) == 1:
            assert ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 1, "misaligned input should use cp.async edges"


@pytest.mark.parametrize("variant", ["aligned", "A+4", "B+4", "A+4,B+4"])
def test_roll_full_size(ap, orc, variant):
    """2**26 rows x 4 floats (1 GiB), shift 1; the +4-byte variants put every
    16-byte row across a 16-byte boundary."""
    import torch

    dev = device()
    rows, cols = 1 << 26, 4
    n = rows * cols
    a_shift = 1 if "A+4" in variant else 0
    b_shift = 1 if "B+4" in variant else 0
    abuf = torch.empty(n + 4, dtype=torch.float32, device=dev)
    A = abuf[a_shift : a_shift + n]
    synth.uniform_pm1_torch(synth.SEED_ROLL, n, dev, out=A)
    bbuf = torch.empty(n + 4, dtype=torch.float32, device=dev)
    B = bbuf[b_shift : b_shift + n]
    ap.ap_row_roll(A, B, rows, cols, 1)
    assert ap.ap_check() == ap.AP_OK
    want = orc.row_roll(to_np(A).reshape(rows, cols), 1)
    assert_bits(to_np(B), want, f"full-size roll {variant}")


@pytest.mark.parametrize("stages", [2, 3, 6])
@pytest.mark.parametrize(
    "rows,cols",
    [(1, 4), (7, 4), (64, 4), (1000, 4), (50000, 4), (333, 8), (40, 12), (129, 256), (50, 64), (77, 128), (3, 200)],
)
def test_roll_tensor_map_producer(ap, orc, stages, rows, cols):
    """The tensor-map producer gives the oracle's result bit for bit: stages
    as one 2-D box of 1 KiB lines where the line view holds them, else 1-D
    boxes of 256 floats (zeros past the end of the input)."""
    dev = device()
    n = rows * cols
    A = synth.uniform_pm1_torch(rows * 7 + cols, n, dev)
    A_h = to_np(A).reshape(rows, cols)
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    ap.ap_debug_set(ap.AP_DBG_ROLL_STAGES, stages)
    for stage_bytes, grid in ((0, 0), (4096, 2), (16384, 3), (1024, 4)):
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, stage_bytes)
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        for shift in (1, 0, -1, rows // 2 + 1, 3 * rows - 2):
            out = Guarded(n, 0, dev)
            ap.ap_row_roll(A, out.view, rows, cols, shift)
            assert ap.ap_check() == ap.AP_OK
            off = (shift % rows) * cols
            assert ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 12 == tensor_flags(ap, n, off), "tensor-map producer"
            assert_bits(to_np(out.view), orc.row_roll(A_h, shift), f"tensor roll {rows}x{cols} shift={shift} S={stages}")
            assert out.intact()


@pytest.mark.parametrize("rows,cols,shift,tensor", [(1000, 3, 4, True), (1000, 3, 1, False), (999, 4, 5, True),
                                                    (250, 2, 2, True), (250, 2, 3, False), (10, 300, 3, True)])
def test_roll_tensor_map_rules(ap, orc, rows, cols, shift, tensor):
    """Rows of any length take the tensor-map producer when every span starts
    on a 16-byte boundary, else the 1-D bulk producer."""
    dev = device()
    n = rows * cols
    A = synth.uniform_pm1_torch(rows + 3 * cols, n, dev)
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, 1024)
    out = Guarded(n, 0, dev)
    ap.ap_row_roll(A, out.view, rows, cols, shift)
    assert ap.ap_check() == ap.AP_OK
    want = tensor_flags(ap, n, (shift % rows) * cols) if tensor else 0
    assert ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 12 == want
    assert_bits(to_np(out.view), orc.row_roll(to_np(A).reshape(rows, cols), shift), f"{rows}x{cols} shift {shift}")
    assert out.intact()


def test_roll_tensor_map_falls_back_when_misaligned(ap, orc):
    dev = device()
    rows, cols = 1000, 4
    src = Guarded(rows * cols, 1, dev, fill=synth.uniform_pm1_torch(5, rows * cols, dev))
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    out = Guarded(rows * cols, 0, dev)
    ap.ap_row_roll(src.view, out.view, rows, cols, 1)
    assert ap.ap_check() == ap.AP_OK
    assert not ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 4
    assert_bits(to_np(out.view), orc.row_roll(to_np(src.view).reshape(rows, cols), 1), "fallback")


@pytest.mark.parametrize("rows,cols,shift", [(1 << 26, 4, 1), (1 << 22, 64, 1), (1 << 26, 4, -12345)])
def test_roll_tensor_map_full_size(ap, orc, rows, cols, shift):
    """1 GiB through the tensor maps: whole stages as 2-D boxes of the line
    view, the stage that wraps as 1-D boxes."""
    import torch

    dev = device()
    A = synth.uniform_pm1_torch(synth.SEED_ROLL, rows * cols, dev)
    B = torch.empty_like(A)
    ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    ap.ap_row_roll(A, B, rows, cols, shift)
    assert ap.ap_check() == ap.AP_OK
    assert ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 12 == 12
    assert_bits(to_np(B), orc.row_roll(to_np(A).reshape(rows, cols), shift), f"full-size tensor roll {rows}x{cols}")

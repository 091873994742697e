"""The C-ABI library without a GPU: it builds, loads, exports every declared
symbol, rejects bad arguments before touching CUDA, and its tile planning
(run on the host by ap_debug_emulate_ring) moves every element to the right
place for any alignment, offset and stage size."""

import os
import re
import subprocess

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ap():
    from async_global_shared_gb300 import build

    build.build()
    import async_global_shared_gb300 as ap

    ap.load()
    return ap


def _declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(ap_\w+)\s*\(", text, flags=re.M))
    return names


def test_exports_every_declared_symbol(ap):
    declared = _declared_symbols()
    assert {"ap_scale", "ap_scale_sync", "ap_row_roll", "ap_poly", "ap_cluster_exchange", "ap_check"} <= declared
    nm = subprocess.run(["nm", "-D", "--defined-only", ap.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (ap_\w+)$", nm.stdout, flags=re.M))
    assert declared <= exported, f"declared but not exported: {declared - exported}"
    assert set(ap.EXPORTED) == declared
    lib = ap.load()
    for name in declared:
        assert hasattr(lib, name)


def test_status_strings(ap):
    for code, name in ap._lib.STATUS_NAMES.items():
        assert ap.ap_status_string(code) == name


FAKE_IN = 0x7F0000000000
FAKE_OUT = 0x7F0100000000


def raw(ap, fn, *args):
    return getattr(ap.load(), fn)(*args)


def test_validation_before_cuda(ap):
    # Every case below is rejected before any CUDA call (fake addresses are safe).
    assert raw(ap, "ap_scale", FAKE_IN, FAKE_OUT, 4, 256, 2.0, 1, None) == ap.AP_ERR_STAGES
    assert raw(ap, "ap_scale", FAKE_IN, FAKE_OUT, 4, 256, 2.0, 7, None) == ap.AP_ERR_STAGES
    assert raw(ap, "ap_scale", FAKE_IN, FAKE_OUT, -1, 256, 2.0, 2, None) == ap.AP_ERR_SHAPE
    assert raw(ap, "ap_scale", FAKE_IN, FAKE_OUT, 4, 0, 2.0, 2, None) == ap.AP_ERR_SHAPE
    assert raw(ap, "ap_scale", FAKE_IN, FAKE_OUT, 1 << 40, 1 << 40, 2.0, 2, None) == ap.AP_ERR_SHAPE
    assert raw(ap, "ap_scale", None, FAKE_OUT, 4, 256, 2.0, 2, None) == ap.AP_ERR_NULL
    assert raw(ap, "ap_scale", FAKE_IN + 2, FAKE_OUT, 4, 256, 2.0, 2, None) == ap.AP_ERR_ALIGN
    assert raw(ap, "ap_scale", FAKE_IN, FAKE_IN + 16, 4, 256, 2.0, 2, None) == ap.AP_ERR_ALIAS
    assert raw(ap, "ap_scale", None, None, 0, 256, 2.0, 2, None) == ap.AP_OK  # empty: no-op
    assert raw(ap, "ap_scale_sync", FAKE_IN, FAKE_OUT, 4, 1 << 20, 2.0, None) == ap.AP_ERR_SMEM
    assert raw(ap, "ap_scale_sync", FAKE_IN, FAKE_IN + 4, 4, 256, 2.0, None) == ap.AP_ERR_ALIAS
    assert raw(ap, "ap_row_roll", FAKE_IN, FAKE_OUT, -1, 4, 1, None) == ap.AP_ERR_SHAPE
    assert raw(ap, "ap_row_roll", FAKE_IN, FAKE_OUT, 0, 4, 1, None) == ap.AP_OK
    assert raw(ap, "ap_row_roll", FAKE_IN, FAKE_IN, 64, 4, 1, None) == ap.AP_ERR_ALIAS  # roll never in place
    assert raw(ap, "ap_row_roll", FAKE_IN, FAKE_OUT + 1, 64, 4, 1, None) == ap.AP_ERR_ALIGN
    assert raw(ap, "ap_poly", FAKE_IN, FAKE_OUT, 100, None, 3, 2, None) == ap.AP_ERR_NULL
    c = (np.zeros(2000, dtype=np.float32)).ctypes.data
    assert raw(ap, "ap_poly", FAKE_IN, FAKE_OUT, 100, c, -1, 2, None) == ap.AP_ERR_ARG
    assert raw(ap, "ap_poly", FAKE_IN, FAKE_OUT, 100, c, 1024, 2, None) == ap.AP_ERR_ARG
    assert raw(ap, "ap_poly", FAKE_IN, FAKE_OUT, 100, c, 8, 9, None) == ap.AP_ERR_STAGES
    assert raw(ap, "ap_cluster_exchange", FAKE_IN, FAKE_OUT, 1 << 20, 3, 32768, None) == ap.AP_ERR_CLUSTER
    assert raw(ap, "ap_cluster_exchange", FAKE_IN, FAKE_OUT, 1 << 20, 16, 32768, None) == ap.AP_ERR_CLUSTER
    assert raw(ap, "ap_cluster_exchange", FAKE_IN, FAKE_OUT, 1 << 20, 2, 24, None) == ap.AP_ERR_SHAPE
    assert raw(ap, "ap_cluster_exchange", FAKE_IN, FAKE_OUT, 1 << 20, 2, 128 * 1024, None) == ap.AP_ERR_SMEM
    assert raw(ap, "ap_cluster_exchange", FAKE_IN, FAKE_OUT, 1000, 4, 32768, None) == ap.AP_ERR_SHAPE
    assert raw(ap, "ap_cluster_exchange", FAKE_IN + 4, FAKE_OUT, 1 << 20, 2, 32768, None) == ap.AP_ERR_ALIGN
    assert raw(ap, "ap_cluster_exchange", FAKE_IN, FAKE_IN, 1 << 20, 2, 32768, None) == ap.AP_ERR_ALIAS
    mc = "ap_masked_copy"
    assert raw(ap, mc, FAKE_IN, FAKE_OUT, 100, FAKE_IN, 1, None) == ap.AP_ERR_STAGES
    assert raw(ap, mc, FAKE_IN, FAKE_OUT, 100, None, 2, None) == ap.AP_ERR_NULL
    assert raw(ap, mc, FAKE_IN + 4, FAKE_OUT, 100, FAKE_IN, 2, None) == ap.AP_ERR_ALIGN
    assert raw(ap, mc, FAKE_IN, FAKE_IN + 16, 100, FAKE_IN, 2, None) == ap.AP_ERR_ALIAS
    assert raw(ap, mc, FAKE_IN, FAKE_OUT, 0, None, 2, None) == ap.AP_OK
    import ctypes

    shape = ap._lib.RingShape()
    at = "ap_autotune"
    big = 1 << 20
    assert raw(ap, at, 9, FAKE_IN, FAKE_OUT, big, 2, 0, ctypes.byref(shape), None) == ap.AP_ERR_ARG
    assert raw(ap, at, ap.AP_TUNE_SCALE, FAKE_IN, FAKE_OUT, big, 7, 0, ctypes.byref(shape), None) == ap.AP_ERR_STAGES
    assert raw(ap, at, ap.AP_TUNE_SCALE, FAKE_IN, FAKE_OUT, 1000, 2, 0, ctypes.byref(shape), None) == ap.AP_ERR_SHAPE
    assert raw(ap, at, ap.AP_TUNE_POLY, FAKE_IN, FAKE_OUT, big, 2, 2000, ctypes.byref(shape), None) == ap.AP_ERR_ARG
    assert raw(ap, at, ap.AP_TUNE_SCALE, FAKE_IN, FAKE_OUT, big, 2, 0, None, None) == ap.AP_ERR_NULL
    assert raw(ap, at, ap.AP_TUNE_SCALE, FAKE_IN, FAKE_IN + 64, big, 2, 0, ctypes.byref(shape), None) == ap.AP_ERR_ALIAS
    assert raw(ap, "ap_autotune_reset") == ap.AP_OK
    ex = "ap_cluster_exchange_ex"
    assert raw(ap, ex, FAKE_IN, FAKE_OUT, 1 << 20, 0, 32768, 1, None) == ap.AP_ERR_CLUSTER
    assert raw(ap, ex, FAKE_IN, FAKE_OUT, 1 << 20, 17, 32768, 1, None) == ap.AP_ERR_CLUSTER
    assert raw(ap, ex, FAKE_IN, FAKE_OUT, 1000, 3, 32768, 1, None) == ap.AP_ERR_SHAPE  # not whole chunks
    assert raw(ap, ex, FAKE_IN, FAKE_OUT, 12, 3, 24, 1, None) == ap.AP_ERR_SHAPE  # chunk not a multiple of 16
    assert raw(ap, ex, FAKE_IN, FAKE_OUT, 0, 5, 32768, 7, None) == ap.AP_OK
    assert raw(ap, ex, FAKE_IN + 8, FAKE_OUT, 1 << 20, 5, 32768, 7, None) == ap.AP_ERR_ALIGN
    assert raw(ap, ex, FAKE_IN, FAKE_IN + 16, 1 << 20, 5, 32768, 7, None) == ap.AP_ERR_ALIAS
    a2a = "ap_cluster_all_to_all"
    assert raw(ap, a2a, FAKE_IN, FAKE_OUT, 1 << 20, 0, 32768, None) == ap.AP_ERR_CLUSTER
    assert raw(ap, a2a, FAKE_IN, FAKE_OUT, 1 << 20, 17, 32768, None) == ap.AP_ERR_CLUSTER
    assert raw(ap, a2a, FAKE_IN, FAKE_OUT, 1 << 20, 4, 32, None) == ap.AP_ERR_SHAPE  # sub-block of 8 bytes
    assert raw(ap, a2a, FAKE_IN, FAKE_OUT, 1 << 20, 3, 32768, None) == ap.AP_ERR_SHAPE  # 32768 not a multiple of 48
    assert raw(ap, a2a, FAKE_IN, FAKE_OUT, 3 * 8192, 4, 32768, None) == ap.AP_ERR_SHAPE  # 3 chunks: no whole group
    assert raw(ap, a2a, FAKE_IN, FAKE_OUT, 0, 4, 32768, None) == ap.AP_OK
    assert raw(ap, a2a, None, FAKE_OUT, 1 << 20, 4, 32768, None) == ap.AP_ERR_NULL
    assert raw(ap, a2a, FAKE_IN + 8, FAKE_OUT, 1 << 20, 4, 32768, None) == ap.AP_ERR_ALIGN
    assert raw(ap, a2a, FAKE_IN, FAKE_IN + 16, 1 << 20, 4, 32768, None) == ap.AP_ERR_ALIAS


def test_strict_alignment_switch(ap):
    """With AP_DBG_STRICT_ALIGN the ring calls refuse buffers off the 16-byte
    grid (before any CUDA call) instead of taking the cp.async fallback."""
    lib = ap.load()
    try:
        assert lib.ap_debug_set(ap.AP_DBG_STRICT_ALIGN, 2) == ap.AP_ERR_ARG
        ap.ap_debug_set(ap.AP_DBG_STRICT_ALIGN, 1)
        assert raw(ap, "ap_scale", FAKE_IN + 4, FAKE_OUT, 4, 256, 2.0, 2, None) == ap.AP_ERR_ALIGN
        assert raw(ap, "ap_scale", FAKE_IN, FAKE_OUT + 8, 4, 256, 2.0, 2, None) == ap.AP_ERR_ALIGN
        c = np.zeros(4, dtype=np.float32).ctypes.data
        assert raw(ap, "ap_poly", FAKE_IN + 12, FAKE_OUT, 100, c, 3, 2, None) == ap.AP_ERR_ALIGN
        assert raw(ap, "ap_row_roll", FAKE_IN, FAKE_OUT + 4, 64, 4, 1, None) == ap.AP_ERR_ALIGN
        assert raw(ap, "ap_scale", FAKE_IN + 4, FAKE_OUT, 0, 256, 2.0, 2, None) == ap.AP_OK  # empty stays a no-op
    finally:
        ap.ap_debug_set(ap.AP_DBG_STRICT_ALIGN, 0)
    if not __import__("torch").cuda.is_available():
        # without the switch a misaligned buffer passes validation (and fails at the first CUDA call here)
        assert raw(ap, "ap_scale", FAKE_IN + 4, FAKE_OUT, 4, 256, 2.0, 2, None) == ap.AP_ERR_CUDA


@pytest.mark.parametrize("value,want", [("tensor", 3), ("cpasync", 2), ("small", 2), ("bulk", 1), ("ring", 1),
                                        ("auto", 0), ("bogus", 0), ("3", 3)])
def test_force_path_environment_variable(value, want):
    """AP_FORCE_PATH chooses the path when ap_debug_set has not; an explicit
    setting still wins."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import async_global_shared_gb300 as ap; print(ap.ap_debug_get(ap.AP_DBG_FORCE_PATH)); "
            "ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 1); print(ap.ap_debug_get(ap.AP_DBG_FORCE_PATH))")
    env = dict(os.environ, AP_FORCE_PATH=value, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == [str(want), "1"]


def test_debug_settings_roundtrip(ap):
    lib = ap.load()
    assert lib.ap_debug_set(ap.AP_DBG_STAGE_BYTES, -5) == ap.AP_ERR_ARG
    assert lib.ap_debug_set(999, 1) == ap.AP_ERR_ARG
    assert lib.ap_debug_get(999) == -1
    for key, val in ((ap.AP_DBG_STAGE_BYTES, 4096), (ap.AP_DBG_GRID, 7), (ap.AP_DBG_TIMEOUT_NS, 12345)):
        ap.ap_debug_set(key, val)
        assert ap.ap_debug_get(key) == val
        ap.ap_debug_set(key, 0)
    assert ap.ap_debug_get(ap.AP_DBG_TIMEOUT_NS) > 0  # default limit applies when unset
    for bad in (3, 5, 16):
        assert lib.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, bad) == ap.AP_ERR_ARG
    for bad in (3, 8):
        assert lib.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, bad) == ap.AP_ERR_ARG
    for good in (1, 2, 4, 0):
        assert lib.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, good) == ap.AP_OK
    assert lib.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, 257) == ap.AP_ERR_ARG
    for good in (1, 2, 256, 0):
        assert lib.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, good) == ap.AP_OK
    for good in (1, 2, 4, 8, 0):
        assert lib.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, good) == ap.AP_OK
    for bad in (3, 5, 6, 32):
        assert lib.ap_debug_set(ap.AP_DBG_EXCHANGE_SEND_SLOTS, bad) == ap.AP_ERR_ARG
    for good in (1, 2, 4, 8, 16, 0):
        assert lib.ap_debug_set(ap.AP_DBG_EXCHANGE_SEND_SLOTS, good) == ap.AP_OK
    for removed in (10, 12):  # the cache-hint and stage-order keys gained nothing and were removed
        assert lib.ap_debug_set(removed, 0) == ap.AP_ERR_ARG
        assert lib.ap_debug_get(removed) == -1
    for good in (0, 1, 2, 12, 1 << 20):
        assert lib.ap_debug_set(ap.AP_DBG_RING_RUN, good) == ap.AP_OK
        assert ap.ap_debug_get(ap.AP_DBG_RING_RUN) == good
    assert lib.ap_debug_set(ap.AP_DBG_RING_RUN, (1 << 20) + 1) == ap.AP_ERR_ARG
    ap.ap_debug_set(ap.AP_DBG_RING_RUN, 0)
    for good in (0, 1, 2, 3):
        assert lib.ap_debug_set(ap.AP_DBG_CONSUMER_GROUPS, good) == ap.AP_OK
    assert lib.ap_debug_set(ap.AP_DBG_CONSUMER_GROUPS, 4) == ap.AP_ERR_ARG
    for good in (0, 8, 12, 16):
        assert lib.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, good) == ap.AP_OK
    for bad in (4, 15, 32):  # 15 warps left one SMSP a warp short and was replaced by 12
        assert lib.ap_debug_set(ap.AP_DBG_CONSUMER_WARPS, bad) == ap.AP_ERR_ARG
    for key in (ap.AP_DBG_LAST_RUN, ap.AP_DBG_LAST_WARPS, ap.AP_DBG_LAST_GROUPS, ap.AP_DBG_LAST_CHAINS):
        assert ap.ap_debug_get(key) >= 0  # read-only, known
        assert lib.ap_debug_set(key, 1) == ap.AP_ERR_ARG


@pytest.mark.skipif(
    __import__("torch").cuda.is_available(), reason="only meaningful where no CUDA device exists"
)
def test_valid_call_without_gpu_reports_cuda_error(ap):
    # Arguments pass validation; the first CUDA call then fails cleanly.
    st = raw(ap, "ap_scale", FAKE_IN, FAKE_OUT, 4, 256, 2.0, 2, None)
    assert st == ap.AP_ERR_CUDA


# ----------------------------------------------------------------- host emulation of the ring


def _emulate(ap, x, off, in_mis, out_mis, se):
    y = np.full_like(x, np.nan)
    st = ap.ap_debug_emulate_ring(x, y, x.size, off, in_mis, out_mis, se)
    return st, y


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 33, 64, 100, 255, 256, 257, 1000, 4099])
def test_emulated_ring_matches_oracle(ap, orc, n):
    x = synth.uniform_pm1_np(n, n)
    offs = sorted({0, 1, n - 1, n // 2, (7 * n) // 11} & set(range(n)))
    for se in (4, 8, 12, 64, 256):
        for off in offs:
            want = orc.row_roll(x.reshape(n, 1), off).ravel()
            for in_mis in (0, 4, 8, 12):
                for out_mis in (0, 4, 8, 12):
                    st, y = _emulate(ap, x, off, in_mis, out_mis, se)
                    assert st == ap.AP_OK, (n, off, in_mis, out_mis, se)
                    assert np.array_equal(y.view(np.uint32), want.view(np.uint32)), (n, off, in_mis, out_mis, se)


def test_emulated_ring_row_shift_geometry(ap, orc):
    # rows x cols matrices as the row shift drives the ring: off = shift * cols
    rng = np.random.default_rng(5)
    for _ in range(300):
        rows = int(rng.integers(1, 60))
        cols = int(rng.integers(1, 9))
        shift = int(rng.integers(-100, 100))
        se = int(rng.choice([4, 8, 16, 20, 64]))
        A = synth.uniform_pm1_np(rows * 100 + cols, rows * cols).reshape(rows, cols)
        s = shift % rows
        st, y = _emulate(ap, A.ravel(), s * cols, int(rng.choice([0, 4, 8, 12])), int(rng.choice([0, 4, 8, 12])), se)
        assert st == ap.AP_OK
        assert np.array_equal(y.reshape(rows, cols).view(np.uint32), orc.row_roll(A, shift).view(np.uint32))


def test_emulator_rejects_bad_arguments(ap):
    x = np.zeros(16, dtype=np.float32)
    y = np.zeros(16, dtype=np.float32)
    assert ap.ap_debug_emulate_ring(x, y, 16, 16, 0, 0, 4) == ap.AP_ERR_SHAPE
    assert ap.ap_debug_emulate_ring(x, y, 16, 0, 2, 0, 4) == ap.AP_ERR_ALIGN
    assert ap.ap_debug_emulate_ring(x, y, 16, 0, 0, 0, 6) == ap.AP_ERR_SHAPE


@pytest.mark.parametrize("line_boxes", [0, 1])
def test_emulated_tensor_ring_matches_oracle(ap, orc, line_boxes):
    """The tensor-map producer's plan: each stage one 2-D box of the line view
    (1 KiB lines from element off mod 256) where it fits, else 1-D boxes of
    256 floats from the span's first element (on a 16-byte boundary, zeros
    past the end); every element moved once. Shift 0 is the plain stream of
    scale and poly, any length."""
    rng = np.random.default_rng(9 + line_boxes)
    for _ in range(200):
        cols = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 64, 300]))
        rows = int(rng.integers(1, 6000 // cols + 2))
        stage_elems = 256 * int(rng.integers(1, 6))
        if rng.random() < 0.4:
            shift = 0
        else:
            # a shift whose element offset is a multiple of 4 (rows * cols too)
            rows = (rows + 3) // 4 * 4 if cols % 4 else rows
            step = 4 // np.gcd(cols, 4)
            shift = int(rng.integers(-rows, rows + 1)) * step
        n = rows * cols
        A = synth.uniform_pm1_np(n + 7, n).reshape(rows, cols)
        y = np.full(n, np.nan, dtype=np.float32)
        st = ap.ap_debug_emulate_ring_tensor(A.ravel(), y, rows, cols, shift, line_boxes, stage_elems)
        assert st == ap.AP_OK, (rows, cols, shift, stage_elems)
        assert np.array_equal(y.reshape(rows, cols).view(np.uint32), orc.row_roll(A, shift).view(np.uint32))
    x = np.zeros(64, dtype=np.float32)
    assert ap.ap_debug_emulate_ring_tensor(x, x.copy(), 64, 1, 1, line_boxes, 256) == ap.AP_ERR_ALIGN  # 4-byte offset
    assert ap.ap_debug_emulate_ring_tensor(x, x.copy(), 32, 2, 1, line_boxes, 256) == ap.AP_ERR_ALIGN  # 8 bytes
    assert ap.ap_debug_emulate_ring_tensor(x[:63], x[:63].copy(), 21, 3, 4, line_boxes, 256) == ap.AP_ERR_ALIGN
    assert ap.ap_debug_emulate_ring_tensor(x, x.copy(), 64, 1, 0, line_boxes, 128) == ap.AP_ERR_SHAPE  # not x256
    assert ap.ap_debug_emulate_ring_tensor(x, x.copy(), 16, 4, 4, line_boxes, 512) == ap.AP_OK
    assert ap.ap_debug_emulate_ring_tensor(x, x.copy(), 16, 4, 4, 2, 512) == ap.AP_ERR_ARG


def test_emulated_tensor_ring_large_line_view(ap, orc):
    """Many whole-stage 2-D boxes: a 2**18 x 4 shift by 1 (line view from
    element 4) and a plain stream with a ragged end."""
    for rows, cols, shift, se in ((1 << 18, 4, 1, 6144), (1 << 18, 4, -77, 4096), (100003, 1, 0, 4096)):
        A = synth.uniform_pm1_np(rows, rows * cols).reshape(rows, cols)
        y = np.full(rows * cols, np.nan, dtype=np.float32)
        assert ap.ap_debug_emulate_ring_tensor(A.ravel(), y, rows, cols, shift, 1, se) == ap.AP_OK
        assert np.array_equal(y.reshape(rows, cols).view(np.uint32), orc.row_roll(A, shift).view(np.uint32))


def test_binding_refuses_pageable_host_tensors(ap):
    """The binding passes CUDA tensors and pinned host tensors; an ordinary
    (pageable) host tensor is refused before any library call."""
    import torch

    x = torch.zeros(256)
    with pytest.raises(TypeError):
        ap.ap_scale(x, x, 1, 256, 2.0, 2)
    with pytest.raises(TypeError):
        ap.ap_scale(torch.zeros(256, dtype=torch.float64), x, 1, 256, 2.0, 2)

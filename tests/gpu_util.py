"""Helpers for the GPU parity tests (imported only by tests marked gpu)."""

from __future__ import annotations

import numpy as np

GUARD = 1024  # floats of sentinel on each side of a guarded buffer (4 KiB)
SENTINEL_BITS = 0x7FC0DEAD


def lib():
    from async_global_shared_gb300 import build

    build.build()
    import async_global_shared_gb300 as ap

    ap.load()
    return ap


def device():
    import torch

    if not torch.cuda.is_available():
        import pytest

        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def reset_debug(ap):
    for key in (
        ap.AP_DBG_FORCE_PATH,
        ap.AP_DBG_EXPECT_TX_EXTRA,
        ap.AP_DBG_TIMEOUT_NS,
        ap.AP_DBG_STAGE_BYTES,
        ap.AP_DBG_GRID,
        ap.AP_DBG_CTAS_PER_SM,
        ap.AP_DBG_ROLL_STAGES,
        ap.AP_DBG_CONSUMER_WARPS,
        ap.AP_DBG_EXCHANGE_STORE,
        ap.AP_DBG_DEVICE_CHECKS,
        ap.AP_DBG_EXCHANGE_GROUP,
        ap.AP_DBG_EXCHANGE_SEND_SLOTS,
        ap.AP_DBG_STRICT_ALIGN,
        ap.AP_DBG_EXCHANGE_LANES,
        ap.AP_DBG_EXCHANGE_BATCH,
        ap.AP_DBG_RING_RUN,
        ap.AP_DBG_CONSUMER_GROUPS,
    ):
        ap.ap_debug_set(key, 0)


class Guarded:
    """A float32 device buffer of n elements starting `shift` floats past a
    16-byte boundary, with GUARD sentinel floats on each side."""

    def __init__(self, n: int, shift: int = 0, dev="cuda:0", fill=None):
        import torch

        self.n = n
        self.shift = shift
        self.base = torch.empty(n + 2 * GUARD + 4, dtype=torch.float32, device=dev)
        self.base.view(torch.int32).fill_(SENTINEL_BITS)
        self.lo = GUARD + shift
        self.view = self.base[self.lo : self.lo + n]
        if fill is not None:
            self.view.copy_(fill)
        assert self.view.data_ptr() % 16 == (4 * shift) % 16

    def intact(self) -> bool:
        import torch

        b = self.base.view(torch.int32)
        head = b[: self.lo]
        tail = b[self.lo + self.n :]
        return bool((head == SENTINEL_BITS).all().item()) and bool((tail == SENTINEL_BITS).all().item())


def to_np(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_bits(got, want, what: str, nan_equal: bool = False):
    g = np.ascontiguousarray(got, dtype=np.float32).ravel()
    w = np.ascontiguousarray(want, dtype=np.float32).ravel()
    assert g.shape == w.shape, f"{what}: shape {g.shape} vs {w.shape}"
    diff = g.view(np.uint32) != w.view(np.uint32)
    if nan_equal:
        diff &= ~(np.isnan(g) & np.isnan(w))
    bad = np.flatnonzero(diff)
    assert bad.size == 0, (
        f"{what}: {bad.size} of {g.size} differ; first {bad[:5].tolist()} got {g[bad[:5]].tolist()} "
        f"want {w[bad[:5]].tolist()}"
    )


def tensor_flags(ap, n: int, off: int) -> int:
    """LAST_FLAGS bits 2-3 the tensor-map producer should report for a stream
    of n floats read at offset off, from the stage size the call used: bit 2
    always; bit 3 when the line view (1 KiB lines from element off mod 256)
    holds at least one whole stage."""
    se = ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS)
    line_h = se // 256
    line_rows = (n - off % 256) // 256
    return 12 if 0 < line_h <= 256 and line_rows >= line_h else 4


def oracle_poly_threads(orc, x: np.ndarray, c: np.ndarray, threads: int | None = None) -> np.ndarray:
    """The oracle's Horner loop (orc_poly) over contiguous ranges of x, one
    range per host core (ctypes releases the GIL during each call). Each
    element is computed exactly as the single-threaded oracle computes it; the
    split only shares the work out for full-size checks."""
    import ctypes
    import os
    import threading

    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    c = np.ascontiguousarray(c, dtype=np.float32).ravel()
    y = np.empty_like(x)
    n = x.size
    threads = threads or max(1, len(os.sched_getaffinity(0)))
    fp = ctypes.POINTER(ctypes.c_float)
    rcs = [0] * threads

    def work(t, lo, hi):
        rcs[t] = orc._lib.orc_poly(x[lo:hi].ctypes.data_as(fp), y[lo:hi].ctypes.data_as(fp), hi - lo,
                                   c.ctypes.data_as(fp), c.size - 1)

    ths = [threading.Thread(target=work, args=(t, t * n // threads, (t + 1) * n // threads)) for t in range(threads)]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    assert all(rc == 0 for rc in rcs), "orc_poly rejected the degree"
    return y

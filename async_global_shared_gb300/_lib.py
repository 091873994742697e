"""ctypes binding of libasyncpipe: argument marshalling only.

Every function has the C entry point's name and arguments. Buffers may be
given as torch tensors (float32, on the current CUDA device, contiguous) or as
raw integer device addresses; ``stream`` may be a ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer, or None for torch's current stream. A status other
than AP_OK raises :class:`APError`. Nothing here computes: every step runs in
the library's CUDA kernels, and a missing library raises instead of falling
back to anything else.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libasyncpipe.so")

AP_OK = 0
STATUS_NAMES = {
    0: "AP_OK",
    1: "AP_ERR_NULL",
    2: "AP_ERR_SHAPE",
    3: "AP_ERR_ALIGN",
    4: "AP_ERR_ALIAS",
    5: "AP_ERR_STAGES",
    6: "AP_ERR_CLUSTER",
    7: "AP_ERR_SMEM",
    8: "AP_ERR_CUDA",
    9: "AP_ERR_DEVICE_TIMEOUT",
    10: "AP_ERR_UNSUPPORTED_DEVICE",
    11: "AP_ERR_ARG",
}
globals().update({name: code for code, name in STATUS_NAMES.items()})

AP_MIN_STAGES = 2
AP_MAX_STAGES = 6
AP_POLY_MAX_DEGREE = 1023

# ap_debug_key
AP_DBG_FORCE_PATH = 1
AP_DBG_EXPECT_TX_EXTRA = 2
AP_DBG_TIMEOUT_NS = 3
AP_DBG_STAGE_BYTES = 4
AP_DBG_GRID = 5
AP_DBG_CTAS_PER_SM = 6
AP_DBG_ROLL_STAGES = 7
AP_DBG_CONSUMER_WARPS = 8
AP_DBG_EXCHANGE_STORE = 9
AP_DBG_DEVICE_CHECKS = 11
AP_DBG_EXCHANGE_GROUP = 13
AP_DBG_STRICT_ALIGN = 14
AP_DBG_EXCHANGE_LANES = 15
AP_DBG_EXCHANGE_BATCH = 16
AP_DBG_EXCHANGE_SEND_SLOTS = 17
AP_DBG_RING_RUN = 18
AP_DBG_CONSUMER_GROUPS = 19
AP_DBG_LAST_PATH = 100
AP_DBG_LAST_GRID = 101
AP_DBG_LAST_STAGE_ELEMS = 102
AP_DBG_LAST_SMEM = 103
AP_DBG_LAST_STAGES = 104
AP_DBG_LAST_FLAGS = 105
AP_DBG_LAST_SITE = 106
AP_DBG_LAST_RUN = 107
AP_DBG_LAST_WARPS = 108
AP_DBG_LAST_GROUPS = 109
AP_DBG_LAST_CHAINS = 110

# Every symbol the headers under include/ declare.
EXPORTED = (
    "ap_scale",
    "ap_scale_sync",
    "ap_row_roll",
    "ap_poly",
    "ap_cluster_exchange",
    "ap_cluster_exchange_ex",
    "ap_cluster_all_to_all",
    "ap_masked_copy",
    "ap_autotune",
    "ap_autotune_reset",
    "ap_check",
    "ap_status_string",
    "ap_debug_set",
    "ap_debug_get",
    "ap_debug_emulate_ring",
    "ap_debug_emulate_ring_tensor",
    "ap_debug_fma_probe",
    "ap_debug_fma_probe_horner",
    "ap_debug_scale_pages_async",
)


AP_TUNE_SCALE = 1
AP_TUNE_ROW_ROLL = 2
AP_TUNE_POLY = 3


class RingShape(ctypes.Structure):
    _fields_ = [("stage_bytes", ctypes.c_int64), ("ctas_per_sm", ctypes.c_int), ("consumer_warps", ctypes.c_int),
                ("stages_per_cta", ctypes.c_int), ("consumer_groups", ctypes.c_int), ("gbs", ctypes.c_double)]


class APError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call} failed: {STATUS_NAMES.get(status, status)}")


_lib = None
_f32p = ctypes.c_void_p
_i64 = ctypes.c_int64


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libasyncpipe.so (built by ``async_global_shared_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libasyncpipe is not built ({p} missing); run `python -c \"import __graft_entry__ as g; g.build()\"`"
        )
    lib = ctypes.CDLL(p)
    vp = ctypes.c_void_p
    lib.ap_scale.argtypes = [vp, vp, _i64, _i64, ctypes.c_float, ctypes.c_int, vp]
    lib.ap_scale_sync.argtypes = [vp, vp, _i64, _i64, ctypes.c_float, vp]
    lib.ap_row_roll.argtypes = [vp, vp, _i64, _i64, _i64, vp]
    lib.ap_poly.argtypes = [vp, vp, _i64, vp, ctypes.c_int, ctypes.c_int, vp]
    lib.ap_cluster_exchange.argtypes = [vp, vp, _i64, ctypes.c_int, _i64, vp]
    lib.ap_cluster_exchange_ex.argtypes = [vp, vp, _i64, ctypes.c_int, _i64, _i64, vp]
    lib.ap_cluster_all_to_all.argtypes = [vp, vp, _i64, ctypes.c_int, _i64, vp]
    lib.ap_masked_copy.argtypes = [vp, vp, _i64, vp, ctypes.c_int, vp]
    lib.ap_autotune.argtypes = [ctypes.c_int, vp, vp, _i64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(RingShape), vp]
    lib.ap_autotune_reset.argtypes = []
    lib.ap_check.argtypes = [vp]
    lib.ap_status_string.argtypes = [ctypes.c_int]
    lib.ap_status_string.restype = ctypes.c_char_p
    lib.ap_debug_set.argtypes = [ctypes.c_int, _i64]
    lib.ap_debug_get.argtypes = [ctypes.c_int]
    lib.ap_debug_get.restype = _i64
    lib.ap_debug_emulate_ring.argtypes = [vp, vp, _i64, _i64, ctypes.c_int, ctypes.c_int, _i64]
    lib.ap_debug_fma_probe.argtypes = [vp, _i64, _i64, vp]
    lib.ap_debug_fma_probe_horner.argtypes = [vp, _i64, _i64, vp]
    lib.ap_debug_scale_pages_async.argtypes = [vp, vp, _i64, _i64, ctypes.c_float, vp]
    lib.ap_debug_emulate_ring_tensor.argtypes = [vp, vp, _i64, _i64, _i64, _i64, _i64]
    for name in ("ap_scale", "ap_scale_sync", "ap_row_roll", "ap_poly", "ap_cluster_exchange",
                 "ap_cluster_exchange_ex", "ap_cluster_all_to_all", "ap_masked_copy", "ap_autotune", "ap_autotune_reset", "ap_check",
                 "ap_debug_set", "ap_debug_emulate_ring", "ap_debug_emulate_ring_tensor", "ap_debug_fma_probe",
                 "ap_debug_fma_probe_horner", "ap_debug_scale_pages_async"):
        getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _addr(buf) -> int | None:
    """Device-accessible address of a tensor (checked: float32, contiguous, on
    the GPU or in pinned host memory, which the GPU reads and writes over the
    host link) or an int."""
    if buf is None:
        return None
    if isinstance(buf, int):
        return buf
    if hasattr(buf, "data_ptr"):
        import torch

        if buf.dtype != torch.float32:
            raise TypeError("libasyncpipe works on float32 tensors")
        if not buf.is_cuda and not buf.is_pinned():
            raise TypeError("libasyncpipe needs CUDA tensors or pinned host tensors")
        if not buf.is_contiguous():
            raise TypeError("libasyncpipe needs contiguous tensors")
        return buf.data_ptr()
    raise TypeError(f"cannot take a device address of {type(buf).__name__}")


_cuda_available = None  # torch.cuda.is_available(), asked once


def _current_stream() -> int | None:
    """torch's current CUDA stream on the current device, as a raw handle."""
    global _cuda_available
    try:
        import torch
    except ImportError:
        return None
    if _cuda_available is None:
        _cuda_available = bool(torch.cuda.is_available())
    if not _cuda_available:
        return None
    # The raw handle without building a Stream object (about 0.3 us against
    # 3 us for current_stream() per call); the public call where a torch
    # build lacks it.
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch._C._cuda_getDevice())
    return torch.cuda.current_stream().cuda_stream


def _stream(stream) -> int | None:
    if stream is None:
        return _current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, call: str):
    if status != AP_OK:
        raise APError(status, call)


def ap_scale(inp, out, n_tiles: int, tile_elems: int, alpha: float, stages: int, stream=None):
    _check(load().ap_scale(_addr(inp), _addr(out), n_tiles, tile_elems, alpha, stages, _stream(stream)), "ap_scale")


def ap_scale_sync(inp, out, n_tiles: int, tile_elems: int, alpha: float, stream=None):
    _check(load().ap_scale_sync(_addr(inp), _addr(out), n_tiles, tile_elems, alpha, _stream(stream)),
           "ap_scale_sync")


def ap_row_roll(A, B, rows: int, cols: int, shift: int, stream=None):
    _check(load().ap_row_roll(_addr(A), _addr(B), rows, cols, shift, _stream(stream)), "ap_row_roll")


def ap_poly(inp, out, n: int, coeffs, degree: int, stages: int, stream=None):
    """``coeffs`` is a HOST sequence of degree + 1 floats (copied by the call)."""
    c = (ctypes.c_float * max(1, len(coeffs)))(*[float(v) for v in coeffs])
    if len(coeffs) < degree + 1:
        raise ValueError("ap_poly needs degree + 1 coefficients")
    _check(load().ap_poly(_addr(inp), _addr(out), n, ctypes.cast(c, ctypes.c_void_p), degree, stages,
                          _stream(stream)), "ap_poly")


def ap_cluster_exchange(inp, out, n: int, cluster_size: int, chunk_bytes: int, stream=None):
    _check(load().ap_cluster_exchange(_addr(inp), _addr(out), n, cluster_size, chunk_bytes, _stream(stream)),
           "ap_cluster_exchange")


def ap_cluster_exchange_ex(inp, out, n: int, cluster_size: int, chunk_bytes: int, shift: int, stream=None):
    _check(load().ap_cluster_exchange_ex(_addr(inp), _addr(out), n, cluster_size, chunk_bytes, shift,
                                         _stream(stream)), "ap_cluster_exchange_ex")


def ap_cluster_all_to_all(inp, out, n: int, cluster_size: int, chunk_bytes: int, stream=None):
    _check(load().ap_cluster_all_to_all(_addr(inp), _addr(out), n, cluster_size, chunk_bytes, _stream(stream)),
           "ap_cluster_all_to_all")


def ap_masked_copy(inp, out, n_chunks: int, codes, stages: int, stream=None):
    """``codes``: a CUDA int8 tensor (or device address) of n_chunks codes."""
    if hasattr(codes, "data_ptr"):
        import torch

        if codes.dtype != torch.int8 or not codes.is_cuda or not codes.is_contiguous():
            raise TypeError("codes must be a contiguous CUDA int8 tensor")
        codes = codes.data_ptr()
    _check(load().ap_masked_copy(_addr(inp), _addr(out), n_chunks, codes, stages, _stream(stream)),
           "ap_masked_copy")


def ap_autotune(op: int, inp, out, n: int, stages: int, degree: int = 0, stream=None) -> dict:
    """Time the ring's shapes over inp/out, install the fastest; returns it."""
    shape = RingShape()
    _check(load().ap_autotune(op, _addr(inp), _addr(out), n, stages, degree, ctypes.byref(shape), _stream(stream)),
           "ap_autotune")
    return {"stage_bytes": shape.stage_bytes, "ctas_per_sm": shape.ctas_per_sm,
            "consumer_warps": shape.consumer_warps, "stages_per_cta": shape.stages_per_cta,
            "consumer_groups": shape.consumer_groups, "gbs": shape.gbs}


def ap_autotune_reset():
    _check(load().ap_autotune_reset(), "ap_autotune_reset")


def ap_check(stream=None) -> int:
    """Wait for the stream and return (not raise) the device status, then clear it."""
    return load().ap_check(_stream(stream))


def ap_status_string(status: int) -> str:
    return load().ap_status_string(status).decode()


def ap_debug_set(key: int, value: int):
    _check(load().ap_debug_set(key, value), "ap_debug_set")


def ap_debug_get(key: int) -> int:
    return load().ap_debug_get(key)


def ap_debug_emulate_ring(in_host, out_host, n: int, off: int, in_mis: int, out_mis: int, stage_elems: int) -> int:
    """Host emulation (numpy float32 arrays); returns the status code."""
    import numpy as np

    assert in_host.dtype == np.float32 and out_host.dtype == np.float32
    return load().ap_debug_emulate_ring(in_host.ctypes.data, out_host.ctypes.data, n, off, in_mis, out_mis,
                                        stage_elems)


def ap_debug_emulate_ring_tensor(in_host, out_host, rows: int, cols: int, shift: int, line_boxes: int,
                                 stage_elems: int) -> int:
    """Host emulation of the tensor-map producer's row shift (numpy float32 arrays); returns the status code."""
    import numpy as np

    assert in_host.dtype == np.float32 and out_host.dtype == np.float32
    return load().ap_debug_emulate_ring_tensor(in_host.ctypes.data, out_host.ctypes.data, rows, cols, shift,
                                               line_boxes, stage_elems)


def ap_debug_fma_probe(out, out_elems: int, iters: int, stream=None):
    _check(load().ap_debug_fma_probe(_addr(out), out_elems, iters, _stream(stream)), "ap_debug_fma_probe")


def ap_debug_fma_probe_horner(out, out_elems: int, iters: int, stream=None):
    _check(load().ap_debug_fma_probe_horner(_addr(out), out_elems, iters, _stream(stream)),
           "ap_debug_fma_probe_horner")


def ap_debug_scale_pages_async(inp, out, n_tiles: int, tile_elems: int, alpha: float, stream=None):
    _check(load().ap_debug_scale_pages_async(_addr(inp), _addr(out), n_tiles, tile_elems, alpha, _stream(stream)),
           "ap_debug_scale_pages_async")

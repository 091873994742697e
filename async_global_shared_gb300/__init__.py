"""async_global_shared_gb300: Python binding of libasyncpipe.

libasyncpipe streams float32 tiles from global to shared memory through an
mbarrier-tracked ring of asynchronous bulk copies on GB300 (sm_103a) and
computes on them: scale, row shift, Horner polynomial, and a CTA-to-CTA
shared-memory hand-off inside a thread-block cluster. The C interface is
declared in ``include/asyncpipe.h``; these functions carry the same names and
arguments and only marshal them. PyTorch provides device memory and streams.
"""

from ._lib import *  # noqa: F401,F403
from ._lib import APError, EXPORTED, LIB_PATH, load  # noqa: F401

__all__ = [
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
    "APError",
    "load",
]

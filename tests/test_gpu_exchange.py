"""ap_cluster_exchange against the oracle, bit for bit. Cluster sizes 4 and 8
tell the hand-off direction apart (for 2 both directions agree)."""

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


@pytest.mark.parametrize("store,group", [(1, 0), (2, 0), (2, 1), (2, 2), (2, 4), (2, 8)])
@pytest.mark.parametrize("cs", [1, 2, 4, 8])
@pytest.mark.parametrize("chunk_bytes,groups", [(16, 1), (16, 37), (48, 5), (1024, 300), (32768, 3), (100000, 4)])
def test_exchange_small(ap, orc, cs, chunk_bytes, groups, store, group):
    """Both receiver forms; the warp form with 1, 2, 4 or 8 warps per piece
    (8, 4, 2 or 1 pieces draining at once) and its automatic choice."""
    dev = device()
    n = groups * cs * chunk_bytes // 4
    x = synth.uniform_pm1_torch(n + cs, n, dev)
    want = orc.cluster_exchange(to_np(x), cs, chunk_bytes)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_STORE, store)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, group)
    # grid cs: one cluster walks every group; CTAs/SM 3 gives a ring depth the
    # loader and pusher lanes (2 or 4) divide
    for grid, piece, lanes, cps in ((0, 0, 0, 0), (cs, 0, 2, 0), (cs, 16, 4, 0), (0, 4096, 4, 3), (0, 1024, 2, 3)):
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, piece)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, lanes)
        ap.ap_debug_set(ap.AP_DBG_CTAS_PER_SM, cps)
        out = Guarded(n, 0, dev)
        ap.ap_cluster_exchange(x, out.view, n, cs, chunk_bytes)
        assert ap.ap_check() == ap.AP_OK
        assert ap.ap_debug_get(ap.AP_DBG_LAST_PATH) == 4
        assert_bits(to_np(out.view), want,
                    f"exchange cs={cs} chunk={chunk_bytes} groups={groups} grid={grid} piece={piece} store={store} "
                    f"lanes={lanes} cps={cps}")
        assert out.intact()


def test_exchange_worked_example(ap, orc):
    import torch

    dev = device()
    x = torch.arange(16, dtype=torch.float32, device=dev)
    # 16-byte chunks, cluster of 4 -> 4 chunks per group, 1 group
    y = torch.empty_like(x)
    ap.ap_cluster_exchange(x, y, 16, 4, 16)
    assert ap.ap_check() == ap.AP_OK
    assert to_np(y).tolist() == [4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 0, 1, 2, 3]


@pytest.mark.parametrize("send", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("store,group", [(1, 0), (2, 8), (2, 1)])
@pytest.mark.parametrize("cs", [1, 2, 4, 8])
def test_exchange_split_rings(ap, orc, cs, store, group, send):
    """The fixed-neighbour hand-off with a split send ring (forced: it is
    automatic only for the all-to-all), plain pieces and batches."""
    dev = device()
    for chunk_bytes, groups, batch in ((32768, 5, 0), (4096, 61, 0), (256, 700, 0), (1024, 90, 8)):
        n = groups * cs * chunk_bytes // 4
        x = synth.uniform_pm1_torch(n + 3 * cs, n, dev)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_SEND_SLOTS, send)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_STORE, store)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, group)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, batch)
        out = Guarded(n, 0, dev)
        ap.ap_cluster_exchange(x, out.view, n, cs, chunk_bytes)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), orc.cluster_exchange(to_np(x), cs, chunk_bytes),
                    f"exchange cs={cs} chunk={chunk_bytes} send={send} store={store} group={group}")
        assert out.intact()


@pytest.mark.parametrize("cs", [2, 4, 8])
def test_exchange_full_size(ap, orc, cs):
    """2**28 floats (1 GiB) in 32 KiB chunks: 32768 chunks, 32768/cs groups."""
    import torch

    dev = device()
    n = 1 << 28
    x = synth.uniform_pm1_torch(synth.SEED_EXCHANGE, n, dev)
    want = orc.cluster_exchange(to_np(x), cs, 32768)
    for store in (0, 1, 2):
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_STORE, store)
        y = torch.full_like(x, float("nan"))
        ap.ap_cluster_exchange(x, y, n, cs, 32768)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(y), want, f"full exchange cs={cs} store={store}")


@pytest.mark.parametrize("batch", [0, 1, 2, 8, 64, 256])
@pytest.mark.parametrize("cs", [1, 2, 4, 8])
@pytest.mark.parametrize("chunk_bytes,groups", [(16, 1), (16, 1000), (48, 37), (256, 513), (1024, 300), (4096, 77),
                                                (2064, 9)])
def test_exchange_batched(ap, orc, cs, chunk_bytes, groups, batch):
    """The batched form: one tensor-map box gathers a rank's chunk from
    `batch` consecutive groups (0: automatic for chunks under 8 KiB, 1: never),
    and the last, partial batch is clipped at the tensor's edge."""
    dev = device()
    n = groups * cs * chunk_bytes // 4
    x = synth.uniform_pm1_torch(n + 3 * cs, n, dev)
    want = orc.cluster_exchange(to_np(x), cs, chunk_bytes)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, batch)
    for grid in (0, cs):
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        out = Guarded(n, 0, dev)
        ap.ap_cluster_exchange(x, out.view, n, cs, chunk_bytes)
        assert ap.ap_check() == ap.AP_OK
        batched = bool(ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 4)
        eligible = chunk_bytes // 4 <= 256 or chunk_bytes // 4 % 256 == 0
        if batch == 1 or not eligible:
            assert not batched
        elif batch >= 2 or chunk_bytes < 8192:
            assert batched
        assert_bits(to_np(out.view), want,
                    f"batched exchange cs={cs} chunk={chunk_bytes} groups={groups} batch={batch} grid={grid}")
        assert out.intact()

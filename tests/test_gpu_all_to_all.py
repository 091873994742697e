"""ap_cluster_all_to_all against the oracle, bit for bit: every CTA of a
cluster sends sub-block j of its chunk to rank j (the block transpose of each
group's sub-blocks), for cluster sizes 1..16 (above 8 with the non-portable
cluster attribute), sub-blocks from one 16-byte unit to several pieces, and
clusters that walk many groups through a ring reused many times."""

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


@pytest.mark.parametrize("cs", [1, 2, 3, 4, 5, 8, 12, 16])
@pytest.mark.parametrize("sub_bytes", [16, 48, 1024, 4096])
def test_all_to_all_small(ap, orc, cs, sub_bytes):
    dev = device()
    chunk_bytes = cs * sub_bytes
    for groups in (1, 3, 40):
        n = groups * cs * chunk_bytes // 4
        x = synth.uniform_pm1_torch(n + cs, n, dev)
        want = orc.cluster_all_to_all(to_np(x), cs, chunk_bytes)
        # defaults, then small pieces, few slots and one cluster (every slot
        # goes through many phases, items of one sender spread over groups)
        for piece, grid, cps in ((0, 0, 0), (16, cs, 0), (512, 2 * cs, 4), (2048, 0, 1)):
            ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, piece)
            ap.ap_debug_set(ap.AP_DBG_GRID, grid)
            ap.ap_debug_set(ap.AP_DBG_CTAS_PER_SM, cps)
            out = Guarded(n, 0, dev)
            ap.ap_cluster_all_to_all(x, out.view, n, cs, chunk_bytes)
            assert ap.ap_check() == ap.AP_OK
            assert ap.ap_debug_get(ap.AP_DBG_LAST_STAGES) % cs == 0, "ring depth must be a multiple of cs"
            assert_bits(to_np(out.view), want, f"a2a cs={cs} sub={sub_bytes} groups={groups} piece={piece} grid={grid}")
            assert out.intact()


def test_all_to_all_twice_is_identity(ap):
    import torch

    dev = device()
    n = 1 << 20
    x = synth.uniform_pm1_torch(11, n, dev)
    a = torch.empty_like(x)
    b = torch.empty_like(x)
    for cs in (2, 4, 8, 16):
        ap.ap_cluster_all_to_all(x, a, n, cs, 16384)
        ap.ap_cluster_all_to_all(a, b, n, cs, 16384)
        assert ap.ap_check() == ap.AP_OK
        assert torch.equal(b.view(torch.int32), x.view(torch.int32)), f"cs={cs}"


@pytest.mark.parametrize("lanes", [1, 2, 4])
@pytest.mark.parametrize("store,group", [(1, 0), (2, 1), (2, 2), (2, 4), (2, 8)])
@pytest.mark.parametrize("cs", [1, 3, 4, 8, 16])
def test_all_to_all_receiver_forms(ap, orc, cs, store, group, lanes):
    """The TMA-store receiver and the warp receiver with 1, 2, 4 or 8 warps
    per piece, with 1, 2 or 4 loader and pusher lanes, over many groups and
    ring shapes."""
    dev = device()
    for sub_bytes, groups, piece, grid in ((16, 9, 0, 0), (1024, 40, 0, cs), (4096, 7, 1024, 0), (2048, 33, 0, 3 * cs)):
        chunk_bytes = cs * sub_bytes
        n = groups * cs * chunk_bytes // 4
        x = synth.uniform_pm1_torch(n + 7 * cs, n, dev)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_STORE, store)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, group)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, lanes)
        ap.ap_debug_set(ap.AP_DBG_STAGE_BYTES, piece)
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        out = Guarded(n, 0, dev)
        ap.ap_cluster_all_to_all(x, out.view, n, cs, chunk_bytes)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), orc.cluster_all_to_all(to_np(x), cs, chunk_bytes),
                    f"a2a cs={cs} sub={sub_bytes} groups={groups} store={store} group={group} lanes={lanes}")
        assert out.intact()


@pytest.mark.parametrize("send", [0, 1, 2, 4, 8, 16])
@pytest.mark.parametrize("store,group,lanes", [(1, 0, 1), (2, 1, 1), (2, 2, 2), (2, 8, 4)])
@pytest.mark.parametrize("cs", [2, 4, 8, 16])
def test_all_to_all_split_rings(ap, orc, cs, store, group, lanes, send):
    """Send rings of 2-16 buffers beside deeper receive rings (freed when a
    piece lands), never split (1) and automatic (0), under every receiver
    form, plain pieces and batches, over many groups."""
    dev = device()
    for sub_bytes, groups, batch, grid in ((1024, 40, 0, cs), (4096, 9, 1, 0), (256, 130, 0, 2 * cs), (2048, 33, 0, 0)):
        chunk_bytes = cs * sub_bytes
        n = groups * cs * chunk_bytes // 4
        x = synth.uniform_pm1_torch(n + 11 * cs, n, dev)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_SEND_SLOTS, send)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_STORE, store)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_GROUP, group)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_LANES, lanes)
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, batch)
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        out = Guarded(n, 0, dev)
        ap.ap_cluster_all_to_all(x, out.view, n, cs, chunk_bytes)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), orc.cluster_all_to_all(to_np(x), cs, chunk_bytes),
                    f"a2a cs={cs} sub={sub_bytes} groups={groups} send={send} store={store} group={group}")
        assert out.intact()


@pytest.mark.parametrize("chunk_bytes,groups", [(32768, 1), (32768, 300), (65536, 97), (40960, 61)])
def test_all_to_all_three_ctas_per_sm(ap, orc, chunk_bytes, groups):
    """Clusters of 8 with sub-blocks of 4 KiB or more run three CTAs per SM
    (8 send and 8 receive slots of 4 KiB, the register-capped instantiation):
    more CTAs than two a SM are resident, and the result is bit-exact, from
    one group to many rounds of the ring; an explicit CTAs-per-SM setting of
    two plans the two-CTA ring instead."""
    import torch

    dev = device()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cs = 8
    n = groups * cs * chunk_bytes // 4
    x = synth.uniform_pm1_torch(n + 3, n, dev)
    want = orc.cluster_all_to_all(to_np(x), cs, chunk_bytes)
    for cps in (0, 2):
        ap.ap_debug_set(ap.AP_DBG_CTAS_PER_SM, cps)
        out = Guarded(n, 0, dev)
        ap.ap_cluster_all_to_all(x, out.view, n, cs, chunk_bytes)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), want, f"a2a cs=8 chunk={chunk_bytes} groups={groups} cps={cps}")
        assert out.intact()
        if chunk_bytes in (32768, 65536):  # 4 KiB pieces either way; 40 KiB chunks take 1280-byte pieces
            assert ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS) == 1024
            assert ap.ap_debug_get(ap.AP_DBG_LAST_STAGES) == (8 if cps == 0 else 16)
        if cps == 0 and groups >= 60:
            assert ap.ap_debug_get(ap.AP_DBG_LAST_GRID) > 2 * sms, "three CTAs a SM expected"


@pytest.mark.parametrize("cs", [2, 4, 8, 16])
def test_all_to_all_full_size(ap, orc, cs):
    """2**28 floats in 32 KiB chunks (32768 chunks)."""
    import torch

    dev = device()
    n = 1 << 28
    x = synth.uniform_pm1_torch(synth.SEED_EXCHANGE, n, dev)
    y = torch.full_like(x, float("nan"))
    ap.ap_cluster_all_to_all(x, y, n, cs, 32768)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.cluster_all_to_all(to_np(x), cs, 32768), f"full all-to-all cs={cs}")


@pytest.mark.parametrize("batch", [0, 1, 8, 32])
@pytest.mark.parametrize("cs", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("sub_bytes,groups", [(16, 3), (16, 700), (48, 51), (256, 129), (1024, 33), (2048, 12)])
def test_all_to_all_batched(ap, orc, cs, sub_bytes, groups, batch):
    """The batched all-to-all: one box gathers a rank's sub-block j from
    `batch` consecutive groups and lands as sub-block r of rank j's chunks."""
    dev = device()
    chunk_bytes = cs * sub_bytes
    n = groups * cs * chunk_bytes // 4
    x = synth.uniform_pm1_torch(n + 5 * cs, n, dev)
    want = orc.cluster_all_to_all(to_np(x), cs, chunk_bytes)
    ap.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, batch)
    for grid in (0, cs):
        ap.ap_debug_set(ap.AP_DBG_GRID, grid)
        out = Guarded(n, 0, dev)
        ap.ap_cluster_all_to_all(x, out.view, n, cs, chunk_bytes)
        assert ap.ap_check() == ap.AP_OK
        if batch == 1:
            assert not ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS) & 4
        assert_bits(to_np(out.view), want, f"batched a2a cs={cs} sub={sub_bytes} groups={groups} batch={batch}")
        assert out.intact()


@pytest.mark.parametrize("op,cs", [("exchange", 4), ("all_to_all", 8), ("exchange_ex", 16)])
def test_beyond_2p32_elements(ap, orc, op, cs):
    """2^32 + 65536 floats (16 GiB in and 16 GiB out) in 32 KiB chunks, so
    chunk and byte offsets pass 2^32 and 2^34: the cluster hand-off, the
    all-to-all over clusters of 8 in its three-CTA form, and the generalised
    hand-off over 16-CTA clusters with shift 5 and a short last group of 8
    chunks (run as a second launch). Checked group by group against the oracle
    (a group of cs chunks is self-contained) at the first and last 64 groups
    and 256 random ones."""
    import torch

    dev = device()
    chunk = 32768
    e = chunk // 4
    n = (1 << 32) + 65536
    g = torch.Generator(device=dev)
    g.manual_seed(0xA5A6)
    x = torch.empty(n, dtype=torch.float32, device=dev).uniform_(-1.0, 1.0, generator=g)
    y = torch.full((n,), float("nan"), dtype=torch.float32, device=dev)
    if op == "exchange":
        ap.ap_cluster_exchange(x, y, n, cs, chunk)
    elif op == "all_to_all":
        ap.ap_cluster_all_to_all(x, y, n, cs, chunk)
    else:
        ap.ap_cluster_exchange_ex(x, y, n, cs, chunk, 5)
    assert ap.ap_check() == ap.AP_OK
    groups = -(-n // (cs * e))  # the last one short for the 16-CTA hand-off
    rng = np.random.default_rng(5)
    pick = sorted(set(list(range(64)) + list(range(groups - 64, groups)) + [int(v) for v in rng.integers(0, groups, 256)]))
    for grp in pick:
        lo, hi = grp * cs * e, min(n, (grp + 1) * cs * e)
        xg = to_np(x[lo:hi])
        if op == "exchange":
            want = orc.cluster_exchange(xg, cs, chunk)
        elif op == "all_to_all":
            want = orc.cluster_all_to_all(xg, cs, chunk)
        else:
            want = orc.cluster_exchange_ex(xg, cs, chunk, 5)
        assert_bits(to_np(y[lo:hi]), want, f"{op} cs={cs} beyond 2^32, group {grp} of {groups}")

"""ap_cluster_exchange_ex against the oracle, bit for bit: cluster sizes
1..16 (above 8 with the non-portable cluster attribute), any shift, and a
short last group (a second launch with a cluster of the leftover chunks)."""

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


@pytest.mark.parametrize("cs", [1, 2, 3, 5, 7, 8, 12, 16])
@pytest.mark.parametrize("chunk_bytes,chunks_extra", [(16, 0), (48, 1), (1024, 0), (8192, 3), (32768, 1)])
def test_exchange_ex_small(ap, orc, cs, chunk_bytes, chunks_extra):
    dev = device()
    chunks = 5 * cs + (chunks_extra % cs if cs > 1 else 0)
    n = chunks * chunk_bytes // 4
    x = synth.uniform_pm1_torch(n + cs, n, dev)
    for shift in (1, 0, -1, 3, cs + 2, -(10**9) - 7):
        out = Guarded(n, 0, dev)
        ap.ap_cluster_exchange_ex(x, out.view, n, cs, chunk_bytes, shift)
        assert ap.ap_check() == ap.AP_OK
        assert_bits(to_np(out.view), orc.cluster_exchange_ex(to_np(x), cs, chunk_bytes, shift),
                    f"exchange_ex cs={cs} chunk={chunk_bytes} chunks={chunks} shift={shift}")
        assert out.intact()


def test_exchange_ex_matches_fixed_neighbour(ap, orc):
    import torch

    dev = device()
    n = 8 * 4 * 8192 // 4
    x = synth.uniform_pm1_torch(3, n, dev)
    a = torch.empty_like(x)
    b = torch.empty_like(x)
    ap.ap_cluster_exchange(x, a, n, 4, 8192)
    ap.ap_cluster_exchange_ex(x, b, n, 4, 8192, 1)
    assert ap.ap_check() == ap.AP_OK
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("cs,shift", [(16, 1), (3, 2), (6, -1)])
def test_exchange_ex_full_size(ap, orc, cs, shift):
    """2**28 floats in 32 KiB chunks (32768 chunks: a short last group for
    cs 3 and 6)."""
    import torch

    dev = device()
    n = 1 << 28
    x = synth.uniform_pm1_torch(synth.SEED_EXCHANGE, n, dev)
    y = torch.full_like(x, float("nan"))
    ap.ap_cluster_exchange_ex(x, y, n, cs, 32768, shift)
    assert ap.ap_check() == ap.AP_OK
    assert_bits(to_np(y), orc.cluster_exchange_ex(to_np(x), cs, 32768, shift), f"full exchange_ex cs={cs}")

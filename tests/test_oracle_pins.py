"""The CPU oracle against its pins (no GPU)."""

import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_round_f32_against_numpy():
    """The exact-rounding helper used by the polynomial pins agrees with numpy's
    float64 -> float32 conversion wherever a float64 holds the value exactly."""
    import numpy as np

    from fractions import Fraction

    import synth

    x = synth.uniform_pm1_np(8, 2000).astype(np.float64)
    y = synth.uniform_pm1_np(9, 2000).astype(np.float64)
    for a, b in zip(x.tolist(), y.tolist()):
        v = a * b * 1.0000001 + b  # any float64
        assert oracle_pins.round_f32(Fraction(v)) == float(np.float32(v))
    # ties go to even
    one = Fraction(1)
    half_ulp = Fraction(1, 2**24)
    assert oracle_pins.round_f32(one + half_ulp) == 1.0
    assert oracle_pins.round_f32(one + 3 * half_ulp) == float(np.float32(1 + 2**-22))
    # subnormal spacing
    assert oracle_pins.round_f32(Fraction(3, 2**150)) == float(np.float32(2**-148))


def test_threaded_oracle_poly_is_the_oracle(orc):
    """The full-size parity test's threaded split of the oracle's Horner loop
    gives the single-threaded oracle's bits (ranges of every remainder)."""
    import numpy as np

    import synth
    from gpu_util import oracle_poly_threads

    x = synth.uniform_pm1_np(synth.SEED_POLY, 100003)
    for degree in (0, 1, 8, 33):
        c = synth.coeffs_np(degree)
        want = orc.poly(x, c)
        for threads in (1, 3, 7, 16):
            got = oracle_poly_threads(orc, x, c, threads)
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (degree, threads)

"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

None of these checks calls the oracle twice to agree with itself or retypes
its loop. Each compares it with a worked example from the pages, a library
routine that computes the same thing a different way (numpy/torch roll,
IEEE-exact float64 products, ldexp), exact rational arithmetic, closed forms
or invariants.

Every ``pin_*`` function takes an :class:`oracle.Oracle` and raises
``AssertionError`` on a mismatch, so the same checks can be run against
deliberately broken copies of the oracle (``test_oracle_mutants.py``). Run as
a script, ``python tests/oracle_pins.py LIB.so`` runs every pin against that
library and exits 1 if any fails.
"""

from __future__ import annotations

import os
import sys
from fractions import Fraction

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

GOLDEN = os.path.join(HERE, "golden")


def bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_bits_equal(got, want, what: str):
    g, w = bits(got), bits(want)
    assert g.shape == w.shape, f"{what}: shape {g.shape} != {w.shape}"
    bad = np.nonzero(g != w)[0] if g.ndim == 1 else np.argwhere(g != w)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:4].tolist()}"


# ---------------------------------------------------------------- exact fp32 rounding

_F32_MAX = Fraction((2**24 - 1) * 2**104)


def round_f32(q: Fraction) -> float:
    """Round a rational to the nearest binary32 value, ties to even (IEEE 754)."""
    if q == 0:
        return 0.0
    neg = q < 0
    a = -q if neg else q
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)  # below 2**-126 the spacing stays 2**-149 (subnormals)
    quantum = Fraction(2) ** (e - 23)
    m = a / quantum
    whole = m.numerator // m.denominator
    rest = m - whole
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and whole % 2 == 1):
        whole += 1
    v = whole * quantum
    if v > _F32_MAX:
        r = float("inf")
    else:
        r = float(v)
    return -r if neg else r


def exact_fma_f32(a: float, b: float, c: float) -> float:
    """fma(a, b, c) in binary32: the exact a*b + c, rounded once."""
    return round_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def horner_exact_steps(x: float, coeffs) -> float:
    p = float(coeffs[-1])
    for k in range(len(coeffs) - 2, -1, -1):
        p = exact_fma_f32(p, x, float(coeffs[k]))
    return p


# ---------------------------------------------------------------- row shift pins


def _load_roll_golden():
    rows = {}
    with open(os.path.join(GOLDEN, "roll_64x4_arange.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            v = [int(t) for t in line.split()]
            rows[v[0]] = v[1:]
    return rows


def pin_roll_worked_example(orc):
    """The 64 x 4 arange example and the page's own torch.roll check."""
    import torch

    A = synth.arange_matrix_np(64, 4)
    B = orc.row_roll(A, 1)
    want = torch.roll(torch.arange(256, dtype=torch.float32).reshape(64, 4), shifts=-1, dims=0).numpy()
    assert_bits_equal(B, want, "64x4 arange vs torch.roll(-1, dims=0)")
    for i, vals in _load_roll_golden().items():
        assert B[i].tolist() == [float(v) for v in vals], f"golden row {i}: {B[i].tolist()} != {vals}"
    # Same example with seeded uniform data.
    U = synth.uniform_pm1_np(synth.SEED_ROLL_SMALL, 256).reshape(64, 4)
    assert_bits_equal(orc.row_roll(U, 1), np.roll(U, -1, axis=0), "64x4 uniform vs np.roll")


def pin_roll_brute_force(orc):
    """Small matrices, every shift in [-10, 10], against numpy's roll."""
    seed = 11
    for R in range(1, 10):
        for C in range(1, 6):
            A = synth.uniform_pm1_np(seed, R * C).reshape(R, C)
            seed += 1
            for s in range(-10, 11):
                want = np.roll(A, -s, axis=0)
                assert_bits_equal(orc.row_roll(A, s), want, f"roll R={R} C={C} shift={s}")


def pin_roll_invariants(orc):
    A = synth.uniform_pm1_np(99, 37 * 5).reshape(37, 5)
    # identity shifts
    for s in (0, 37, -37, 74):
        assert_bits_equal(orc.row_roll(A, s), A, f"identity shift {s}")
    # a permutation of the rows: sorted multiset preserved
    B = orc.row_roll(A, 13)
    assert np.array_equal(np.sort(B, axis=None), np.sort(A, axis=None)), "roll is not a permutation"
    assert sorted(map(tuple, B.tolist())) == sorted(map(tuple, A.tolist())), "rows not preserved"
    # composition: roll by a then by b equals roll by a + b
    for a, b in ((3, 5), (-7, 2), (36, 36), (100, -1)):
        assert_bits_equal(orc.row_roll(orc.row_roll(A, a), b), orc.row_roll(A, a + b), f"compose {a}+{b}")
    # one row: always the identity
    one = synth.uniform_pm1_np(5, 7).reshape(1, 7)
    assert_bits_equal(orc.row_roll(one, 12345), one, "R=1")


# ---------------------------------------------------------------- scale pins


def pin_scale_doubling(orc):
    """alpha = 2 (the pages' kernels) is exact doubling: ldexp(x, 1), signs kept."""
    x = synth.uniform_pm1_np(synth.SEED_SCALE, 1 << 14)
    assert_bits_equal(orc.scale(x, 2.0), np.ldexp(x, 1).astype(np.float32), "2x vs ldexp")
    sp = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3.0e38, 1.17549435e-38], dtype=np.float32)
    got = orc.scale(sp, 2.0)
    want = np.array([0.0, -0.0, np.inf, -np.inf, 2.8e-45, -2.8e-45, np.inf, 2.3509887e-38], dtype=np.float32)
    assert_bits_equal(got, want, "2x special values")
    nan = orc.scale(np.array([np.nan], dtype=np.float32), 2.0)
    assert np.isnan(nan[0])


def pin_scale_general(orc):
    """Any alpha: one correctly rounded product, computed here as the exact
    float64 product of two floats rounded once to float32."""
    x = synth.uniform_pm1_np(1234, 1 << 13)
    for alpha in (1.0, -1.0, 0.5, 3.0, 0.1, -7.25, 1.0 / 3.0, 1e-30, 6.02e23):
        a = np.float32(alpha)
        want = (np.float64(a) * x.astype(np.float64)).astype(np.float32)
        assert_bits_equal(orc.scale(x, float(a)), want, f"alpha={alpha}")
    assert_bits_equal(orc.scale(x, 1.0), x, "alpha=1 identity")
    z = orc.scale(np.array([-0.0, 0.0], dtype=np.float32), 3.0)
    assert bits(z).tolist() == bits(np.array([-0.0, 0.0], dtype=np.float32)).tolist(), "signed zeros"


# ---------------------------------------------------------------- polynomial pins


def pin_poly_exact_fma(orc):
    """Horner steps against exact rational fma rounded once per step."""
    rng_x = synth.uniform_pm1_np(4321, 600)
    for K in (1, 2, 3, 8):
        c = synth.coeffs_np(K)
        got = orc.poly(rng_x, c)
        for i, xv in enumerate(rng_x.tolist()):
            want = horner_exact_steps(xv, c.tolist())
            g = float(got[i])
            assert g == want, f"K={K} x={xv!r}: {g!r} != {want!r}"


def pin_poly_closed_forms(orc):
    x = synth.uniform_pm1_np(77, 1000)
    c0 = np.array([0.3125], dtype=np.float32)
    assert np.all(orc.poly(x, c0) == np.float32(0.3125)), "degree 0 is the constant c0"
    for K in (0, 1, 8, 32, 128):
        c = synth.coeffs_np(K)
        zero = orc.poly(np.zeros(4, dtype=np.float32), c)
        assert np.all(zero == c[0]), f"K={K}: p(0) != c0"
    # degree 1 is one fma: c1*x + c0 rounded once
    c = synth.coeffs_np(1)
    got = orc.poly(x, c)
    for i, xv in enumerate(x[:200].tolist()):
        assert float(got[i]) == exact_fma_f32(float(c[1]), xv, float(c[0])), f"K=1 at {i}"
    # integer coefficients at x = +-1 are exact sums: sum c_k and sum (-1)^k c_k
    ci = np.array([3, -1, 4, 1, -5, 9, 2, -6], dtype=np.float32)
    pm = orc.poly(np.array([1.0, -1.0], dtype=np.float32), ci)
    assert pm[0] == ci.sum(), "p(1) != sum c"
    assert pm[1] == sum(((-1) ** k) * float(v) for k, v in enumerate(ci)), "p(-1) alternating sum"


def pin_poly_error_bound(orc):
    """|Horner(x) - p(x)| <= gamma_2K * sum |c_k||x|^k (Higham, Accuracy and
    Stability of Numerical Algorithms, section 5.1), with p(x) exact."""
    u = Fraction(1, 2**24)
    x = synth.uniform_pm1_np(555, 60)
    for K in (8, 32, 128):
        c = [Fraction(float(v)) for v in synth.coeffs_np(K)]
        got = orc.poly(x, synth.coeffs_np(K))
        m = 2 * K
        gamma = m * u / (1 - m * u)
        for i, xv in enumerate(x.tolist()):
            X = Fraction(xv)
            exact = Fraction(0)
            mag = Fraction(0)
            for k in range(K, -1, -1):
                exact = exact * X + c[k]
                mag = mag * abs(X) + abs(c[k])
            assert abs(Fraction(float(got[i])) - exact) <= gamma * mag, f"K={K} x={xv}: bound violated"


# ---------------------------------------------------------------- exchange pins


def _load_exchange_golden():
    cases = []
    with open(os.path.join(GOLDEN, "exchange_small.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, tail = line.split(":")
            n, cs, cb = (int(t) for t in head.split())
            cases.append((n, cs, cb, [float(t) for t in tail.split()]))
    return cases


def pin_exchange_worked_examples(orc):
    for n, cs, cb, want in _load_exchange_golden():
        got = orc.cluster_exchange(np.arange(n, dtype=np.float32), cs, cb)
        assert got.tolist() == want, f"n={n} cs={cs} chunk={cb}: {got.tolist()} != {want}"


def pin_exchange_library(orc):
    """Against numpy: view as (groups, cs, E) and roll the rank axis by -1."""
    for cs in (1, 2, 3, 4, 8):
        for E in (1, 2, 5, 8):
            for groups in (1, 2, 7):
                n = groups * cs * E
                x = synth.uniform_pm1_np(1000 + n, n)
                want = np.roll(x.reshape(groups, cs, E), -1, axis=1).reshape(-1)
                assert_bits_equal(orc.cluster_exchange(x, cs, 4 * E), want, f"cs={cs} E={E} g={groups}")


def pin_exchange_invariants(orc):
    x = synth.uniform_pm1_np(31337, 3 * 8 * 16)
    assert_bits_equal(orc.cluster_exchange(x, 1, 64), x, "cs=1 identity")
    for cs in (2, 4, 8):
        y = x
        for _ in range(cs):
            y = orc.cluster_exchange(y, cs, 64)
        assert_bits_equal(y, x, f"cs={cs} applied cs times")
        once = orc.cluster_exchange(x, cs, 64).reshape(-1, 16)
        assert sorted(map(tuple, once.tolist())) == sorted(map(tuple, x.reshape(-1, 16).tolist())), "not a chunk permutation"
    for bad in ((x[:100], 4, 64), (x, 5, 64), (x, 2, 6)):
        try:
            orc.cluster_exchange(*bad)
        except ValueError:
            continue
        raise AssertionError(f"partial cluster or chunk accepted: n={bad[0].size} cs={bad[1]} chunk={bad[2]}")


def _load_exchange_ex_golden():
    cases = []
    with open(os.path.join(GOLDEN, "exchange_ex_small.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, tail = line.split(":")
            n, cs, cb, sh = (int(t) for t in head.split())
            cases.append((n, cs, cb, sh, [float(t) for t in tail.split()]))
    return cases


def pin_exchange_ex_worked_examples(orc):
    for n, cs, cb, sh, want in _load_exchange_ex_golden():
        got = orc.cluster_exchange_ex(np.arange(n, dtype=np.float32), cs, cb, sh)
        assert got.tolist() == want, f"n={n} cs={cs} chunk={cb} shift={sh}: {got.tolist()} != {want}"


def pin_exchange_ex_library(orc):
    """Against numpy: whole groups as a (groups, cs, E) view rolled by -shift on
    the rank axis, the short last group as an (m, E) view rolled alike."""
    for cs in (1, 2, 3, 4, 5, 8, 16):
        for E in (1, 3):
            for chunks in (cs, 3 * cs, 3 * cs + 1, 2 * cs + cs // 2 + 1):
                n = chunks * E
                x = synth.uniform_pm1_np(7000 + n + cs, n)
                G, m = divmod(chunks, cs)
                for shift in (0, 1, 2, -1, cs - 1, 7, -13):
                    full = np.roll(x[: G * cs * E].reshape(G, cs, E), -shift, axis=1).reshape(-1)
                    tail = np.roll(x[G * cs * E:].reshape(m, E), -shift, axis=0).reshape(-1) if m else x[:0]
                    want = np.concatenate([full, tail])
                    got = orc.cluster_exchange_ex(x, cs, 4 * E, shift)
                    assert_bits_equal(got, want, f"cs={cs} E={E} chunks={chunks} shift={shift}")


def pin_exchange_ex_invariants(orc):
    x = synth.uniform_pm1_np(4242, 38 * 4)  # 38 chunks of 4 floats: a short last group for cs 3, 4, 6
    for cs in (2, 3, 4, 6):
        assert_bits_equal(orc.cluster_exchange_ex(x, cs, 16, 0), x, f"cs={cs} shift 0 is the identity")
        for a, b in ((1, 2), (3, -1), (5, 5)):
            once = orc.cluster_exchange_ex(orc.cluster_exchange_ex(x, cs, 16, a), cs, 16, b)
            assert_bits_equal(once, orc.cluster_exchange_ex(x, cs, 16, a + b), f"cs={cs} compose {a}+{b}")
        y = orc.cluster_exchange_ex(x, cs, 16, 1)
        assert sorted(map(tuple, y.reshape(-1, 4).tolist())) == sorted(map(tuple, x.reshape(-1, 4).tolist()))
    try:
        orc.cluster_exchange_ex(x[:-1], 4, 16, 1)
    except ValueError:
        pass
    else:
        raise AssertionError("a partial chunk was accepted")


def pin_all_to_all_worked_examples(orc):
    with open(os.path.join(GOLDEN, "all_to_all_small.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, tail = line.split(":")
            n, cs, cb = (int(t) for t in head.split())
            want = [float(t) for t in tail.split()]
            got = orc.cluster_all_to_all(np.arange(n, dtype=np.float32), cs, cb)
            assert got.tolist() == want, f"n={n} cs={cs} chunk={cb}: {got.tolist()} != {want}"


def pin_all_to_all_library(orc):
    """Against numpy: each group viewed as a (cs, cs, B) array of sub-blocks,
    the first two axes swapped."""
    for cs in (1, 2, 3, 4, 5, 8, 16):
        for B in (1, 3, 4):
            for groups in (1, 2, 5):
                E = cs * B
                n = groups * cs * E
                x = synth.uniform_pm1_np(9000 + n + cs, n)
                want = x.reshape(groups, cs, cs, B).transpose(0, 2, 1, 3).reshape(-1)
                assert_bits_equal(orc.cluster_all_to_all(x, cs, 4 * E), want, f"cs={cs} B={B} groups={groups}")


def pin_all_to_all_invariants(orc):
    x = synth.uniform_pm1_np(4343, 6 * 4 * 8)  # 6 groups of cs 4 with 8-float chunks, or 3 groups of cs 8
    for cs, E in ((1, 8), (2, 8), (4, 8), (8, 8), (4, 4)):
        once = orc.cluster_all_to_all(x, cs, 4 * E)
        assert_bits_equal(orc.cluster_all_to_all(once, cs, 4 * E), x, f"cs={cs}: a block transpose twice is the identity")
        if cs == 1:
            assert_bits_equal(once, x, "cs 1 is the identity")
        # each output sub-block is some input sub-block of the same group
        B = E // cs
        blocks = lambda a: sorted(map(tuple, a.reshape(-1, B).tolist()))
        assert blocks(once) == blocks(x), f"cs={cs}: not a permutation of sub-blocks"
        # with B == E / cs and cs == E (one float per sub-block) it is the matrix transpose
        if B == 1:
            assert_bits_equal(once, x.reshape(-1, cs, cs).transpose(0, 2, 1).reshape(-1), f"cs={cs} matrix transpose")
    for bad in ((x, 3, 32), (x[:-8], 4, 32), (x, 4, 6)):
        try:
            orc.cluster_all_to_all(*bad)
        except ValueError:
            continue
        raise AssertionError(f"partial sub-block or group accepted: n={bad[0].size} cs={bad[1]} chunk={bad[2]}")


def pin_masked_copy_worked_example(orc):
    with open(os.path.join(GOLDEN, "masked_copy_small.txt")) as f:
        lines = [l.strip() for l in f if l.strip() and not l.startswith("#")]
    codes = [int(t) for t in lines[0].split(":")[1].split()]
    want = [float(t) for t in lines[1].split(":")[1].split()]
    x = np.arange(1, 25, dtype=np.float32)
    got = orc.masked_copy(x, np.full(24, -1.0, dtype=np.float32), codes)
    assert got.tolist() == want, f"{got.tolist()} != {want}"


def pin_masked_copy_bytes(orc):
    """Against a byte-level numpy restatement: prefix bytes from the input,
    zeros after, untouched chunks where the predicate is off."""
    rng = np.random.default_rng(17)
    for n_chunks in (1, 7, 300):
        x = synth.uniform_pm1_np(n_chunks, 4 * n_chunks)
        before = synth.uniform_pm1_np(n_chunks + 1, 4 * n_chunks)
        codes = rng.integers(-2, 17, n_chunks).astype(np.int8)
        xb = x.view(np.uint8).reshape(n_chunks, 16)
        want = before.copy().view(np.uint8).reshape(n_chunks, 16)
        cols = np.arange(16)[None, :]
        keep = np.where(codes < 0, 0, codes)[:, None]
        filled = np.where(cols < keep, xb, 0).astype(np.uint8)
        on = (codes != -1)[:, None]
        want = np.where(on, filled, want).astype(np.uint8).reshape(-1).view(np.float32)
        assert_bits_equal(orc.masked_copy(x, before, codes), want, f"masked copy n={n_chunks}")


def pin_masked_copy_special_codes(orc):
    x = synth.uniform_pm1_np(3, 64)
    before = synth.uniform_pm1_np(4, 64)
    assert_bits_equal(orc.masked_copy(x, before, np.full(16, 16, np.int8)), x, "all 16: plain copy")
    assert_bits_equal(orc.masked_copy(x, before, np.full(16, -1, np.int8)), before, "all -1: unchanged")
    zeros = np.zeros(64, dtype=np.float32)
    assert_bits_equal(orc.masked_copy(x, before, np.full(16, 0, np.int8)), zeros, "all 0: zeros")
    assert_bits_equal(orc.masked_copy(x, before, np.full(16, -2, np.int8)), zeros, "all -2: zeros")
    try:
        orc.masked_copy(x, before, np.full(16, 17, np.int8))
    except ValueError:
        pass
    else:
        raise AssertionError("code 17 accepted")


ALL_PINS = [
    pin_roll_worked_example,
    pin_roll_brute_force,
    pin_roll_invariants,
    pin_scale_doubling,
    pin_scale_general,
    pin_poly_exact_fma,
    pin_poly_closed_forms,
    pin_poly_error_bound,
    pin_exchange_worked_examples,
    pin_exchange_library,
    pin_exchange_invariants,
    pin_exchange_ex_worked_examples,
    pin_exchange_ex_library,
    pin_exchange_ex_invariants,
    pin_all_to_all_worked_examples,
    pin_all_to_all_library,
    pin_all_to_all_invariants,
    pin_masked_copy_worked_example,
    pin_masked_copy_bytes,
    pin_masked_copy_special_codes,
]


def run_all(orc) -> list[str]:
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError as e:
            failed.append(f"{pin.__name__}: {e}")
    return failed


if __name__ == "__main__":
    import oracle

    lib = sys.argv[1] if len(sys.argv) > 1 else None
    failures = run_all(oracle.Oracle(lib))
    for f in failures:
        print("FAIL", f)
    sys.exit(1 if failures else 0)

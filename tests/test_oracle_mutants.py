"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of ``oracle/oracle.cpp`` (a dropped
term, a wrong sign or index, a wrong operation), compiles the copy on the CPU
and runs every pin against it in a child process. The pins must report a
failure (exit status 1; a crash does not count as catching it).
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = {
    "scale_adds_zero": ("out[i] = alpha * in[i];", "out[i] = alpha * in[i] + 0.0f;"),
    "scale_doubles": ("out[i] = alpha * in[i];", "out[i] = in[i] + in[i];"),
    "scale_via_double_sum": ("out[i] = alpha * in[i];", "out[i] = (float)((double)in[i] * (double)alpha + 1e-300);"),
    "roll_wrong_direction": ("(i + s) % rows", "(i + rows - s) % rows"),
    "roll_ignores_shift": ("(i + s) % rows", "(i + 1) % rows"),
    "roll_column_reversed": ("A[src_row * cols + j]", "A[src_row * cols + (cols - 1 - j)]"),
    "roll_shift_not_reduced_sign": ("((shift % rows) + rows) % rows", "((-shift % rows) + rows) % rows"),
    "poly_no_fma": ("p = std::fma(p, x, coeffs[k]);", "p = p * x + coeffs[k];"),
    "poly_drops_c0": ("k >= 0; --k", "k >= 1; --k"),
    "poly_reversed_order": ("float p = coeffs[degree];", "float p = coeffs[0];"),
    "poly_wrong_sign": ("p = std::fma(p, x, coeffs[k]);", "p = std::fma(p, -x, coeffs[k]);"),
    "exchange_wrong_direction": ("(r + 1) % cs", "(r + cs - 1) % cs"),
    "exchange_drops_group": ("group * cs + (r + 1) % cs", "(r + 1) % cs"),
    "exchange_accepts_partial": ("if (n % (E * cs) != 0) return -1;", ""),
    "exchange_ex_last_group_uses_cs": ("const int64_t m = left < cs ? left : cs;", "const int64_t m = cs;"),
    "exchange_ex_shift_sign": ("const int64_t s = ((shift % m) + m) % m;", "const int64_t s = ((-shift % m) + m) % m;"),
    "masked_skip_writes": ("if (c == -1) continue;", "if (c == -1) { }"),
    "masked_no_zero_fill": ("dst[16 * k + b] = b < keep ? src[16 * k + b] : 0;", "if (b < keep) dst[16 * k + b] = src[16 * k + b];"),
    "masked_ignore_copies": ("const int keep = c < 0 ? 0 : c;", "const int keep = c < 0 ? 16 : c;"),
    "exchange_ex_ignores_shift": ("const int64_t src = first + (r + s) % m;", "const int64_t src = first + (r + 1) % m;"),
    "a2a_no_transpose": ("const float* src = in + (g * cs + r) * E + d * B;",
                         "const float* src = in + (g * cs + d) * E + r * B;"),
    "a2a_wrong_sub_block": ("float* dst = out + (g * cs + d) * E + r * B;", "float* dst = out + (g * cs + d) * E + d * B;"),
    "a2a_drops_group": ("const float* src = in + (g * cs + r) * E + d * B;", "const float* src = in + r * E + d * B;"),
    "a2a_accepts_partial_block": ("if (E % cs != 0 || n % (E * cs) != 0) return -1;", "if (n % (E * cs) != 0) return -1;"),
}


def _compile(src_text: str, tmp_path, name: str) -> str:
    sys.path.insert(0, ROOT)
    from oracle import build as obuild

    src = tmp_path / f"{name}.cpp"
    src.write_text(src_text)
    lib = tmp_path / f"lib{name}.so"
    obuild.build(str(src), str(lib), force=True)
    return str(lib)


def _run_pins(lib: str) -> subprocess.CompletedProcess:
    return subprocess.run(
        [sys.executable, os.path.join(ROOT, "tests", "oracle_pins.py"), lib],
        capture_output=True,
        text=True,
        timeout=600,
        cwd=ROOT,
    )


def test_unmutated_copy_passes(tmp_path):
    with open(SRC) as f:
        text = f.read()
    r = _run_pins(_compile(text, tmp_path, "clean"))
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation site for {name} not unique/found"
    r = _run_pins(_compile(text.replace(old, new), tmp_path, name))
    assert r.returncode == 1, f"{name} not caught (exit {r.returncode}):\n{r.stdout}{r.stderr}"
    assert "FAIL" in r.stdout

"""Host logic of bench.py's clock sampler, against a fake nvidia-smi.

The sampler must not hand control back until nvidia-smi has written real
samples: its start-up can hold the driver, and a timed region that overlaps
it measures idle time. No GPU is used; the fake writes CSV lines to the file
named after -f.
"""

import os
import stat
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

FAKE_SLOW_START = """#!/bin/sh
# fake nvidia-smi: 0.6 s of start-up, then one sample line every 0.05 s
out=""
while [ $# -gt 0 ]; do
  if [ "$1" = "-f" ]; then out="$2"; shift; fi
  shift
done
sleep 0.6
i=0
while [ $i -lt 200 ]; do
  echo "2026/01/01 00:00:00.000, 0, 2070, 2070, 500.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active" >> "$out"
  i=$((i + 1))
  sleep 0.05
done
"""

FAKE_EXITS = """#!/bin/sh
exit 3
"""


def _install(tmp_path, body):
    p = tmp_path / "nvidia-smi"
    p.write_text(body)
    p.chmod(p.stat().st_mode | stat.S_IXUSR | stat.S_IXGRP | stat.S_IXOTH)
    return str(tmp_path)


@pytest.mark.timeout(60)
def test_sampler_waits_for_first_samples(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", _install(tmp_path, FAKE_SLOW_START) + os.pathsep + os.environ["PATH"])
    t0 = time.monotonic()
    with bench.ClockSampler(0) as clk:
        waited = time.monotonic() - t0
        with open(clk.path) as fh:
            lines = [line for line in fh if line.strip()]
        assert len(lines) >= 2, "returned before nvidia-smi wrote two samples"
        assert 0.6 <= waited < 5.0


@pytest.mark.timeout(60)
def test_sampler_returns_when_nvidia_smi_exits(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", _install(tmp_path, FAKE_EXITS) + os.pathsep + os.environ["PATH"])
    t0 = time.monotonic()
    with bench.ClockSampler(0):
        assert time.monotonic() - t0 < 5.0

"""The benchmark's multi-rank path on CPU (gloo, world size 2): barrier and
max-over-ranks timing, and one JSON line from rank 0 only."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist()
    d.barrier()
    q.put((rank, d.max(values[rank])))
    d.close()


def test_dist_max_over_ranks_gloo():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("CPU-only check of the gloo path")
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [3.25, 7.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 7.5, 1: 7.5}


def test_reference_arm_under_torchrun_two_ranks():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("CPU-only check of the gloo path")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_results_log_appends_with_provenance(tmp_path, monkeypatch, capsys):
    """Every printed bench line is also appended to results/<kind>.jsonl with
    the GPU name, git commit, a hash of the CUDA sources, time and argv."""
    import json
    import sys

    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setattr(bench, "RESULTS_DIR", str(tmp_path))
    bench.emit({"metric": "m", "value": 1.5}, "sweep")
    bench.emit({"metric": "m", "value": 2.5}, "sweep")
    printed = [json.loads(l) for l in capsys.readouterr().out.splitlines()]
    assert printed == [{"metric": "m", "value": 1.5}, {"metric": "m", "value": 2.5}]
    rows = [json.loads(l) for l in (tmp_path / "sweep.jsonl").read_text().splitlines()]
    assert [r["value"] for r in rows] == [1.5, 2.5]
    prov = rows[0]["provenance"]
    assert set(prov) >= {"gpu", "git_sha", "source_hash", "argv", "time"}
    assert len(prov["source_hash"]) == 16

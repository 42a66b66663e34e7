"""bench.py --gpus N without a torchrun environment starts N replicas itself
(one process per local GPU, torchrun's environment variables, 127.0.0.1
rendezvous).  The launcher runs here with gloo stand-in ranks on the CPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_spawn_replicas_runs_n_ranks_and_one_line():
    code = ("import sys, bench; sys.exit(bench.spawn_replicas(2, ['--steps', '3'], "
            f"script={os.path.join(ROOT, 'tests', 'replica_worker.py')!r}))")
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                       # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["local_ranks_seen"] == 2
    assert d["ms_per_step"] == 15.0              # the slower rank sets the step time
    assert abs(d["value"] - 2 * 1e12 / 15e-3 / 1e12) < 1e-9
    assert d["argv"] == ["--steps", "3"] and d["master"] == "127.0.0.1"


def test_gpus_flag_without_torchrun_dispatches_to_the_launcher(monkeypatch):
    seen = {}
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench, "spawn_replicas", lambda n, argv: seen.update(n=n, argv=argv) or 0)
    assert bench.main(["--gpus", "4", "--steps", "2"]) == 0
    assert seen == {"n": 4, "argv": ["--gpus", "4", "--steps", "2"]}


def test_a_rank_under_torchrun_does_not_spawn(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(bench, "spawn_replicas", lambda *a: (_ for _ in ()).throw(AssertionError))
    monkeypatch.setattr(bench, "run_reference", lambda args: None)
    assert bench.main(["--gpus", "2", "--impl", "reference"]) == 0


def test_a_failing_rank_stops_the_others(tmp_path):
    """Rank 1 exits with an error before the collective; rank 0 would wait in
    it forever, so the launcher stops it and returns the failure."""
    worker = tmp_path / "fail_worker.py"
    worker.write_text(
        "import os, sys, time\n"
        "if os.environ['RANK'] == '1':\n"
        "    sys.exit(3)\n"
        "time.sleep(600)\n")
    code = ("import sys, bench; sys.exit(bench.spawn_replicas(2, [], "
            f"script={str(worker)!r}))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 3


def test_link_floor_takes_the_binding_term():
    """The end-to-end floor is the slowest of: inputs at the host->device
    rate, outputs at the device->host rate, everything at the combined
    rate."""
    import bench
    rates = {"h2d": 200.0, "d2h": 100.0, "both": 250.0}
    gb = 1e9
    assert abs(bench.link_floor_ms(2 * gb, 1 * gb, rates) - 12.0) < 1e-9      # combined: 3 / 250
    assert abs(bench.link_floor_ms(0.5 * gb, 2 * gb, rates) - 20.0) < 1e-9    # out: 2 / 100
    assert abs(bench.link_floor_ms(4 * gb, 0.1 * gb, rates) - 20.0) < 1e-9    # in: 4 / 200

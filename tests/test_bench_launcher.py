"""bench.py's rank launcher on CPU (gloo, world size 2): ``--gpus 2`` without a launcher's
WORLD_SIZE starts two ranks itself; both join one process group, the reported step time is
the slowest rank's, and rank 0 alone prints the line with n_gpus = 2.  ``--dry-run`` replaces
the GPU work with a sleep so the launcher and the max-over-ranks reduction run here."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_launcher_runs_two_ranks_and_reports_the_slowest():
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "5",
                        "--warmup", "0", "--dry-run"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout           # rank 0 only
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["dry_run"] is True
    assert line["ranks"] == [0, 1]
    # rank 1 sleeps 20 ms a step: the line carries the maximum over the ranks
    assert line["ms_per_step"] >= 19.0, line
    assert line["value"] > 0


def test_launcher_reports_a_failing_rank():
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    # zero steps: rank 0 divides by a zero time after the collectives and exits non-zero; the
    # launcher (which parsed the arguments itself first) must pass that status on
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "0",
                        "--dry-run"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ZeroDivisionError" in r.stderr

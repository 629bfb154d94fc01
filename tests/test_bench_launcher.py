"""bench.py's rank launcher on CPU: ``--gpus N`` without torchrun starts N rank processes
(gloo in the dry run), every rank joins the group, rank 0 alone prints one line with
n_gpus == N, and a rank count that disagrees with --gpus is refused."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None):
    e = dict(os.environ)
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "LOCAL_WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT"):
        e.pop(k, None)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=e, cwd=ROOT,
                          capture_output=True, text=True, timeout=300)


@pytest.mark.parametrize("n", [2, 3])
@pytest.mark.parametrize("impl", ["ours", "reference"])
def test_gpus_n_starts_n_ranks(n, impl):
    r = _run(["--gpus", str(n), "--dry-run", "--impl", impl])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout          # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["n_gpus"] == n and line["ranks_started"] == n
    assert line["impl"] == impl


def test_rank_count_must_match_gpus():
    r = _run(["--gpus", "2", "--dry-run"], env={"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode == 2
    assert "--gpus 2" in r.stderr

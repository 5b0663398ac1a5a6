"""bench.py --gpus N starts its own N ranks when no launcher did (CPU: the reference arm,
which touches no GPU, over two ranks), and refuses a launcher whose rank count disagrees."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _env_without_launcher():
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT", "LOCAL_WORLD_SIZE"):
        env.pop(k, None)
    return env


def test_gpus_2_runs_two_ranks_and_prints_one_line():
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1", "--cpu-sample-rows", "4"], capture_output=True, text=True,
                       cwd=ROOT, env=_env_without_launcher(), timeout=900)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2  # the printing rank saw a world of two ranks
    assert d["impl"] == "reference" and d["value"] > 0


def test_launcher_rank_count_must_match_gpus():
    env = dict(_env_without_launcher(), RANK="0", WORLD_SIZE="3", LOCAL_RANK="0")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, cwd=ROOT, env=env,
                       timeout=300)
    assert p.returncode != 0 and "--gpus 2" in p.stderr

"""bench.py's launcher and record on CPU: `--gpus N` runs N ranks (torchrun,
one process per GPU), a WORLD_SIZE that disagrees with --gpus is an error,
and the reference arm's line carries the GPU arm's config keys, the host CPU
model and an explicit label on its extrapolated step time."""
import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None, timeout=300):
    e = dict(os.environ)
    e.pop("WORLD_SIZE", None)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=timeout, env=e, cwd=ROOT)


@pytest.fixture(scope="module", autouse=True)
def built_oracle():
    import oracle
    oracle.build()


def test_launch_command_is_torchrun_with_n_ranks():
    cmd = bench.launch_command(4, ["--steps", "2"])
    assert cmd[:3] == [sys.executable, "-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--nnodes=1" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-3:] == [os.path.join(ROOT, "bench.py"), "--steps", "2"]


def test_gpus_two_runs_two_ranks_and_rank0_prints_one_line():
    r = _run(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "tiny-mha",
              "--cpu-seconds", "0.5"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["impl"] == "reference"
    # the same config keys as the GPU arm's line for this workload
    assert d["config"] == bench.workload_config("tiny-mha", 2)
    assert "extrapolated" in d["ms_per_step_source"]
    cb = d["cpu_baseline"]
    assert cb["cpu_model"] and cb["kind"] == "oracle"
    assert cb["cores"] == bench.host_threads()          # not torchrun's OMP_NUM_THREADS=1


def test_world_size_must_match_gpus():
    r = _run(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"], env={"WORLD_SIZE": "1"})
    assert r.returncode == 2
    assert "WORLD_SIZE=1" in r.stderr


def test_timed_repeats_reach_the_target():
    assert bench.timed_repeats(3.6) * 3.6 >= bench.TIMED_TARGET_MS
    assert bench.timed_repeats(1000.0) == 1
    assert 1 <= bench.timed_repeats(0.0) <= 200

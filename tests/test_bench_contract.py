"""bench.py's reference arm on the CPU: one JSON line with the contract's
keys, and ranks other than 0 exit without output."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
        "e2e"}


def _run(extra_env=None, extra_args=()):
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "2", "--warmup", "1", *extra_args], capture_output=True,
                          text=True, timeout=600, cwd=ROOT, env=env)


def test_reference_arm_json_line():
    r = _run()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert KEYS <= set(j)
    assert j["impl"] == "reference" and j["steps"] == 2 and j["warmup"] >= 3
    assert j["warmup_requested"] == 1
    assert j["unit"] == "GB/s" and j["value"] > 0 and j["higher_is_better"] is True
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert j["config"]["workload"] == "instancenorm2d_fp32_112x64x512x512"


def test_reference_arm_other_ranks_silent():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, ["--gpus", "2"])
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def _plan(gpus, extra_env=None):
    r = _run(extra_env, ["--gpus", str(gpus), "--dry-run"])
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    return r.returncode, json.loads(lines[-1])


def test_gpus_without_launcher_spawns_one_process_per_gpu():
    """--gpus 2 without torchrun re-launches under torch.distributed.run with
    two processes on 127.0.0.1; --gpus 1 runs in place."""
    rc, plan = _plan(2)
    assert rc == 0 and plan["action"] == "relaunch" and plan["world_size"] == 2
    cmd = plan["cmd"]
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=2" in cmd and "127.0.0.1" in cmd
    i = cmd.index(os.path.join(ROOT, "bench.py"))
    assert cmd[i + 1:] == ["--impl", "reference", "--steps", "2", "--warmup", "1", "--gpus", "2",
                           "--dry-run"]
    rc, plan = _plan(1)
    assert rc == 0 and plan == {"action": "run", "world_size": 1}


def test_gpus_must_match_the_launchers_world_size():
    rc, plan = _plan(2, {"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert rc == 0 and plan == {"action": "run", "world_size": 2}
    rc, plan = _plan(4, {"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert rc == 2 and plan["action"] == "error"
    r = _run({"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"}, ["--gpus", "4"])
    assert r.returncode == 2 and "WORLD_SIZE=2" in r.stderr and r.stdout.strip() == ""


def test_relaunch_runs_the_reference_arm_on_two_ranks():
    """The re-launched run: two CPU processes under torch.distributed.run,
    rank 0 prints one line with n_gpus 2, rank 1 prints nothing."""
    r = _run(None, ["--gpus", "2"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2

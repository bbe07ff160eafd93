"""bench.py's reference arm on CPU: the oracle timed on a bounded sample, printed as one JSON
line with the bench contract's keys; under a multi-rank launch only rank 0 prints; the arm
loads the oracle's library and never the product's."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# runs the arm as `python bench.py --impl reference --steps 1 --warmup 0` would, then reports which
# shared libraries of the repository the process mapped
_PROG = """
import runpy, sys
sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]
runpy.run_path("bench.py", run_name="__main__")
maps = open("/proc/self/maps").read()
print("MAPPED", "libkvsel" in maps, "_liboracle" in maps)
"""


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "-c", _PROG], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=900)


def test_reference_arm_prints_one_contract_line():
    out = _run({})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "KV rows scored/s" and d["unit"] == "rows/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["dtype"] == "f64" and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert cb["host"]["nproc"] >= 1 and cb["host"]["model"] and cb["nproc"] == os.cpu_count()
    assert d["e2e"] == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # measured and scaled parts are declared separately, and the figures follow from them
    tok, blk = cb["token_step"], cb["block_step"]
    assert tok["extrapolated"] is False and tok["work_fraction"] == 1.0 and tok["procs"] == cb["cores"]
    assert blk["extrapolated"] is True and 0 < blk["work_fraction"] < 1 and blk["procs"] == cb["cores"]
    est = tok["measured_s"] + blk["measured_s"] / blk["work_fraction"]
    assert abs(cb["est_full_step_s"] - est) <= 1e-9 * est
    assert abs(d["value"] - (tok["rows"] + blk["rows"]) / est) <= 1e-9 * d["value"]
    # one sample step's wall time is what ms_per_step reports (it fits in the run)
    assert abs(d["ms_per_step"] - 1e3 * d["wall_s"]) <= 1e-6 * d["ms_per_step"]
    assert d["ms_per_step"] >= 1e3 * cb["measured_s"] * 0.99
    # the arm maps the oracle's library, never the product's
    assert "MAPPED False True" in out.stdout


def test_reference_arm_other_ranks_exit_quietly():
    out = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.returncode == 0, out.stderr[-2000:]
    assert not [ln for ln in out.stdout.splitlines() if ln.startswith("{")]

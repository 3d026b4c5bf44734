"""CPU checks of bench.py's output contract on its oracle arm (no GPU needed):
rank 0 prints exactly one JSON line with the keys every bench line carries,
the e2e and cpu_baseline objects agree with the line's own value, and under
torchrun any other rank exits 0 without work or output."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TINY = "tiny_mha_T1024_D64_f32"


def _bench(*argv, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], cwd=ROOT,
                          env=e, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _bench("--impl", "reference", "--workload", TINY, "--steps", "2", "--warmup", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == TINY and "model" not in d["config"]
    cb = d["cpu_baseline"]
    # tokens/s of the work done: the sampled layers' share of the prompt per step
    L, n = (int(t) for t in cb["scale"].split("/"))
    assert L == d["config"]["layers"] and 1 <= n <= L
    want = d["config"]["seq_len"] * n / L / (d["ms_per_step"] / 1e3)
    assert abs(d["value"] - want) <= want * (0.05 / d["ms_per_step"] + 1e-6)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _bench("--impl", "reference", "--workload", TINY, "--steps", "1", "--warmup", "0",
               env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""

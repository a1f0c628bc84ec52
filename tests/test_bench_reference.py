"""The benchmark's reference arm (the CPU oracle, timed as it stands) keeps the JSON contract the
benchmark driver reads: one line with the metric, value, unit, cpu_baseline and e2e, printed by
rank 0 only. No GPU is involved."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, **env):
    e = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        e.pop(k, None)
    e.update(env)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=600, cwd=ROOT, env=e)
    assert r.returncode == 0, r.stderr[-3000:]
    return [ln for ln in r.stdout.splitlines() if ln.strip()]


def test_reference_arm_prints_one_contract_line():
    lines = _run("--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1")
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    sys.path.insert(0, ROOT)
    import bench
    assert d["config"]["workload"] == bench.workload_desc("tiny")  # the GPU arm's string, character for character
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert abs(d["ms_per_step"] - 256 / d["value"] * 1e3) < 1e-6 * d["ms_per_step"]  # tiny: B * N = 256 tokens
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    assert _run("--impl", "reference", "--config", "tiny", "--steps", "2", RANK="1", WORLD_SIZE="2",
                LOCAL_RANK="1") == []


def test_roofline_bounds_arithmetic():
    """The line's two bounds: the scoring's tensor work is QK^T over the M = G (n_r + n_b) observation
    rows, twice (one pass for the log-sum-exp, one for the max), 4 M D FLOP per cached key, none for
    fp32 caches; the governing bound is the larger of the bytes at the copy peak and the FLOP at the
    bf16 peak. Checked against the R1-Qwen-7B shape's numbers worked by hand (G = 7, 32 rows each)."""
    import types
    sys.path.insert(0, ROOT)
    import bench
    inp = types.SimpleNamespace(dtype="bf16", Hq=28, Hkv=4, n_r=16, n_b=16, D=128, heads=28 * 8 * 4, N=8192)
    flop = bench.score_flop(inp)
    assert flop == 4 * 224 * 128 * 896 * 8192 == 841_813_590_016
    assert bench.score_flop(types.SimpleNamespace(**{**vars(inp), "dtype": "f32"})) == 0
    pk = {"hbm_gbs": 6782.8, "bf16_tflops": 1934.3}
    b = bench.bounds(2.81e9, flop, 1.0, pk)
    assert abs(b["hbm_ms"] - 2.81e9 / 6782.8e9 * 1e3) < 1e-12
    assert abs(b["tensor_ms"] - flop / 1934.3e12 * 1e3) < 1e-12
    assert b["governing"] == "tensor" and abs(b["frac"] - b["tensor_ms"]) < 1e-12  # 1 ms step
    b = bench.bounds(96.6e9, 10 * flop, 20.0, pk)  # bytes dominate: the Qwen3-14B-shaped step's order
    assert b["governing"] == "hbm" and abs(b["frac"] - b["hbm_ms"] / 20.0) < 1e-12

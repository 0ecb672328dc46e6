"""The reference arm of bench.py (the fp64 oracle timed on the host cores) on
CPU: the JSON line it prints, and that ranks other than 0 exit without work."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny_f32",
           "--steps", "1", "--warmup", "3", *args]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["unit"] == "Gelem/s" and j["higher_is_better"] is True
    assert j["steps"] == 1 and j["warmup"] == 3 and j["n_gpus"] == 1
    assert j["config"]["workload"] == "tiny_f32" and j["config"]["seqlen"] == 256
    assert j["value"] > 0 and j["cpu_baseline"]["value"] == j["value"]
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_other_ranks_exit_without_work():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_parity_check_on_cpu():
    """The bench's all-element parity check (host logic): the oracle's own
    output passes, one element moved past the tolerance fails."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    from selective_state_space_02_gb300 import synth
    p = synth.make_problem(1, 6, 16, 50, dtype="bf16", gate=True, final_state=True, seed=7)
    full = bench.oracle_full(p)
    y = torch.from_numpy(full[0].reshape(1, 6, 50)).to(torch.bfloat16)
    fs = torch.from_numpy(full[1].reshape(1, 6, 16)).float()
    r = bench.parity_check(p, y, fs, full)
    assert r["ok"] and r["elements"] == 300 and r["y_max_scaled_err"] <= 2 ** -8
    y[0, 3, 17] += 1.0
    r = bench.parity_check(p, y, fs, full)
    assert not r["ok"] and r["y_max_scaled_err"] > 2e-2


def test_cpu_baseline_reports_one_thread_beside_all_cores():
    """The bench line's cpu_baseline: the oracle on all host cores over a
    bounded sample, and on one thread beside it."""
    sys.path.insert(0, ROOT)
    import bench
    from selective_state_space_02_gb300 import synth
    p = synth.make_problem(1, 12, 16, 200, dtype="f32", seed=8)
    c = bench.cpu_baseline(p, max_seconds=1.0)
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1
    one = c["single_thread"]
    assert one["cores"] == 1 and one["value"] > 0 and one["unit"] == c["unit"]


def test_seqlen_override_for_profiling():
    """--seqlen runs a workload's shape with another sequence length (smaller
    profiler captures); the problem and the reported config follow it."""
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args(["--workload", "wide_state_bf16", "--seqlen", "64"])
    assert args.seqlen == 64
    old = bench.SEQLEN_OVERRIDE
    try:
        bench.SEQLEN_OVERRIDE = 64
        p, cfg = bench.workload_problem("mid_bf16", 0)
        assert p.seqlen == 64 and (p.batch, p.dim, p.dstate) == (4, 1536, 16)
    finally:
        bench.SEQLEN_OVERRIDE = old
    assert bench.parse_args([]).seqlen is None

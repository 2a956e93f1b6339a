"""Host-side pieces of bench.py, on the CPU: the multi-rank launch (gloo,
world size 2) of the reference arm, the algorithmic byte/flop accounting and
the clock-sample parser."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from sparse_moe_expert_02_gb300 import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_world_size_2_gloo():
    """Under torchrun with two ranks, rank 0 alone times the oracle and prints
    one JSON line; rank 1 exits 0 without output."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--workload", synth.TINY_F32.name, "--ref-tokens", "2"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["dtype"] == "f64"


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_algorithmic_accounting():
    shape = synth.DECODE_BF16
    counts = np.zeros(shape.E + 1, np.int64)
    counts[:475] = 1
    a = bench.algorithmic(shape, counts)
    D, I, E, T, k = shape.D, shape.I, shape.E, shape.T, shape.top_k
    per_expert = 3 * D * I * 2
    assert a["touched_experts"] == 475
    # bf16 x in, bf16 out (the bf16 layer's output), 8 bytes of routing per slot
    assert bench.out_dtype(shape) == "bf16" and bench.out_dtype(synth.TINY_F32) == "f32"
    assert a["layer_bytes"] == 476 * per_expert + E * D * 2 + T * D * 2 + T * D * 2 + 8 * T * k
    assert a["flops"] == T * (2 * D * E + (k + 1) * 6 * D * I)
    assert a["gemm_gateup_bytes"] > 476 * 2 * I * D * 2


def test_clock_summary_keeps_samples_inside_the_timed_window(tmp_path):
    c = bench.ClockSampler(0)
    c.proc = object()
    c.path = str(tmp_path / "clk.csv")
    rows = [("2026/12/02 10:00:00.000", 1000), ("2026/12/02 10:00:01.000", 2000), ("2026/12/02 10:00:01.200", 2050),
            ("2026/12/02 10:00:05.000", 900)]
    with open(c.path, "w") as fh:
        for ts, mhz in rows:
            fh.write(f"{ts}, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active\n")
    import datetime
    c.t_begin = datetime.datetime.strptime(rows[1][0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
    c.t_end = datetime.datetime.strptime(rows[2][0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
    s = c.summary()
    assert s["sm_mhz"] == 2025.0 and s["sm_max_mhz"] == 2070.0 and s["reasons"] == ["sw_power_cap"]


def test_our_arm_refuses_more_than_one_rank_before_loading_the_library():
    """--impl ours is single-GPU: under WORLD_SIZE=2 it exits non-zero with a
    message, and libmoe is never mapped into the process."""
    probe = (
        "import runpy, sys\n"
        "sys.argv = ['bench.py', '--impl', 'ours', '--steps', '2', '--warmup', '3']\n"
        "rc = 0\n"
        "try:\n"
        "    runpy.run_path('bench.py', run_name='__main__')\n"
        "except SystemExit as e:\n"
        "    rc = e.code\n"
        "maps = open('/proc/self/maps').read()\n"
        "print('LIBMOE_MAPPED' if 'libmoe' in maps else 'LIBMOE_ABSENT')\n"
        "sys.exit(rc)\n")
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", probe], capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode != 0
    assert "one GPU only" in r.stderr and "refused before loading libmoe" in r.stderr
    assert "LIBMOE_ABSENT" in r.stdout


def test_traffic_lookup_needs_every_source_unchanged(tmp_path, monkeypatch):
    """roofline.traffic: the stored ncu bytes of a stage are reported only
    while every kernel source they were taken on hashes as it did then (a
    split stage lists two); a single-source entry works the same way."""
    import hashlib
    csrc = tmp_path / "sparse_moe_expert_02_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "a.cu").write_text("one")
    (csrc / "b.cu").write_text("two")

    def sha(name):
        return hashlib.sha256((csrc / name).read_bytes()).hexdigest()[:16]

    table = {"w": {"gemm_gateup": {"source_files": ["a.cu", "b.cu"], "source_shas": [sha("a.cu"), sha("b.cu")],
                                   "dram_bytes_per_launch": 123},
                   "gemm_down": {"source_file": "a.cu", "source_sha": sha("a.cu"), "dram_bytes_per_launch": 45}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(table))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("gemm_gateup", "w") == 123
    assert bench.traffic_for("gemm_down", "w") == 45
    assert bench.traffic_for("gemm_gateup", "other") is None
    (csrc / "b.cu").write_text("two, edited")
    assert bench.traffic_for("gemm_gateup", "w") is None   # one of the two sources changed
    assert bench.traffic_for("gemm_down", "w") == 45
    (csrc / "a.cu").write_text("one, edited")
    assert bench.traffic_for("gemm_down", "w") is None

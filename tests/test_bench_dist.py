"""The multi-rank host logic of bench.py, on CPU with the gloo backend and two
ranks: the timing reduction takes the slowest rank's values, and the
reference arm prints on rank 0 only (other ranks exit 0 without work)."""
import os
import socket
import subprocess
import sys

from conftest import ROOT

_RANK_CODE = r"""
import os, sys, json
sys.path.insert(0, os.environ["BENCH_ROOT"])
import torch.distributed as dist
dist.init_process_group("gloo")
import bench
rank = dist.get_rank()
out = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 3.0], "cpu")
print(json.dumps({"rank": rank, "out": out}), flush=True)
dist.barrier()
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_two_gloo_ranks():
    import json

    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), BENCH_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_CODE], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE))
    outs = []
    for p in procs:
        so, se = p.communicate(timeout=120)
        assert p.returncode == 0, se.decode()[-2000:]
        outs.append(json.loads(so.decode().strip().splitlines()[-1]))
    for o in outs:
        assert o["out"] == [2.0, 5.0, 3.0]
    assert sorted(o["rank"] for o in outs) == [0, 1]


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, timeout=300)
    assert r.returncode == 0, r.stderr.decode()[-2000:]
    assert r.stdout.strip() == b""


def test_reference_arm_json_line():
    """The reference arm (the oracle on the host's cores) prints one JSON line
    with the contract's keys, its own value as cpu_baseline and e2e."""
    import json

    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "bitlinear-1024", "--steps", "2", "--warmup", "1", "--ref-step-seconds", "0.3"],
                       cwd=ROOT, env=env, capture_output=True, timeout=300)
    assert r.returncode == 0, r.stderr.decode()[-2000:]
    lines = r.stdout.decode().strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 1 and line["value"] > 0
    assert line["config"]["workload"] == "bitlinear-1024"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_stacks_stream_from_hbm_or_say_so():
    """Single-matrix workloads default to enough copies to stream three times
    the L2 per step; the line's L2 note follows the stack's actual size."""
    sys.path.insert(0, ROOT)
    import bench
    from ternary_weight_05_b300 import synth

    for w in ("gateup-sweep", "bitlinear-1024"):
        args = bench.parse(["--workload", w])
        L = synth.workload(w).layers[0]
        assert args.layers * L.N * L.K // 4 >= 3 * bench.L2_BYTES
    assert bench.parse(["--workload", "2b-decode"]).layers == 30
    assert bench.parse(["--workload", "bitlinear-1024", "--layers", "5"]).layers == 5
    assert bench.l2_note(496e6).startswith("inputs larger than L2")
    assert bench.l2_note(7.9e6).startswith("L2-resident")


def test_cpu_baseline_object():
    """The native line's cpu_baseline: the oracle on all host cores and on one
    thread, over a bounded sample of the workload."""
    sys.path.insert(0, ROOT)
    import bench

    cb = bench.cpu_baseline(bench.parse(["--workload", "bitlinear-1024", "--cpu-seconds", "0.4"]))
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["cores"] >= 1
    assert cb["value"] > 0 and cb["value_1thread"] > 0
    assert "pass(es)" in cb["sample"] and "one thread" in cb["sample_1thread"]

"""CPU checks of bench.py's multi-process plumbing (no GPU): the max / sum reductions over ranks on
a world-size-2 gloo group, and the reference arm under torchrun with two ranks (rank 0 alone runs
the oracle and prints one JSON line; the other rank exits 0 without work)."""

import json
import os
import socket
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.max_over_ranks(dist, float(rank + 1))
        sm = bench.sum_over_ranks(dist, float(10 * (rank + 1)))
        bench.barrier(dist)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"max": mx, "sum": sm}, f)
    finally:
        dist.destroy_process_group()


def test_reductions_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    port = _free_port()
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_reduce_worker, args=(2, port, d), nprocs=2, join=True, start_method="spawn")
        for r in range(2):
            got = json.load(open(os.path.join(d, f"r{r}.json")))
            assert got == {"max": 2.0, "sum": 30.0}


def test_single_process_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.sum_over_ranks(None, 2.0) == 2.0


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=540, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 1
    assert line["config"]["workload"] == "tiny"
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_algorithmic_bytes_match_the_closed_forms():
    """bench.step_bytes (the numerator of every roofline fraction) against the per-call byte counts
    written out for the workloads: K+V of every visible key once, q in / o out, the logits once
    plus the one re-read row pair, and the draft ring's visible slots."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    from workloads.configs import CONFIGS
    md = CONFIGS["magicdec-64k"]
    inp = {"kv_len_h": np.full(md.B, 65536), "pos0": np.full(md.B, 65536)}
    nb = bench.step_bytes(md, inp)
    assert nb["verify_kv"] == 32 * 65536 * 8 * 128 * 2 * 2                  # 8.59 GB
    assert nb["verify_total"] == nb["verify_kv"] + 32 * 5 * 32 * 128 * (2 + 4)
    assert nb["sample"] == 32 * 9 * 128256 * 4 + 32 * 2 * 128256 * 4
    assert nb["window"] == 32 * 512 * 8 * 128 * 2 * 2 + 32 * 32 * 128 * (2 + 4)
    tr = CONFIGS["medusa-tree-8k"]
    nb = bench.step_bytes(tr, {"kv_len_h": np.full(tr.B, 8192)})
    assert nb["verify_kv"] == 4 * 8192 * 8 * 128 * 2 * 2                      # 134 MB
    assert nb["sample"] == 4 * 64 * 32000 * 4
    b8 = CONFIGS["llama3-8b-layer"]
    lens = np.array([16384, 20000, 32768, 17000, 25000, 30000, 16500, 31000])
    nb = bench.step_bytes(b8, {"kv_len_h": lens})
    assert nb["verify_kv"] == int(lens.sum()) * 8 * 128 * 4
    assert nb["window"] == 0


def test_committed_counters_attach_only_to_the_workloads_own_sizes():
    """roofline.traffic comes from an ncu capture of one kernel revision at one workload's sizes:
    a run with a --batch or --context override must not carry it."""
    sys.path.insert(0, ROOT)
    import bench
    from workloads.configs import get_config, scaled
    for name in ("magicdec-64k", "llama3-8b-layer"):
        cfg = get_config(name)
        full = bench.profile_counters(cfg)
        if full is not None:
            assert full.get("kernel_rev") == bench.KERNEL_REVS[name]
        assert bench.profile_counters(scaled(cfg, ctx=(4096, 4096))) is None
        assert bench.profile_counters(scaled(cfg, B=2)) is None

"""The N>1 path of the benchmark on CPU: gloo ranks (world size 2) exercise
the max-over-ranks timing and the whole-job rate the benchmark reports.  The
op itself shards by tokens with no collective on the data path, so this
host logic is all that multi-GPU runs add."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist, "cpu")
        value, tok = bench.whole_job_rates(1_000_000, 4096, world, ms)
        out[rank] = (ms, value, tok)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_whole_job_rate(world):
    times = [0.020, 0.025][:world]
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), times, out), nprocs=world, join=True)
    for r in range(world):
        ms, value, tok = out[r]
        assert ms == max(times)
        assert value == pytest.approx(1_000_000 * world / (max(times) / 1e3) / 1e9)
        assert tok == pytest.approx(4096 * world / (max(times) / 1e3))


def test_single_process_passthrough():
    assert bench.max_over_ranks(1.5, None, "cpu") == 1.5
    v, t = bench.whole_job_rates(2_000_000_000, 1000, 1, 1000.0)
    assert v == pytest.approx(2.0) and t == pytest.approx(1000.0)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    class A:
        workload, steps, warmup = "llama_fp8_per_token", 3, 3
    bench.run_reference(A, rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the oracle timed on the host cores) prints
    one JSON line with the contract's keys, on the default workload."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, cwd=root, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "dsv3_fp8_group128_row"
    # the same config object as the GPU arm prints for this workload
    import rmsq_inputs as ri
    assert d["config"] == json.loads(json.dumps(bench.workload_config("dsv3_fp8_group128_row", ri.dsv3(8192),
                                                                       "fp8_group128_row")))
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}

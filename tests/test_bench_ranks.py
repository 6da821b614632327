"""The multi-rank launch logic of ``bench.py`` on host-only ``gloo`` ranks
(world size 2): rendezvous, barrier, max-over-ranks timing, whole-job
throughput, and the reference arm printing on rank 0 only.  The layer runs
replicas only (no collective on the data path), so this host logic is the
whole of the N > 1 path."""

import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import contextlib
    import io

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    args = bench.parse_args_from(["--gpus", str(world), "--impl", "reference", "--workload", "tiny",
                                  "--steps", "1", "--warmup", "0"])
    w, r, _ = bench.dist_setup(args)
    # rank 1 is the slower one: the job's step time is its time
    ms = bench.max_over_ranks(w, 10.0 + 5.0 * r)
    bench.barrier(w)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.run_reference(args)
    bench.barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "ms": ms, "rc": rc, "stdout": buf.getvalue(),
                   "tflops": bench.job_tflops(w, 1e12, ms)}, f)


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["world"] == world and d["rank"] == r and d["rc"] == 0
        assert d["ms"] == 15.0                       # max over ranks, on every rank
        assert d["tflops"] == pytest.approx(2 * 1e12 / 15e-3 / 1e12)
    assert res[1]["stdout"] == ""                    # only rank 0 prints
    lines = [l for l in res[0]["stdout"].splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == world and line["value"] > 0
    assert line["config"]["parallelism"] == "replicas"


def test_job_tflops_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_tflops(1, 18e12, 18.0) == pytest.approx(1000.0)
    assert bench.job_tflops(4, 18e12, 18.0) == pytest.approx(4000.0)

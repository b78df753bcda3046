"""World-size-2 checks of the bench's multi-process host logic on the CPU
(gloo): the slowest rank's time is the job's time on every rank, the job's
throughput counts every rank's work, and the reference arm runs on rank 0
only.  (On GPUs the same functions run over NCCL; the ranks are replicas and
exchange nothing but these numbers.)"""
import io
import json
import os
import socket
import sys
from argparse import Namespace
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.0][rank]
    ms = bench.max_over_ranks(local_ms)
    value = bench.whole_job_tflops(1e12, world, ms)
    buf = io.StringIO()
    ref_printed = None
    if rank != 0:  # the reference arm does no work and prints nothing off rank 0
        with redirect_stdout(buf):
            bench.bench_reference(Namespace(gpus=world, steps=1, warmup=3))
        ref_printed = buf.getvalue()
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value, "ref_printed": ref_printed}, f)


def test_two_ranks_gloo(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["ms"] == r1["ms"] == 5.0                      # the slower rank decides
    assert r0["value"] == pytest.approx(2 * 1e12 / 5e-3 / 1e12)  # both ranks' work over that time
    assert r1["ref_printed"] == ""


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.whole_job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)

"""Host logic of the multi-GPU bench path, on CPU: two gloo ranks.

The path has no exchange step, so N GPUs run independent replicas; what the
bench needs from torch.distributed is the barrier around the timed region and
the max of the elapsed times over ranks.  These tests run that logic with
world_size 2 on the gloo backend, plus the reference arm's rule that only
rank 0 runs and prints.
"""
import json
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, _ = bench.dist_env()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    # each rank "measured" a different elapsed time; every rank must see the slowest one
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"ms": ms}, f)
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [json.load(open(tmp_path / ("rank%d.json" % r)))["ms"] for r in range(2)]
    assert got == [15.0, 15.0]


def _ref_worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import contextlib
    import io
    import types
    import bench
    args = types.SimpleNamespace(config="tiny", steps=2, warmup=1, gpus=world)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, world, rank)
    with open(os.path.join(out_dir, "ref%d.txt" % rank), "w") as f:
        f.write(buf.getvalue())


def test_reference_arm_prints_on_rank0_only(tmp_path):
    port = _free_port()
    mp.spawn(_ref_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    out0 = (tmp_path / "ref0.txt").read_text().strip().splitlines()
    out1 = (tmp_path / "ref1.txt").read_text().strip()
    assert out1 == ""
    assert len(out0) == 1
    line = json.loads(out0[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0

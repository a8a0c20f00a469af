"""The multi-rank host logic of bench.py on CPU with gloo, world size 2.

Each rank draws its own batch (seed = rank: weak scaling, no data exchange),
the per-rank times are reduced with a max, and the whole-job value counts all
ranks' bytes over the slowest rank's time.  The oracle arm runs on rank 0 only.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from paged_kv_cache_293_gb300 import workloads
    w = workloads.make("tiny", seed=rank, device="cpu")
    fake_ms = 1.0 + rank                               # rank 1 is the slow one
    worst = bench.max_over_ranks(fake_ms, world, torch.device("cpu"))
    bench.barrier(world)
    np.save(os.path.join(out_dir, "q%d.npy" % rank), workloads.storage_numpy(w.q))
    with open(os.path.join(out_dir, "r%d.txt" % rank), "w") as f:
        f.write("%r" % worst)
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_ranks_take_the_slowest_time_and_draw_their_own_batches(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    worst = [float((tmp_path / ("r%d.txt" % r)).read_text()) for r in range(world)]
    assert worst == [2.0, 2.0]
    q0, q1 = np.load(tmp_path / "q0.npy"), np.load(tmp_path / "q1.npy")
    assert q0.shape == q1.shape and not np.array_equal(q0, q1)


def _ref_worker(rank, world, port, out_dir):
    import contextlib
    import io
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    args = type("A", (), dict(workload="tiny", seed=0, steps=2, warmup=3))()
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args)
    with open(os.path.join(out_dir, "ref%d.txt" % rank), "w") as f:
        f.write(buf.getvalue())


@pytest.mark.timeout(300)
def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    import json
    world, port = 2, _free_port()
    mp.spawn(_ref_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    out0 = (tmp_path / "ref0.txt").read_text().strip()
    out1 = (tmp_path / "ref1.txt").read_text().strip()
    assert out1 == ""
    line = json.loads(out0)
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0

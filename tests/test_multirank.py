"""Host-side multi-rank logic of bench.py with two gloo ranks on CPU.

Each rank runs its own independent heads (weak scaling, no data-path
collective); only the timing is reduced with a max over ranks.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from online_softmax_tiling_gb300 import synth
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    t = bench.max_over_ranks(10.0 + rank, world)       # per-rank timings -> slowest rank
    bench.barrier(world)
    wl = synth.Workload("tiny", 1, 2, 8, 16, synth.BF16, 0.25, False, 9000)
    q, _, _ = synth.make_inputs(wl, seed_base=bench.rank_seed_base(wl, rank))
    np.save(os.path.join(out_dir, f"q{rank}.npy"), q)
    with open(os.path.join(out_dir, f"t{rank}.txt"), "w") as fh:
        fh.write(repr(t))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timing_and_draw_disjoint_units(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    times = [float(open(tmp_path / f"t{r}.txt").read()) for r in range(world)]
    assert times == [11.0, 11.0]
    q0, q1 = (np.load(tmp_path / f"q{r}.npy") for r in range(world))
    assert q0.shape == q1.shape and not np.array_equal(q0, q1)

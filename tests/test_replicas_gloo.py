"""The multi-GPU path is data parallel with independent replicas: no
collective touches the data path; only the timings are reduced (max over
ranks). Checked here with two gloo ranks on CPU."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synth
    wl = bench.replica_workload(rank)
    x0 = synth.hidden_states(wl.replace(batch=1), 1)[0]       # one block of this replica's inputs
    live, dec = synth.block_masks(wl.replace(batch=1), 4)
    reduced = bench.reduce_max_over_ranks([1.0 + rank, 10.0 - rank])
    out[rank] = (wl.iid, wl.wid, float(x0.astype(np.float64).sum()), live.sum(), reduced)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_have_distinct_inputs_and_max_reduced_timings():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        r0, r1 = out[0], out[1]
    assert r0[1] == r1[1]                  # same layer weights on every replica
    assert r0[0] != r1[0] and r0[2] != r1[2]  # each replica serves its own requests
    assert r0[4] == r1[4] == [2.0, 10.0]   # timings reduced with a max over ranks


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max_over_ranks([3.5, 1.0]) == [3.5, 1.0]

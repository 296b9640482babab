"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each an independent replica;
the whole-job value divides all ranks' tokens by the slowest rank's time."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    seconds = [2.0, 3.0][rank]          # rank 1 is the slowest
    v = bench.whole_job_tokens_per_s(4096, 10, world, seconds)
    m = bench.max_over_ranks(float(rank + 5), world)
    out[rank] = (v, m)
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    for r in range(world):
        v, m = out[r]
        assert abs(v - 2 * 4096 * 10 / 3.0) < 1e-6
        assert m == 6.0


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert abs(bench.whole_job_tokens_per_s(100, 4, 1, 2.0) - 200.0) < 1e-12


def test_reference_half_layer_steps_are_one_layer_forward():
    """The reference arm's two half-layer steps compute exactly the oracle's layer forward
    (same library calls on the same blocks), so its tokens/s counts two steps as one
    layer of T tokens."""
    import numpy as np

    import bench
    from oracle import moe_oracle as O
    from routing_dispatch_expert_04_b300.workloads import WORKLOADS, make_inputs
    for name in ("tiny",):
        wl = WORKLOADS[name]
        inp = make_inputs(wl, "cpu", seed=0)
        orc = bench.HalfLayerOracle(wl, inp)
        orc.step()
        orc.step()
        ref = O.moe_forward(inp["x"].numpy(), inp["w_r"].numpy(), None, inp["w1"].numpy(),
                            inp["w2"].numpy(), wl.K, O.capacity(wl.T, wl.E, wl.capacity_factor),
                            wl.alpha)
        assert np.array_equal(orc.y, ref["y"])


def test_both_arms_print_the_same_config():
    import bench
    from routing_dispatch_expert_04_b300.workloads import WORKLOADS
    wl = WORKLOADS["mixtral"]
    c = bench.workload_config(wl, 640, 1)
    assert c == bench.workload_config(wl, 640, 1)
    assert c["workload"].startswith("mixtral: T=4096 d=4096 E=8 K=2 F=16384")
    assert set(c) == {"workload", "capacity", "parallelism", "l2"}

"""The N > 1 host logic of bench.py on CPU: two gloo ranks.

Each rank runs its own replica of the workload (weak scaling, no collective on the
data path); the only cross-rank steps are the barrier and the max over ranks of the
timed region, which the reported throughput divides by.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.barrier(world)
    t = bench.max_over_ranks(10.0 + rank, world)
    seeds = [bench.replica_seed(4096, q) for q in range(world)]
    out[rank] = (t, seeds[rank], len(set(seeds)))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time_and_distinct_replicas():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 11.0          # max over ranks
    assert out[0][1] != out[1][1] and out[0][2] == world  # each rank draws its own replica


def test_single_rank_defaults():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    assert bench.dist_env()[0] == 1
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_seed(7, 0) == 7


def test_bench_helpers_without_a_gpu():
    """The parts of the benchmark line that need no GPU: kernel counting per step, the
    comment-insensitive kernel hash, the roofline bound choice and the measured-traffic key."""
    import importlib.util
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    from attention_forward_07_gb300 import inputs as inp
    assert bench.kernels_per_step(inp.WORKLOADS["short_masked"]) == 3
    assert bench.kernels_per_step(inp.WORKLOADS["gqa8_causal_S8192"]) == 1
    h = bench.kernel_hash()
    assert len(h) == 12 and h == bench.kernel_hash()
    w = inp.WORKLOADS["gqa8_causal_S8192"]
    r = bench.roofline(w, 1.4e-3)
    assert r["bound"] == "tensor" and abs(r["achieved"] - w.flops() / 1.4e-3 / 1e12) < 1e-6
    assert bench.config_key(w) == "B4_Hq32_Hkv8_S8192_d128_causal_none"
    r = bench.roofline(inp.WORKLOADS["short_masked"], 60e-6)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"


def test_bench_algorithmic_units_of_the_masked_workloads():
    """The 90 %-masked workload's algorithmic bytes count the Q rows of the 16-row blocks that
    keep anything (measured from the mask), not the whole Q; the live fraction is exact on a
    hand-built mask."""
    import importlib.util
    import os
    import numpy as np
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    from dataclasses import replace
    from attention_forward_07_gb300 import inputs as inp
    w = replace(inp.WORKLOADS["short_masked90"], B=2, S=40)
    keep = np.ones((2, 40, 40), bool)
    keep[0, 0:16] = False          # block 0 of entry 0 keeps nothing
    keep[1, 32:40] = False         # the ragged last block of entry 1 keeps nothing
    keep[1, 20, :] = False         # one empty row inside a live block does not empty it
    assert bench.live_fraction(w, inp.pack_bits(keep)) == 4 / 6
    assert bench.live_fraction(w, None) == 1.0
    w90 = inp.WORKLOADS["short_masked90"]
    _, _, _, bits = w90.make(w90.seed(list(inp.WORKLOADS).index("short_masked90")))
    live = bench.live_fraction(w90, bits)
    assert 0.15 < live < 0.25
    q_bytes = w90.B * w90.Hq * w90.S * w90.d * 2
    assert bench.algorithmic_bytes(w90) - bench.algorithmic_bytes(w90, live) == q_bytes - round(q_bytes * live)
    r = bench.roofline(w90, 49.3e-6, live)
    assert r["bound"] == "hbm" and r["algorithmic_bytes"] == bench.algorithmic_bytes(w90, live)

"""The multi-process path of bench.py on CPU: two ranks over gloo.

Each rank verifies its own batch of the seeded row stream (weak scaling, no
data-path collective); the only collectives are the barrier around the timed
region and the max over ranks of the elapsed time, and the reference arm
runs on rank 0 only.
"""

import json
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank) and dist.get_backend() == "gloo"
    case = bench.make_workload("c1", row0=bench.rank_row0(rank))
    # every rank's batch, gathered only here, to check that ranks do not share rows
    t = case.target.reshape(-1).double()
    got = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(got, t)
    bench.barrier(w)
    mx = bench.max_over_ranks(float(rank + 1) * 1.5, w, torch.device("cpu"))
    ref_line = bench.run_reference(None, w, r) if r != 0 else "rank0"
    res = {"max": mx, "distinct": bool(not torch.equal(got[0], got[1])),
           "ref_other_ranks": ref_line, "row0": bench.rank_row0(rank)}
    # rank r's batch is the seeded stream from rank_row0(r): regenerate one row alone
    from speculative_decoding_verification_48_gb300 import workloads as W
    one = W.make_chain("c1_check", 1001, 1, 4, 1000, "f32", target="normal", target_sigma=2.0,
                       draft_sigma=(0.5, 0.5), temperature=1.0, row0=bench.rank_row0(rank))
    res["stream_consistent"] = bool(torch.equal(one.target[0], case.target[0]))
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_batches_and_take_max_time(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["max"] == 3.0                 # max over ranks of (rank + 1) * 1.5
        assert r["distinct"]                   # the two batches are different rows
        assert r["stream_consistent"]
    assert res[1]["ref_other_ranks"] is None   # the reference arm returns at once off rank 0
    assert res[0]["row0"] != res[1]["row0"]
    assert np.isfinite([r["max"] for r in res]).all()

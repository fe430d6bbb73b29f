"""The multi-GPU mode is replicas only: every rank runs the whole layer on
its own tokens with its own copy of the table, and the only exchange is the
slowest rank's time. This checks that host-side logic on two gloo ranks on
the CPU: the max-over-ranks reduction every rank applies to its timings, the
whole-job throughput, and that the ranks' token batches (and so their
outputs, computed here with the oracle on a tiny layer) are independent."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
dist = pytest.importorskip("torch.distributed")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    import bench
    from oracle import moe_oracle as O
    from w4a16_routed_expert_gb300 import synth

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # per-rank step times: the slowest one is what every rank reports
        local_ms = 1.0 + 0.5 * rank
        slowest = bench._max_over_ranks(torch, torch.device("cpu"), world, local_ms)
        value = bench.replica_throughput(4, world, slowest)
        # each replica's own batch (the seeds the bench uses) through the oracle
        shape = synth.TINY
        lay = synth.make_layer(shape, seed=0)
        x = synth.make_tokens(shape.hidden, 4, seed=1000 * (rank + 1))
        ref = O.moe_forward(x, lay.router_w, None, lay.records, lay.expert_to_slot, H=shape.hidden,
                            I=shape.intermediate, E=shape.num_experts, k=shape.top_k, G=shape.group_size,
                            renormalize=shape.renormalize)
        np.savez(os.path.join(outdir, f"rank{rank}.npz"), slowest=slowest, value=value, x=x, out=ref["out"],
                 ids=ref["ids"])
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r = [np.load(tmp_path / f"rank{i}.npz") for i in range(world)]
    for i in range(world):
        assert float(r[i]["slowest"]) == 1.5  # every rank holds the slowest rank's time
        assert float(r[i]["value"]) == pytest.approx(4 * world / 1.5e-3)
    # replicas see different tokens, so their results differ; each is the
    # oracle's own answer for its batch
    assert not np.array_equal(r[0]["x"], r[1]["x"])
    assert not np.allclose(r[0]["out"], r[1]["out"])
    sys.path.insert(0, ROOT)
    from oracle import moe_oracle as O
    from w4a16_routed_expert_gb300 import synth
    lay = synth.make_layer(synth.TINY, seed=0)
    s = synth.TINY
    for i in range(world):
        ref = O.moe_forward(r[i]["x"], lay.router_w, None, lay.records, lay.expert_to_slot, H=s.hidden,
                            I=s.intermediate, E=s.num_experts, k=s.top_k, G=s.group_size,
                            renormalize=s.renormalize)
        assert np.array_equal(ref["ids"], r[i]["ids"])
        assert np.array_equal(ref["out"], r[i]["out"])

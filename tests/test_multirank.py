"""Multi-rank host logic of the benchmark (weak scaling, one process per GPU),
run as two gloo ranks on the CPU: each rank verifies its own batch, ranks
draw independent Philox streams, and the job's throughput is the units of all
ranks over the slowest rank's time.  The verify itself has no exchange step
between ranks (sequences are independent), so these are the only collectives.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from speculative_decoding_verification_vocab_gb300 import synth

    r, w, _ = bench.dist_env()
    seq0, B = bench.shard_batch(8, r, w)
    # each rank: rows processed and a made-up duration (rank 1 is slower)
    total, ms_max, value = bench.aggregate(100.0 * (r + 1), 2.0 + r, w)
    # one small chain round per rank, through the oracle, with the rank's key
    cfg = synth.CONFIGS[1]
    vq, dp, d = synth.chain_inputs(cfg, seed=11, B=B, V=64, N=3)
    o = oracle.verify_chain(vq.float().numpy(), dp.float().numpy(), d.numpy(), T=1.0,
                            seed=bench.rank_seed(1234, r), step=0)
    dist.barrier()
    np.savez(os.path.join(out, f"rank{r}.npz"), seq0=seq0, B=B, total=total, ms_max=ms_max,
             value=value, tokens=o["tokens"], accept=o["accept_len"])
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    import oracle
    oracle.build()
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    # weak scaling: same per-rank batch, disjoint global sequence ranges
    assert [int(x["B"]) for x in res] == [8, 8]
    assert [int(x["seq0"]) for x in res] == [0, 8]
    # whole-job throughput: sum of units over the max time, identical on ranks
    for x in res:
        assert float(x["total"]) == 300.0
        assert float(x["ms_max"]) == 3.0
        assert float(x["value"]) == pytest.approx(300.0 / 3e-3)
    # same inputs, different keys: the ranks' draws differ
    assert not (np.array_equal(res[0]["tokens"], res[1]["tokens"]) and
                np.array_equal(res[0]["accept"], res[1]["accept"]))


def test_reference_arm_only_rank0(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    bench.run_reference(bench.parse())
    assert capsys.readouterr().out == ""

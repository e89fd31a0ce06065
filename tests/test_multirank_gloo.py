"""The multi-rank host path on CPU: two gloo ranks.

* the expert partition of ``quantized_moe_expert_topk_gb300.ep`` covers every
  expert exactly once, and each rank's layer (its own expert weights, its
  ``expert_map``, computed here by the fp64 oracle) sums over the ranks to the
  full layer -- the per-rank computation of expert parallelism;
* ``replica_max`` gives every rank the slowest rank's time, as the benchmark
  needs when it runs one replica per GPU.
"""
import os
import socket

import numpy as np
import pytest

from quantized_moe_expert_topk_gb300.ep import expert_map_for_rank, expert_partition, local_weights


def test_expert_partition_covers_each_expert_once():
    for E in (1, 5, 8, 32, 257):
        for world in (1, 2, 3, 4, 8):
            owner = np.full(E, -1)
            for rank in range(world):
                first, count = expert_partition(E, world, rank)
                assert count in (E // world, E // world + 1)
                assert (owner[first:first + count] == -1).all()
                owner[first:first + count] = rank
                emap, El = expert_map_for_rank(E, world, rank)
                assert El == count
                assert (emap[first:first + count] == np.arange(count)).all()
                assert (np.delete(emap, np.arange(first, first + count)) == -1).all()
            assert (owner >= 0).all() and (np.diff(owner) >= 0).all()
    with pytest.raises(ValueError):
        expert_partition(8, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_dir):
    import torch
    import torch.distributed as dist

    import oracle
    from moe_workloads import make_custom, to_host
    from quantized_moe_expert_topk_gb300.ep import replica_max

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # slowest-rank time
        assert replica_max(1.0 + 10.0 * rank) == 1.0 + 10.0 * (world - 1)

        # expert-parallel partition of a small MXFP4 SwiGLU-OAI layer with biases
        E = 6
        wl = make_custom(M=24, K=64, N=32, E=E, T=2, wfmt="mxfp4", afmt="bf16",
                         act="swiglu_oai", gate="interleaved", bias=True, seed=21, name="ep_gloo")
        h = to_host(wl)
        emap, El = expert_map_for_rank(E, world, rank)
        prob = dict(h["problem"], El=El)
        w13 = {k: (local_weights(v, E, world, rank) if v is not None and v.ndim >= 1 else v)
               for k, v in h["w13"].items()}
        w2 = {k: (local_weights(v, E, world, rank) if v is not None and v.ndim >= 1 else v)
              for k, v in h["w2"].items()}
        part = oracle.fused_experts(prob, h["x"], w13, w2, h["topk_ids"], h["topk_weights"], emap)
        total = torch.from_numpy(part.copy())
        dist.all_reduce(total, op=dist.ReduceOp.SUM)
        if rank == 0:
            full = oracle.fused_experts(h["problem"], h["x"], h["w13"], h["w2"], h["topk_ids"],
                                        h["topk_weights"], h["expert_map"])
            rms = float(np.sqrt((full ** 2).mean()))
            err = float(np.abs(total.numpy() - full).max())
            assert rms > 0 and err <= 1e-12 * rms, (err, rms)
        open(os.path.join(result_dir, f"ok{rank}"), "w").close()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    import oracle
    oracle.lib()  # build the oracle library once, before the ranks load it
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for rank in range(world):
        assert (tmp_path / f"ok{rank}").exists()

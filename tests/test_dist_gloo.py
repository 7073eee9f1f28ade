"""World-size-2 gloo checks of the weak-scaling plumbing (CPU only): the process group comes up from
the launcher's environment, the timing reduction takes the max over ranks, shards partition the
units, and each rank's shard is its own independent workload: the oracle over the two shards run
separately equals the oracle over the two shards stacked as one bank (streams never interact)."""

from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, outdir: str):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from decode_state_gb300 import dist as sdist, workloads
    import oracle

    r = sdist.init_from_env(backend="gloo")
    assert (r.rank, r.world) == (rank, world)
    sdist.barrier(r)
    assert sdist.max_over_ranks(r, 10.0 + rank) == 10.0 + world - 1
    assert sdist.sum_over_ranks(r, 1.0) == float(world)
    lo, hi = sdist.shard_range(1027, r)
    wl = workloads.C0.scaled(n_streams=3, T=4)
    x = workloads.make_decode_inputs(wl, seed=sdist.shard_seed(wl.seed, r))
    bank = x["bank"].numpy().copy()
    out = oracle.decode_seq(bank, *(x[k].numpy() for k in ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")))
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), lo=lo, hi=hi, out=out, bank_after=bank,
             **{k: x[k].numpy() for k in ("bank", "k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")})
    sdist.shutdown(r)


def test_two_rank_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    import oracle

    r0, r1 = (np.load(tmp_path / f"rank{i}.npz") for i in range(2))
    assert (int(r0["lo"]), int(r0["hi"]), int(r1["lo"]), int(r1["hi"])) == (0, 514, 514, 1027)
    assert not np.array_equal(r0["v"], r1["v"]), "ranks must draw different shards"
    # the two shards stacked as one job (stream slots of rank 1 shifted past rank 0's bank)
    n0 = r0["bank"].shape[0]
    joint = np.concatenate([r0["bank"], r1["bank"]])
    args = []
    for k in ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val"):
        b = r1[k] + n0 if k in ("k_idx", "q_idx") else r1[k]
        args.append(np.concatenate([r0[k], b], axis=1))
    out = oracle.decode_seq(joint, *args)
    assert np.array_equal(out, np.concatenate([r0["out"], r1["out"]], axis=1))
    assert np.array_equal(joint, np.concatenate([r0["bank_after"], r1["bank_after"]]))

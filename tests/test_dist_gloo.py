"""World-size-2 gloo checks of the multi-process plumbing (CPU only): the process group comes up from
the launcher's environment, the timing reduction takes the max over ranks, shards partition the
units, and one decode job split over the ranks by stream ranges (each rank drawing only its own
streams and their bank rows) gives, from the oracle on each rank's shard, exactly the readings and
bank of the oracle over the whole job in one process (streams never interact)."""

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
    # one job of 5 streams in blocks of 2 (the last block shorter): this rank's stream range only
    job = workloads.C0.scaled(n_streams=5, T=4, slots_per_stream=48)
    s0, s1 = sdist.stream_shard(job.n_streams, r, 2)
    x = workloads.make_decode_shard(job, s0, s1, block=2)
    bank = x["bank"].numpy().copy()
    out = oracle.decode_seq(bank, *(x[k].numpy() for k in ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")))
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), lo=lo, hi=hi, s0=s0, s1=s1, out=out, bank_after=bank,
             **{k: x[k].numpy() for k in ("bank", "k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")})
    sdist.shutdown(r)


def test_two_rank_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    import oracle

    from decode_state_gb300 import workloads

    r0, r1 = (np.load(tmp_path / f"rank{i}.npz") for i in range(2))
    assert (int(r0["lo"]), int(r0["hi"]), int(r1["lo"]), int(r1["hi"])) == (0, 514, 514, 1027)
    # 3 blocks of 2, 2 and 1 streams: rank 0 holds streams [0, 4), rank 1 stream 4
    assert (int(r0["s0"]), int(r0["s1"]), int(r1["s0"]), int(r1["s1"])) == (0, 4, 4, 5)
    assert r0["v"].shape[1] == 4 and r1["v"].shape[1] == 1 and r1["bank"].shape[0] == 48
    # slots are local to each rank's bank rows
    for rr in (r0, r1):
        n = rr["bank"].shape[0]
        assert rr["k_idx"].min() >= 0 and rr["k_idx"].max() < n and rr["q_idx"].max() < n
    # the whole job in one process: the same streams, the same bank, and the union of the two
    # ranks' oracle runs equals the oracle over it
    job = workloads.C0.scaled(n_streams=5, T=4, slots_per_stream=48)
    x = workloads.make_decode_shard(job, 0, 5, block=2)
    keys = ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")
    assert np.array_equal(x["bank"].numpy(), np.concatenate([r0["bank"], r1["bank"]]))
    assert np.array_equal(x["v"].numpy(), np.concatenate([r0["v"], r1["v"]], axis=1))
    bank = x["bank"].numpy().copy()
    out = oracle.decode_seq(bank, *(x[k].numpy() for k in keys))
    assert np.array_equal(out, np.concatenate([r0["out"], r1["out"]], axis=1))
    assert np.array_equal(bank, np.concatenate([r0["bank_after"], r1["bank_after"]]))

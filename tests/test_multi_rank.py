"""The N > 1 path on CPU: two gloo ranks as separate processes.

The GEMM runs as independent replicas (no data-path collective), so what is
tested here is the host logic that crosses ranks: the rank object bench.py
uses (barrier, max / sum over ranks), the output-column sharding, and the
gather of column blocks -- each rank computing its block with the oracle and
the gathered matrix compared bit for bit with the unsharded oracle result.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import workloads
from block_scaled_precision_persistent_gb300.replicas import Ranks, shard_range


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r = Ranks("gloo", expected_world=world)
    try:
        assert (r.rank, r.world) == (rank, world)
        r.barrier()
        # the job takes as long as its slowest rank; totals add up
        assert r.max(1.5 + rank) == 1.5 + (world - 1)
        assert r.sum(float(rank + 1)) == world * (world + 1) / 2
        # column-sharded GEMM: this rank's block with the oracle, then gathered
        M, N, K = 40, 200, 512
        p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)
        n0, n1 = shard_range(N, world, rank)
        o = oracle.get()
        _, _, bits = o.nvfp4_gemm(p["A"].numpy(), p["sfA"].numpy(), p["B"].numpy(), p["sfB"].numpy(),
                                  p["alpha"], K, cols=list(range(n0, n1)), nthreads=1)
        block = torch.from_numpy(bits.astype(np.int32)).reshape(M, n1 - n0)
        full = r.gather_columns(block, N)
        np.save(os.path.join(out_dir, f"gathered_{rank}.npy"), full.numpy())
    finally:
        r.close()


def test_shard_range_covers_columns_once():
    for n in (0, 1, 8, 136, 200, 3072, 12289):
        for world in (1, 2, 3, 4, 8):
            edges = [shard_range(n, world, r) for r in range(world)]
            assert edges[0][0] == 0 and edges[-1][1] == n
            for (a0, a1), (b0, b1) in zip(edges, edges[1:]):
                assert a1 == b0                     # contiguous, disjoint
            for a0, a1 in edges:
                assert a0 <= a1 and a0 % 8 == 0     # every block starts on an 8-column edge
                assert (a1 - a0) % 8 == 0 or a1 == n
            widths = [a1 - a0 for a0, a1 in edges]
            assert max(widths) - min(widths) <= 8 or n < 8 * world


def test_shard_range_rejects_bad_arguments():
    with pytest.raises(ValueError):
        shard_range(16, 0, 0)
    with pytest.raises(ValueError):
        shard_range(16, 2, 2)
    with pytest.raises(ValueError):
        shard_range(-1, 2, 0)


def test_single_rank_is_identity(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    r = Ranks("gloo")
    assert (r.world, r.rank, r.pg) == (1, 0, False)
    assert r.max(3.0) == 3.0 and r.sum(2.0) == 2.0
    x = torch.arange(6).reshape(2, 3)
    assert r.gather_columns(x, 3) is x
    r.barrier()
    r.close()


def test_two_gloo_ranks_shard_and_gather(tmp_path):
    oracle.build()                    # once, before the ranks start
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    M, N, K = 40, 200, 512
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)
    _, _, ref = oracle.get().nvfp4_gemm(p["A"].numpy(), p["sfA"].numpy(), p["B"].numpy(), p["sfB"].numpy(),
                                        p["alpha"], K, nthreads=2)
    for rank in range(world):
        got = np.load(tmp_path / f"gathered_{rank}.npy")
        assert got.shape == (M, N)
        np.testing.assert_array_equal(got.astype(np.uint16), ref.astype(np.uint16))

"""World-size-2 gloo checks of the multi-GPU host logic (CPU only): ranks
take disjoint problem ranges, the timing reduction is a max over ranks, and
independent problems sharded over ranks reproduce the single-process result
with no data exchange (checked with the oracle on tiny inputs)."""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import oracle
    from long_context_attention_seqattn_gb300 import dist
    r, w = dist.init("gloo")
    assert (r, w) == (rank, world)
    # 5 independent (batch entry, kv head) problems split over the ranks
    lo, hi = dist.shard_units(5, r, w)
    rng = np.random.default_rng(0)
    q = rng.standard_normal((5, 24, 2, 4))
    k = rng.standard_normal((5, 24, 1, 4))
    v = rng.standard_normal((5, 24, 1, 4))
    do = rng.standard_normal((5, 24, 2, 4))
    res = oracle.chunked_layer(q[lo:hi], k[lo:hi], v[lo:hi], do[lo:hi], 8, 0.5)
    np.savez(os.path.join(out_dir, f"rank{r}.npz"), lo=lo, hi=hi, *res)
    m = dist.max_over_ranks(float(r + 1))
    s = dist.sum_over_ranks(float(hi - lo))
    dist.barrier()
    np.save(os.path.join(out_dir, f"red{r}.npy"), np.array([m, s]))
    dist.finalize()


def test_shard_units_cover_disjointly():
    from long_context_attention_seqattn_gb300 import dist
    for n in (1, 5, 8, 13):
        for world in (1, 2, 3, 8):
            ranges = [dist.shard_units(n, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [hi - lo for lo, hi in ranges]
            assert max(sizes) - min(sizes) <= 1


def test_two_rank_gloo_sharding_matches_single_process(tmp_path):
    import oracle
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    rng = np.random.default_rng(0)
    q = rng.standard_normal((5, 24, 2, 4))
    k = rng.standard_normal((5, 24, 1, 4))
    v = rng.standard_normal((5, 24, 1, 4))
    do = rng.standard_normal((5, 24, 2, 4))
    full = oracle.chunked_layer(q, k, v, do, 8, 0.5)
    for r in range(2):
        z = np.load(tmp_path / f"rank{r}.npz")
        lo, hi = int(z["lo"]), int(z["hi"])
        for i, ref in enumerate(full):
            np.testing.assert_array_equal(z[f"arr_{i}"], ref[lo:hi])
        red = np.load(tmp_path / f"red{r}.npy")
        assert red[0] == 2.0 and red[1] == 5.0

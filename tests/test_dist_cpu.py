"""The multi-rank path of bench.py on CPU with gloo (world size 2): each rank decodes its own
shard of the sequences (no collective on the data path) and only timings and byte counts are
reduced across ranks."""

import os
import socket
import sys
from pathlib import Path

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    sys.path[:0] = [str(ROOT), str(ROOT / "tests")]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import bench
    import oracle
    from paged_kv_cache_244_gb300 import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.make("tiny")
    part = W.shard(w, rank, world)
    orc = oracle.default()
    kc, vc = part.k_cache[0].copy(), part.v_cache[0].copy()
    q = orc.rope_kv_store(part.q[0], part.k[0], part.v[0], part.positions, part.cos_sin,
                          part.slot_mapping, kc, vc)
    out, _ = orc.decode(q, kc, vc, part.block_tables, part.context_lens, part.scale, nthreads=1)
    my_ms = 10.0 + rank            # stand-in timings: rank 1 is the slow one
    (t_max,), (b_sum, n_sum) = bench.reduce_over_ranks(
        [my_ms], [float(part.kv_bytes_per_layer()), float(part.num_seqs)], dist,
        torch.device("cpu"))
    np.save(Path(outdir) / f"out{rank}.npy", out)
    np.save(Path(outdir) / f"agg{rank}.npy", np.array([t_max, b_sum, n_sum]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_sequences_and_reduce_timings(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    sys.path[:0] = [str(ROOT)]
    import oracle
    from paged_kv_cache_244_gb300 import workloads as W
    w = W.make("tiny")
    for r in range(world):
        t_max, b_sum, n_sum = np.load(tmp_path / f"agg{r}.npy")
        assert t_max == 11.0                                  # max over ranks
        assert b_sum == w.kv_bytes_per_layer()                # bytes of all ranks
        assert n_sum == w.num_seqs                            # every sequence once
    # the shards together give exactly the single-process result
    orc = oracle.default()
    kc, vc = w.k_cache[0].copy(), w.v_cache[0].copy()
    q = orc.rope_kv_store(w.q[0], w.k[0], w.v[0], w.positions, w.cos_sin, w.slot_mapping, kc, vc)
    full, _ = orc.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
    got = np.concatenate([np.load(tmp_path / f"out{r}.npy") for r in range(world)])
    assert np.array_equal(got, full)

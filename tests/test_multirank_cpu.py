"""The multi-rank host logic of bench.py on CPU with a gloo process group (world size 2): each
rank gets its own sequences (distinct seeds, so distinct inputs) and the job's step time is the
slowest rank's. Decode shards by sequence, so no collective touches the data path."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from synth import generate_layer, get_config
        wl = get_config("csa_decode_128k")
        seed = bench.rank_seed(wl, rank)
        small = wl.layers[0].scaled(B=2, N=256, q_pos0=255, compress_begin=252)
        x = generate_layer(small, seed, 0, device="cpu")
        # every rank computes its own slice; gather only the fingerprints to compare them
        fp = torch.tensor([float(x["q"].float().sum()), float(x["ki_codes"].float().sum())],
                          dtype=torch.float64)
        fps = [torch.zeros_like(fp) for _ in range(world)]
        dist.all_gather(fps, fp)
        ms = bench.max_over_ranks(1.0 + rank, world, "cpu")
        out[rank] = (seed, [f.tolist() for f in fps], ms)
    finally:
        dist.destroy_process_group()


def test_two_rank_seeds_and_max_timing():
    world = 2
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    seeds = {res[r][0] for r in range(world)}
    assert len(seeds) == world                       # distinct sequences per rank
    fps = res[0][1]
    assert fps[0] != fps[1]                          # so distinct inputs
    assert all(res[r][2] == 2.0 for r in range(world))  # step time = slowest rank

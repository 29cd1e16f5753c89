"""The multi-process path on CPU: two gloo ranks, each running its shard of
a sequence-partitioned batch through a bookkeeping-only head (no GPU), with
no exchange on the data path. Every rank's page tables must match the
position-level simulator of its own pool, the shards must cover every
sequence once, and the job time is the slowest rank's (max reduction, as
bench.py reports it)."""
import os
import socket
import sys
from dataclasses import replace

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, n_seq, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from block_diffusion_speculative_forward_gb300 import binding as B
        from block_diffusion_speculative_forward_gb300 import synthetic as syn
        from tests.test_oracle_state import PositionSim
        from tests.test_oracle_pins import MICRO, cfg_of
        geom = replace(MICRO, gamma=8, ctx_window=64, kv_block=16, prefill_chunk=64)
        mine = bench.shard(n_seq, rank, world)
        lib = B.DraftHead(cfg_of(geom, max_batch=len(mine), max_seq_len=2048), None)
        sim = PositionSim(lib.debug_pool()[1], geom.kv_block, geom.ctx_window)
        ctx = syn.uniform_ints(20, 120, n_seq, 9, 1)
        states, ok = {}, True
        for i in mine:
            states[i] = lib.alloc_state()
            sim.new(i)
            lib.prefill(states[i], torch.empty((ctx[i], 8), dtype=torch.bfloat16))
            sim.step([i], [ctx[i]])
        pos, n_new = {i: ctx[i] for i in mine}, {i: 0 for i in mine}
        for rnd in range(6):
            pos = {i: pos[i] + n_new[i] for i in mine}
            rows = [torch.empty((n_new[i], 8), dtype=torch.bfloat16) if n_new[i] else None
                    for i in mine]
            res = lib.propose_batch([states[i] for i in mine], [1] * len(mine),
                                    [pos[i] for i in mine], rows, 7)
            ok &= res is not None
            sim.step(mine, [n_new[i] for i in mine])
            ks = syn.uniform_ints(0, 7, n_seq, 9, 100 + rnd)
            for i in mine:
                ok &= lib.debug_state(states[i]) == sim.table(i)
                lib.after_verify(states[i], ks[i])
                sim.verify(i, pos[i], ks[i])
                ok &= lib.debug_state(states[i]) == sim.table(i)
            n_new = {i: ks[i] + 1 for i in mine}
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine, bool(ok)))
        t = bench.max_over_ranks([1.0 + rank, 10.0 - rank], dist, "cpu")
        if rank == 0:
            q.put((gathered, t))
    finally:
        dist.destroy_process_group()


def test_two_rank_sequence_shards():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()
    world, n_seq = 2, 5
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n_seq, q)) for r in range(world)]
    for p in procs:
        p.start()
    gathered, t = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    covered = sorted(i for mine, _ in gathered for i in mine)
    assert covered == list(range(n_seq))
    assert all(ok for _, ok in gathered)
    assert t == [2.0, 10.0]

"""bench.py's multi-GPU host logic on CPU with two gloo ranks: disjoint per-rank sequences, the
max-over-ranks timing reduce, and the whole-job throughput (CPU only, no GPU)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    import synth

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.WORKLOADS["prefill32k_decode"].with_(T=4, decode_steps=0, Hk=1, Hv=2, dk=16, dv=16)
        inp = synth.make_inputs(wl, b0=bench.rank_batch_offset(rank, wl.B))
        ms = 1.0 + rank  # rank 1 is the slow one
        ms_max = bench.reduce_max(ms, world)
        val = bench.job_throughput(100, world, ms_max)
        out[rank] = (ms_max, val, float(inp.v[0, 0, 0, 0]), float(inp.v[-1, -1, -1, -1]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 2.0                     # the max over ranks
    assert out[0][1] == pytest.approx(2 * 100 / 2e-3)        # all ranks' tokens over the slowest time
    assert out[0][2] != out[1][2] and out[0][3] != out[1][3]  # ranks hold different sequences


def test_rank_offsets_match_a_single_large_batch():
    import bench
    import synth

    wl = synth.WORKLOADS["prefill32k_decode"].with_(T=3, decode_steps=0, Hk=1, Hv=2, dk=16, dv=16)
    whole = synth.make_inputs(wl.with_(B=4))
    for r in range(2):
        part = synth.make_inputs(wl, b0=bench.rank_batch_offset(r, wl.B))
        assert np.array_equal(part.v, whole.v[2 * r:2 * r + 2])
        assert np.array_equal(part.q, whole.q[2 * r:2 * r + 2])
    assert bench.reduce_max(3.5, 1) == 3.5

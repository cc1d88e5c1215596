"""Multi-process (N > 1) host logic on CPU ranks with the gloo backend.

The hot path shards with no exchange: every rank owns its own pool and
requests (replicas).  What the N > 1 benchmark adds is host logic: the slowest
rank's time (max over ranks), the whole-job rate, and the reference arm that
only rank 0 runs.  These run here as two gloo ranks, no GPU involved.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from hybrid_linear_attention_gdn_gb300 import synth
        # each rank: its own pool and requests (replica), a few oracle decode steps
        shape = synth.TINY
        g = synth.generator(100 + rank)
        conv_w, A_log, dt_bias = synth.params(shape, g)
        ssm, conv = synth.pool(shape, g)
        od = oracle.Dims(shape.hk, shape.hv, shape.dk, shape.dv, shape.w)
        op = oracle.Params(conv_w.double().numpy(), A_log.double().numpy(), dt_bias.double().numpy())
        pool = oracle.Pool(ssm.double().numpy(), conv.double().numpy())
        ids = synth.slot_ids(8, 4, g).numpy()
        outs = []
        for _ in range(3):
            qkv, a, b = (t.double().numpy() for t in synth.tokens(shape, g, (4,)))
            o, err = oracle.decode_step(od, pool, op, ids, qkv, a, b)
            outs.append(o)
        local_ms = 10.0 + 5.0 * rank          # a stand-in elapsed time per rank
        ms = bench.reduce_max(local_ms)
        rate = bench.whole_job_rate(4 * 3, world, ms)
        dist.barrier()
        q.put((rank, ms, rate, float(np.abs(np.stack(outs)).sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    # both ranks see the slowest rank's time; the rate counts both ranks' work
    assert res[0][1] == res[1][1] == 15.0
    assert res[0][2] == pytest.approx(2 * 12 / 15e-3)
    # replicas: different seeds, different (finite, non-zero) results
    assert res[0][3] != res[1][3] and all(np.isfinite(r[3]) and r[3] > 0 for r in res)


def _reference_rank(rank, world, port, q):
    import contextlib
    import io
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    class A:
        steps, warmup = 1, 1

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(A)
    q.put((rank, buf.getvalue()))


def test_reference_arm_runs_on_rank_zero_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_reference_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import json
    line = json.loads(res[0][1].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert res[1][1] == ""

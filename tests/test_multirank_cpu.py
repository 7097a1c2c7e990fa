"""The multi-process path, on CPU with gloo (world size 2).

Routing is independent per token (attention over depth, not over tokens), so
a data-parallel job shards tokens across ranks with no exchange inside the
path; only dq/dg, being sums over tokens, need a sum across ranks (the
training framework's gradient all-reduce). Checked here with the oracle:
sharded forward/backward + all-reduce(sum) of dq/dg equals the unsharded run.
Also checks the benchmark's max-over-ranks timing reduction.
"""

import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    import torch
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        import synth
        T, d, H, N = 96, 64, 4, 5
        srcs = [synth.misc_normal(3, 200 + n, (T, d)).astype(np.float64) for n in range(N)]
        qv = synth.misc_normal(3, 1, (d,), 0.5).astype(np.float64)
        gv = 1.0 + synth.misc_normal(3, 2, (d,), 0.1).astype(np.float64)
        G = synth.misc_normal(3, 3, (T, d)).astype(np.float64)
        lo, hi = rank * T // world, (rank + 1) * T // world
        out, lse = oracle.route_fwd([s[lo:hi] for s in srcs], qv, gv, H)
        ds, dq, dg = oracle.route_bwd([s[lo:hi] for s in srcs], qv, gv, G[lo:hi], H)
        t = torch.tensor(np.concatenate([dq, dg]))
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        parts = [None] * world
        dist.all_gather_object(parts, (lo, hi, out, lse, ds))
        timing = bench.max_over_ranks([1.0 + rank, 5.0 - rank])
        q.put((rank, t.numpy(), parts, timing))
    finally:
        dist.destroy_process_group()


def test_token_sharded_routing_matches_unsharded():
    import oracle
    import synth
    oracle.build()
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    T, d, H, N = 96, 64, 4, 5
    srcs = [synth.misc_normal(3, 200 + n, (T, d)).astype(np.float64) for n in range(N)]
    qv = synth.misc_normal(3, 1, (d,), 0.5).astype(np.float64)
    gv = 1.0 + synth.misc_normal(3, 2, (d,), 0.1).astype(np.float64)
    G = synth.misc_normal(3, 3, (T, d)).astype(np.float64)
    out, lse = oracle.route_fwd(srcs, qv, gv, H)
    ds, dq, dg = oracle.route_bwd(srcs, qv, gv, G, H)
    for rank, red, parts, timing in res:
        assert np.allclose(red[:d], dq, rtol=1e-12, atol=1e-12)
        assert np.allclose(red[d:], dg, rtol=1e-12, atol=1e-12)
        assert timing == [2.0, 5.0]
        for lo, hi, o, l, dsh in parts:
            assert np.array_equal(o, out[lo:hi]) and np.array_equal(l, lse[lo:hi])
            for n in range(N):
                assert np.array_equal(dsh[n], ds[n][lo:hi])


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the oracle's benchmark runs on rank 0 alone: another rank
    exits 0 at once and prints nothing."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], cwd=root, capture_output=True, text=True,
                       timeout=120, env={**os.environ, "RANK": "1", "WORLD_SIZE": "2"})
    assert p.returncode == 0 and p.stdout == ""

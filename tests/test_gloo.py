"""Two-rank tests of the multi-process paths, on CPU with the gloo backend.

  * the bench's rank helpers: max-over-ranks timing, per-rank seeds (each rank
    its own batch: weak scaling) and the whole-job throughput;
  * the channel-sharded proj_rms_compute_h protocol (RL-Kernel PR #383 task
    P1-6, the fp32_gemm_rms TP/SP contract): each rank owns half of the
    channels of every stream, computes its partial sums, an all-reduce sums
    them, compute_h runs on the totals, and each rank forms dx and dW for its
    own channels.  Rank 0 checks the result against the unsharded oracle.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(fn, world=2):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(fn, r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    results = [q.get(timeout=5) for _ in procs]
    for p in procs:
        assert p.exitcode == 0, f"rank exited with {p.exitcode}"
    errs = [r for r in results if r[1] is not None]
    assert not errs, errs


def _worker(fn, rank, world, port, q):
    err = None
    try:
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                world_size=world)
        fn(rank, world)
        dist.barrier()
    except Exception as e:  # reported to the parent
        import traceback
        err = traceback.format_exc() + repr(e)
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()
        q.put((rank, err))


def _bench_helpers(rank, world):
    import bench
    t = bench.max_over_ranks(1.5 + rank, world, "cpu")
    assert t == 1.5 + world - 1
    assert bench.rank_seed(3, rank) == 3 + 1000 * rank
    assert bench.job_tokens_per_s(1000, world, 2.0) == 1000 * world / 2e-3


def test_bench_rank_helpers_gloo():
    _run(_bench_helpers)


def _sharded_proj(rank, world):
    import oracle as orc
    g = np.random.Generator(np.random.PCG64(7))
    T, n, C = 4, 4, 16
    O = n * n + 2 * n
    K = n * C
    x = g.standard_normal((T, n, C)); W = 0.3 * g.standard_normal((K, O))
    alpha = np.array([0.7, 1.1, 0.9]); b = 0.5 * g.standard_normal(O)
    dHp = g.standard_normal((T, n)); dHq = g.standard_normal((T, n)); dHr = g.standard_normal((T, n, n))
    iters, eps_sk, eps_rms = 20, 1e-6, 1e-6
    Cs = C // world
    c0, c1 = rank * Cs, (rank + 1) * Cs
    xs = np.ascontiguousarray(x[:, :, c0:c1])
    Ws = np.concatenate([W[i * C + c0:i * C + c1] for i in range(n)], axis=0)
    p = orc.proj_rms_partials(xs, Ws)
    tot = torch.tensor(np.concatenate([p["u"].ravel(), p["s"]]))
    dist.all_reduce(tot, op=dist.ReduceOp.SUM)
    tot = tot.numpy()
    u, s = tot[:T * O].reshape(T, O), tot[T * O:]
    h = orc.compute_h_from_sums(u, s, K, alpha, b, n, iters, eps_sk, eps_rms)
    cb = orc.compute_h_bwd_from_sums(dHp, dHq, dHr, u, s, K, alpha, b, n, iters, eps_sk, eps_rms)
    pb = orc.proj_rms_partial_bwd(xs, Ws, cb["du"], cb["coef"])
    parts = [torch.zeros(T * n * Cs, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(parts, torch.tensor(pb["dx"].ravel()))
    if rank == 0:
        ref = orc.proj_rms_compute_h_fwd(x, W, alpha, b, n, iters, eps_sk, eps_rms)
        for k in ("H_pre", "H_post", "H_res"):
            np.testing.assert_allclose(h[k], ref[k], rtol=1e-12, atol=1e-13)
        rb = orc.proj_rms_compute_h_bwd(dHp, dHq, dHr, x, W, alpha, b, n, iters, eps_sk, eps_rms)
        dx = np.concatenate([q.numpy().reshape(T, n, Cs) for q in parts], axis=2)
        np.testing.assert_allclose(dx.reshape(T, -1), rb["dx"].reshape(T, -1), rtol=1e-10,
                                   atol=1e-12)
        np.testing.assert_allclose(cb["dalpha"], rb["dalpha"], rtol=1e-11, atol=1e-12)


def test_sharded_proj_rms_gloo():
    _run(_sharded_proj)

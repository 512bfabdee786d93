"""Multi-process checks on CPU (gloo, world size 2).

1. The distributed form of one CA-SGD outer iteration -- features split across
   processes, one sum of the partial Gram matrix and margins per outer iteration, the
   recurrence repeated on every rank, each rank updating its own slice of w -- equals
   the single-process oracle.  This is the exchange the paper's abstract describes (one
   AllReduce of an sb x sb Gram replacing s per-step AllReduces); it is exercised here
   with the oracle only, on the host.
2. The bench's multi-rank reduction (max of per-rank times) over gloo.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth_inputs as si


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _sharded_step(rank, world, port, out_q, kind):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = si.make_random(400, 23, kind, seed=5)
        b, s, eta, seed, k = 6, 4, 0.2, 3, 2
        S = b * s
        w0 = si.random_weights(23, seed=9, scale=0.3).astype(np.float64)
        cols = np.array_split(np.arange(23), world)[rank]
        idx = oracle.sample_indices(p.m, S, seed, k * S)        # same rows on every rank
        Yr = p.X[idx][:, cols].astype(np.float64)
        G = torch.from_numpy(Yr @ Yr.T)                          # partial Gram
        r = torch.from_numpy(Yr @ w0[cols])                      # partial margins
        dist.all_reduce(G)                                       # the one exchange
        dist.all_reduce(r)
        G, r = G.numpy(), r.numpy()
        yY = p.y[idx].astype(np.float64)
        alpha = np.zeros(S)
        for j in range(s):                                       # redundant recurrence
            rows = slice(j * b, (j + 1) * b)
            z = r[rows] + G[rows, : j * b] @ alpha[: j * b]
            alpha[rows] = -(eta / b) * oracle.loss_grad(z, yY[rows], kind)
        w_local = w0[cols] + Yr.T @ alpha
        out_q.put((rank, cols, w_local))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("kind", [si.LOGISTIC, si.POISSON])
def test_feature_sharded_outer_step_equals_single_process(kind):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sharded_step, args=(r, 2, port, q, kind)) for r in range(2)]
    for pr in procs:
        pr.start()
    parts = [q.get(timeout=120) for _ in range(2)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    w = np.zeros(23)
    for _, cols, wl in parts:
        w[cols] = wl
    p = si.make_random(400, 23, kind, seed=5)
    w0 = si.random_weights(23, seed=9, scale=0.3).astype(np.float64)
    ref = oracle.outer_step(p.X, p.y, w0, 6, 4, 0.2, kind, 3, 2, mode="fp64")
    assert np.linalg.norm(w - ref) <= 1e-12 * np.linalg.norm(ref)


def _exchange_hook(rank, world, port, out_q):
    """The library's exchange hook (make_exchange), as casgd_train_sharded calls it once
    per outer iteration, summing a rank's buffer over a gloo group in place."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import communication_avoiding_step_gb300 as casgd
        xbuf = torch.arange(10, dtype=torch.float32) * (rank + 1)
        hook = casgd.make_exchange(xbuf, dist.all_reduce)
        rc_ok = hook(None, xbuf.data_ptr(), 7, None)            # sums the first 7 floats
        rc_bad_ptr = hook(None, xbuf.data_ptr() + 4, 7, None)   # not the buffer: refused
        rc_bad_len = hook(None, xbuf.data_ptr(), 11, None)      # longer than the buffer

        def failing(t):
            raise RuntimeError("peer lost")

        rc_fail = casgd.make_exchange(xbuf, failing)(None, xbuf.data_ptr(), 7, None)
        out_q.put((rank, rc_ok, rc_bad_ptr, rc_bad_len, rc_fail, xbuf.numpy().copy()))
    finally:
        dist.destroy_process_group()


def test_exchange_hook_sums_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_exchange_hook, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    got = {v[0]: v[1:] for v in (q.get(timeout=120) for _ in range(2))}
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    for rank, (rc_ok, rc_bad_ptr, rc_bad_len, rc_fail, buf) in got.items():
        assert (rc_ok, rc_bad_ptr, rc_bad_len, rc_fail) == (0, 1, 1, 1)
        want = np.arange(10, dtype=np.float32) * (rank + 1)
        want[:7] = np.arange(7, dtype=np.float32) * 3          # 1x + 2x over the two ranks
        assert np.array_equal(buf, want)


def _bench_reduce(rank, world, port, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t = bench.world_max(1.5 + rank, torch.device("cpu"))
        out_q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_bench_world_max_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bench_reduce, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    got = dict(q.get(timeout=120) for _ in range(2))
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    assert got == {0: 2.5, 1: 2.5}

"""Feature-sharded CA-SGD (the paper's distributed setting) through the C ABI, on one GPU.

The features are split into column shards, each with its own BF16 matrix, weight slice,
workspace and exchange buffer.  casgd_outer_step_local runs on every shard; the exchange
buffers are then summed (here with a torch add on the device: the sum over processes an
ncclAllReduce would perform) and casgd_outer_step_finish runs on every shard.  The
concatenated weights must match the oracle's unsharded outer iteration at the bars of
the other parity tests: G within 1e-5 relative Frobenius, margins within one BF16 ulp on
at most 0.5% of entries, w within 1e-4 relative L2.  casgd_train_sharded is driven by
two host threads (one per shard) whose exchange hooks meet at a barrier and sum the
buffers; both threads enqueue on one stream, so no two kernels run at the same time.
"""
import threading

import numpy as np
import pytest

import oracle
import synth_inputs as si

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

G_TOL, W_TOL, FLIP_FRAC = 1e-5, 1e-4, 0.005


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _shards(casgd, p, cuts):
    """Column shards [c0, c1) of the problem as device datasets (full labels each)."""
    X32 = torch.from_numpy(p.X).cuda()
    y = torch.from_numpy(p.y).cuda()
    out = []
    for c0, c1 in zip(cuts[:-1], cuts[1:]):
        out.append((c0, c1, casgd.Dataset.from_fp32(X32[:, c0:c1].contiguous(), y)))
    return out


CASES = [
    # name, problem, (b, s, eta) or None for the recipe's, column cuts
    ("recipe5_m20000", lambda: si.make_problem(5, m=20000), None, [0, 200, 512]),
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), None, [0, 1000, 2000]),
    ("ragged_3000x130_b100_s6_3way", lambda: si.make_random(3000, 130, si.LOGISTIC, seed=3),
     (100, 6, 0.3), [0, 37, 90, 130]),
    ("narrow_n18_b256_s8", lambda: si.make_problem(3, m=60000), (256, 8, 0.05), [0, 9, 18]),
]


@pytest.mark.parametrize("name,factory,override,cuts", CASES, ids=[c[0] for c in CASES])
def test_sharded_outer_step_matches_oracle(gpu_lib, name, factory, override, cuts):
    casgd = gpu_lib
    p = factory()
    r = p.recipe
    b, s, eta = override if override else (r.b, r.s, r.eta)
    kind = r.loss
    params = casgd.Params(b, s, eta, kind, seed=0)
    S = b * s
    shards = _shards(casgd, p, cuts)
    w0 = si.random_weights(p.n, seed=11, scale=0.3)
    k = 1
    xb, ws, ws_w, taps = [], [], [], []
    for c0, c1, d in shards:
        ws.append(casgd.workspace_sharded(d, params))
        xb.append(casgd.exchange_buffer(params))
        ws_w.append(torch.from_numpy(w0[c0:c1].copy()).cuda())
        taps.append(casgd.Taps(idx_out=torch.empty(S, dtype=torch.int32, device="cuda"),
                               r_out=torch.empty(S, dtype=torch.int16, device="cuda"),
                               alpha_out=torch.empty(S, dtype=torch.float32, device="cuda")))
    for i, (_, _, d) in enumerate(shards):
        casgd.outer_step_local(d, params, ws_w[i], k, ws[i], xb[i], taps[i])
    total = torch.stack(xb).sum(0)              # the sum over processes
    for i in range(len(shards)):
        xb[i].copy_(total)
    for i, (_, _, d) in enumerate(shards):
        casgd.outer_step_finish(d, params, ws_w[i], ws[i], xb[i], taps[i])
    for i in range(len(shards)):
        assert casgd.get_status(ws[i]) == 0
    want = oracle.outer_step(p.X, p.y, w0, b, s, eta, kind, 0, k, mode="emulate",
                             return_parts=True)
    # every shard drew the same rows, equal to the oracle's
    for t in taps:
        assert np.array_equal(t.idx_out.cpu().numpy(), want["idx"].astype(np.int32))
    # the summed G against the oracle's packed block-lower Gram
    ge = casgd.gram_elems(b, s)
    G = total[:ge].cpu().numpy()
    Gref = oracle.gram_packed(want["Y"], b, s)
    assert _rel(G, Gref) <= G_TOL
    # the summed margins, rounded once: at most one BF16 ulp apart, on few entries
    rb = taps[0].r_out.cpu().numpy().astype(np.uint16).astype(np.uint32) << 16
    r_gpu = rb.view(np.float32)
    r_ref = np.asarray(want["r"], np.float32)
    diff = r_gpu != r_ref
    if diff.any():
        ulp = np.abs(r_ref[diff]) * 2.0 ** -7
        assert np.all(np.abs(r_gpu[diff] - r_ref[diff]) <= ulp * 1.0001 + 1e-30)
    assert diff.mean() <= FLIP_FRAC
    # alpha identical on every shard (the same recurrence on the same sums)
    a0 = taps[0].alpha_out.cpu().numpy()
    for t in taps[1:]:
        assert np.array_equal(t.alpha_out.cpu().numpy().view(np.uint32), a0.view(np.uint32))
    w = np.concatenate([x.cpu().numpy() for x in ws_w])
    assert _rel(w, want["w"]) <= W_TOL


def test_sharded_one_process_equals_full_g_outer_steps(gpu_lib):
    """With one process the exchange is the identity: train_sharded over three
    iterations stays within FP32 summation order of casgd_outer_step with FULL_G."""
    casgd = gpu_lib
    p = si.make_problem(5, m=20000)
    r = p.recipe
    d = casgd.Dataset.from_fp32(torch.from_numpy(p.X).cuda(), torch.from_numpy(p.y).cuda())
    params = casgd.Params(r.b, r.s, r.eta, r.loss, seed=4)
    ws = casgd.workspace_sharded(d, params)
    xbuf = casgd.exchange_buffer(params)
    w = torch.zeros(p.n, device="cuda")
    launches, kind = casgd.train_sharded(d, params, w, 3, ws, xbuf, None, k0=2)
    assert kind == 7 and launches >= 3 * 4
    pf = casgd.Params(r.b, r.s, r.eta, r.loss, seed=4, flags=casgd.FLAG_FULL_G)
    wsf = casgd.workspace(d, pf)
    wf = torch.zeros(p.n, device="cuda")
    for k in range(2, 5):
        casgd.outer_step(d, pf, wf, k, wsf)
    assert casgd.get_status(wsf) == 0
    assert _rel(w.cpu().numpy(), wf.cpu().numpy()) <= 1e-5


def test_train_sharded_two_threads_match_oracle(gpu_lib):
    """Two shards driven by two host threads through casgd_train_sharded: each thread's
    exchange hook waits at a barrier, one thread sums both buffers (after a device
    synchronize) and writes the sum into both, then both continue.  Both threads enqueue
    on the same stream, so kernels never run concurrently."""
    casgd = gpu_lib
    p = si.make_problem(5, m=20000)
    r = p.recipe
    params = casgd.Params(r.b, r.s, r.eta, r.loss, seed=0)
    shards = _shards(casgd, p, [0, 300, 512])
    xb = [casgd.exchange_buffer(params) for _ in shards]
    ws = [casgd.workspace_sharded(d, params) for _, _, d in shards]
    w = [torch.zeros(c1 - c0, device="cuda") for c0, c1, _ in shards]
    stream = torch.cuda.current_stream()
    barrier = threading.Barrier(2)
    iters = 3

    def make_sum(i):
        def all_reduce(t):
            barrier.wait(timeout=60)
            if i == 0:
                torch.cuda.synchronize()
                tot = xb[0] + xb[1]
                xb[0].copy_(tot)
                xb[1].copy_(tot)
                torch.cuda.synchronize()
            barrier.wait(timeout=60)
        return all_reduce

    errs = []

    def run(i):
        try:
            d = shards[i][2]
            casgd.train_sharded(d, params, w[i], iters, ws[i], xb[i], make_sum(i), k0=0,
                                stream=stream)
        except Exception as e:  # noqa: BLE001
            errs.append(e)
            barrier.abort()

    th = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join(timeout=300)
    assert not errs, errs
    got = np.concatenate([x.cpu().numpy() for x in w])
    want, _ = oracle.train(p.X, p.y, r.b, r.s, r.eta, r.loss, 0, iters, mode="emulate")
    assert _rel(got, want) <= W_TOL


def test_sharded_unsupported_flags_and_failed_exchange(gpu_lib):
    casgd = gpu_lib
    p = si.make_random(3000, 130, si.LOGISTIC, seed=3)
    d = casgd.Dataset.from_fp32(torch.from_numpy(p.X).cuda(), torch.from_numpy(p.y).cuda())
    for flags in (casgd.FLAG_FAR_FROM_GRAM, casgd.FLAG_G_BF16):
        params = casgd.Params(256, 4, 0.1, si.LOGISTIC, flags=flags)
        with pytest.raises(casgd.CasgdError) as e:
            casgd.workspace_sharded(d, params)
        assert e.value.code == 7
    params = casgd.Params(256, 4, 0.1, si.LOGISTIC)
    ws = casgd.workspace_sharded(d, params)
    xbuf = casgd.exchange_buffer(params)
    w = torch.zeros(p.n, device="cuda")

    def broken(t):
        raise RuntimeError("peer lost")

    with pytest.raises(casgd.CasgdError) as e:
        casgd.train_sharded(d, params, w, 2, ws, xbuf, broken)
    assert e.value.code == 9                      # CASGD_ERR_EXCHANGE
    torch.cuda.synchronize()
    # the loop stopped before finish: w was not touched
    assert torch.count_nonzero(w).item() == 0
    assert casgd.get_status(ws) == 0

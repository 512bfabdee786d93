"""casgd_update_static: the weight update w += Y^T alpha for callers that cannot
allocate device memory where they apply it (code inside another framework's memory
pool that forbids raw cudaMalloc, loops that must not block on an allocator, or
embedders that own only their input and output buffers).  Its scratch is a fixed array
inside the library, shared by every call.

Checked three ways, each on two calls in a row (so the second call runs on the scratch
the first one left behind):
  * against the regular casgd_outer_step's update (the same alpha and rows);
  * against the oracle's FP32 update Y^T alpha on the oracle's own rows and alpha;
  * requests larger than the scratch are refused before anything runs, with real
    device buffers.
This file is collected last on purpose: a run that stops at the first failure has then
already run every other test.
"""
import numpy as np
import pytest

import oracle
import synth_inputs as si

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

W_TOL = 1e-4


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


@pytest.mark.parametrize("cid,m", [(5, 20000), (2, 20000)])
def test_update_static_matches_outer_step(gpu_lib, cid, m):
    casgd = gpu_lib
    p = si.make_problem(cid, m=m)
    r = p.recipe
    data = casgd.Dataset.from_fp32(torch.from_numpy(p.X).cuda(), torch.from_numpy(p.y).cuda())
    params = casgd.Params(r.b, r.s, r.eta, r.loss)
    ws = casgd.workspace(data, params)
    w_start = torch.from_numpy(si.random_weights(p.n, seed=3, scale=0.2)).cuda()
    for k in range(2):                        # two calls in a row
        taps = casgd.Taps.alloc(params, G=False)
        w_ref = w_start.clone()
        casgd.outer_step(data, params, w_ref, k, ws, taps)
        assert casgd.get_status(ws) == 0
        Y = data.X[taps.idx_out.long()].contiguous()     # the gathered BF16 rows
        w_static = w_start.clone()
        casgd.update_static(Y, taps.alpha_out, w_static, p.n)
        torch.cuda.synchronize()
        got, want = w_static.cpu().numpy(), w_ref.cpu().numpy()
        assert _rel(got, want) <= W_TOL
        w_start = w_ref


@pytest.mark.parametrize("cid,m", [(5, 20000), (1, 4096)])
def test_update_static_matches_oracle(gpu_lib, cid, m):
    """The oracle's emulating-mode outer iteration gives Y (BF16 values), alpha and
    w = w0 + Y^T alpha in FP32; the allocation-free update applied to the same Y, alpha
    and w0 must land within the w bar of the parity tests."""
    casgd = gpu_lib
    p = si.make_problem(cid, m=m)
    r = p.recipe
    w0 = si.random_weights(p.n, seed=5, scale=0.2)
    for k in range(2):                        # two calls in a row
        parts = oracle.outer_step(p.X, p.y, w0, r.b, r.s, r.eta, r.loss, 0, k,
                                  mode="emulate", return_parts=True)
        ld = (p.n + 7) // 8 * 8
        Yh = np.zeros((parts["Y"].shape[0], ld), np.float32)
        Yh[:, :p.n] = parts["Y"]                          # BF16 values: exact in BF16
        Y = torch.from_numpy(Yh).to(torch.bfloat16).cuda()
        alpha = torch.from_numpy(np.asarray(parts["alpha"], np.float32)).cuda()
        w = torch.from_numpy(w0.copy()).cuda()
        casgd.update_static(Y, alpha, w, p.n)
        torch.cuda.synchronize()
        assert _rel(w.cpu().numpy(), parts["w"]) <= W_TOL
        w0 = np.asarray(parts["w"], np.float32)


def test_update_static_rejects_oversized_requests(gpu_lib):
    """P * ldY > 1,048,576 partial floats (P = min(ceil(S/32), 320)) is refused with
    CASGD_ERR_SCRATCH_LIMIT and w stays as it was.  Real device buffers of the stated
    sizes are passed, so nothing would read past them even if a check moved."""
    casgd = gpu_lib
    S, ld = 320 * 32, 3280                    # P = 320: 320 * 3280 = 1,049,600 floats
    Y = torch.zeros((S, ld), dtype=torch.bfloat16, device="cuda")
    alpha = torch.ones(S, dtype=torch.float32, device="cuda")
    w = torch.full((ld,), 2.0, dtype=torch.float32, device="cuda")
    with pytest.raises(casgd.CasgdError) as e:
        casgd.update_static(Y, alpha, w, ld)
    assert e.value.code == 8                  # CASGD_ERR_SCRATCH_LIMIT
    assert b"fixed scratch" in casgd.load().casgd_strerror(8)
    torch.cuda.synchronize()
    assert torch.all(w == 2.0).item()
    # one column less fits: P * ldY = 320 * 3272 <= 1,048,576
    Y2 = torch.zeros((S, 3272), dtype=torch.bfloat16, device="cuda")
    w2 = torch.full((3272,), 2.0, dtype=torch.float32, device="cuda")
    casgd.update_static(Y2, alpha, w2, 3272)  # Y = 0: w unchanged, and no error
    torch.cuda.synchronize()
    assert torch.all(w2 == 2.0).item()

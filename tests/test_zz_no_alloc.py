"""casgd_update_static: the allocation-free weight update, checked against the regular
outer iteration's update.

Some callers cannot allocate device memory where they apply an update, so this entry
point keeps its scratch in a fixed array inside the library.  The test runs the
regular casgd_outer_step (which uses a caller workspace), rebuilds the gathered rows Y
from its sampled indices, applies casgd_update_static to the starting weights with the
same alpha, and compares the results -- on two calls in a row, so the second call runs
on scratch the first one left behind.  This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest

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


def test_update_static_rejects_oversized_requests(gpu_lib):
    casgd = gpu_lib
    lib = casgd.load()
    fake = C.c_void_p(1 << 20)          # never touched: the size check comes first
    rc = lib.casgd_update_static(fake, 65536, 16384, 16384, fake, fake, None)
    assert rc == 8                      # CASGD_ERR_SCRATCH_LIMIT
    assert b"fixed scratch" in lib.casgd_strerror(8)
    rc = lib.casgd_update_static(fake, 65536, 3280, 3280, fake, fake, None)
    assert rc == 8

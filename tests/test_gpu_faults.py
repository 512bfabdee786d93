"""Boundary checks and device-side failure reporting on the GPU.

Failures are made on the host side only: bad arguments, out-of-range indices, and a
test flag that keeps one producer from signalling so that every waiter of the
recurrence runs into its (short) time bound.  No test faults, traps or hangs the GPU;
each checks that the error comes back as a status code and that the context stays
usable afterwards.
"""
import numpy as np
import pytest

import synth_inputs as si

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _data(casgd, cid=1, m=None):
    p = si.make_problem(cid, m=m)
    return p, casgd.Dataset.from_fp32(torch.from_numpy(p.X).cuda(), torch.from_numpy(p.y).cuda())


def test_workspace_too_small_launches_nothing(gpu_lib):
    casgd = gpu_lib
    p, data = _data(casgd)
    params = casgd.Params(16, 4, 0.1, si.LOGISTIC)
    ws = casgd.workspace(data, params)
    w = torch.zeros(p.n, device="cuda")
    small = ws[: ws.numel() - 256]
    with pytest.raises(casgd.CasgdError) as e:
        casgd.outer_step(data, params, w, 0, small)
    assert e.value.code == 2
    with pytest.raises(casgd.CasgdError) as e:
        casgd.outer_step(data, params, w, 0, ws[8:])       # misaligned
    assert e.value.code == 2
    torch.cuda.synchronize()
    assert torch.count_nonzero(w).item() == 0
    assert casgd.get_status(ws) == 0


def test_stalled_producer_times_out_and_context_survives(gpu_lib):
    casgd = gpu_lib
    p, data = _data(casgd)
    stall = casgd.Params(16, 4, 0.1, si.LOGISTIC, flags=casgd.FLAG_TEST_STALL, timeout_us=20000)
    ws = casgd.workspace(data, stall)
    w = torch.zeros(p.n, device="cuda")
    casgd.outer_step(data, stall, w, 0, ws)
    assert casgd.get_status(ws) == 5                     # CASGD_ERR_TIMEOUT
    assert casgd.get_status(ws) == 0                     # cleared
    ok = casgd.Params(16, 4, 0.1, si.LOGISTIC)
    w.zero_()
    casgd.outer_step(data, ok, w, 0, ws)
    assert casgd.get_status(ws) == 0
    assert torch.isfinite(w).all() and torch.count_nonzero(w).item() > 0


def test_stall_in_fused_launch_times_out_and_context_survives(gpu_lib):
    """The paired-SM Gram storing G with the recurrence in the same launch (recipe 2
    shape): the Gram warps finish their tiles, every recurrence waiter runs into its
    bound."""
    casgd = gpu_lib
    p, data = _data(casgd, cid=2, m=20000)
    r = p.recipe
    full = casgd.FLAG_FULL_G
    stall = casgd.Params(r.b, r.s, r.eta, r.loss, flags=full | casgd.FLAG_TEST_STALL,
                         timeout_us=20000)
    ws = casgd.workspace(data, stall)
    w = torch.zeros(p.n, device="cuda")
    _, _, kind = casgd.train(data, casgd.Params(r.b, r.s, r.eta, r.loss, flags=full), w, 1, ws)
    assert kind == 3                                     # the fused launch ran
    casgd.outer_step(data, stall, w, 0, ws)
    assert casgd.get_status(ws) == 5                     # CASGD_ERR_TIMEOUT
    assert casgd.get_status(ws) == 0
    w.zero_()
    casgd.outer_step(data, casgd.Params(r.b, r.s, r.eta, r.loss, flags=full), w, 0, ws)
    assert casgd.get_status(ws) == 0
    assert torch.isfinite(w).all() and torch.count_nonzero(w).item() > 0


def test_stall_in_pipelined_train_times_out(gpu_lib):
    """casgd_train with the next Gram in the recurrence's launch: a stalled recurrence
    ends the run with CASGD_ERR_TIMEOUT; the workspace works again afterwards."""
    casgd = gpu_lib
    p, data = _data(casgd, cid=2, m=20000)
    r = p.recipe
    full = casgd.FLAG_FULL_G
    stall = casgd.Params(r.b, r.s, r.eta, r.loss, flags=full | casgd.FLAG_TEST_STALL,
                         timeout_us=20000)
    ws = casgd.workspace(data, stall)
    w = torch.zeros(p.n, device="cuda")
    with pytest.raises(casgd.CasgdError) as e:
        casgd.train(data, stall, w, 3, ws)
    assert e.value.code == 5
    w.zero_()
    _, _, kind = casgd.train(data, casgd.Params(r.b, r.s, r.eta, r.loss, flags=full), w, 2, ws)
    assert kind == 4
    assert torch.isfinite(w).all() and torch.count_nonzero(w).item() > 0


def test_stall_in_far_forming_launch_times_out(gpu_lib):
    """CASGD_FLAG_FAR_FROM_GRAM: the Gram's epilogue waits on alpha itself.  With alpha_0
    never stored, those waits and the recurrence's run into their bound; the Gram warps
    still drain every tile, and the workspace works again afterwards."""
    casgd = gpu_lib
    p, data = _data(casgd, cid=2, m=20000)
    r = p.recipe
    far = casgd.FLAG_FAR_FROM_GRAM
    stall = casgd.Params(r.b, r.s, r.eta, r.loss, flags=far | casgd.FLAG_TEST_STALL,
                         timeout_us=20000)
    ws = casgd.workspace(data, stall)
    w = torch.zeros(p.n, device="cuda")
    casgd.outer_step(data, stall, w, 0, ws)
    assert casgd.get_status(ws) == 5                     # CASGD_ERR_TIMEOUT
    assert casgd.get_status(ws) == 0
    with pytest.raises(casgd.CasgdError) as e:
        casgd.train(data, stall, w, 3, ws)
    assert e.value.code == 5
    w.zero_()
    ok = casgd.Params(r.b, r.s, r.eta, r.loss, flags=far)
    _, _, kind = casgd.train(data, ok, w, 2, ws)
    assert kind == 6
    assert torch.isfinite(w).all() and torch.count_nonzero(w).item() > 0


def test_nonfinite_weights_reported(gpu_lib):
    casgd = gpu_lib
    p, data = _data(casgd, cid=5, m=5000)
    params = casgd.Params(64, 2, 1e30, si.POISSON)
    ws = casgd.workspace(data, params)
    w = torch.full((p.n,), 50.0, device="cuda")
    casgd.outer_step(data, params, w, 0, ws)
    assert casgd.get_status(ws) == 4                     # CASGD_ERR_NONFINITE


def test_train_returns_sticky_status(gpu_lib):
    casgd = gpu_lib
    p, data = _data(casgd)
    stall = casgd.Params(16, 4, 0.1, si.LOGISTIC, flags=casgd.FLAG_TEST_STALL, timeout_us=10000)
    ws = casgd.workspace(data, stall)
    w = torch.zeros(p.n, device="cuda")
    with pytest.raises(casgd.CasgdError) as e:
        casgd.train(data, stall, w, 2, ws)
    assert e.value.code == 5

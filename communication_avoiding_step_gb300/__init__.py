"""GB300-native mixed-precision communication-avoiding SGD (CA-SGD) for GLMs.

Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
GPUs (abstract).  Every step of the outer iteration runs in the CUDA kernels of
libcasgd.so (sm_103a); this module only marshals PyTorch tensors into the C ABI of
include/casgd.h.  There is no CPU fallback: if the library is missing, `load()` and
every call raise.
"""
from __future__ import annotations

import contextlib
import ctypes as C
from dataclasses import dataclass

import torch

from ._native import (  # noqa: F401
    CASGD_LOGISTIC, CASGD_LSQ, CASGD_POISSON, ExchangeFn as _ExchangeFn, FLAG_GRAM_NO_CLUSTER,
    FLAG_FAR_FROM_GRAM, FLAG_FULL_G, FLAG_GRAM_PAIR, FLAG_SAMPLE_PERMUTED, FLAG_NO_FUSE,
    FLAG_TRACE_CHAIN, FLAG_MARGINS_FP32, FLAG_G_BF16, FLAG_GATHER_ROWS,
    FLAG_GRAM_SIMT,
    FLAG_GRAM_TENSOR,
    FLAG_TEST_STALL, FLAG_WRITE_DIAG_BLOCKS, STAGE_EVENTS, CasgdError, Data as _Data,
    Params as _Params, Profile as _Profile, Taps as _Taps, check as _check, header_symbols,
    load,
)

LOGISTIC, LSQ, POISSON = CASGD_LOGISTIC, CASGD_LSQ, CASGD_POISSON


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _ptr(t) -> C.c_void_p | None:
    return None if t is None else C.c_void_p(t.data_ptr())


def _need_cuda(t: torch.Tensor, name: str, dtype=None) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


@dataclass
class Params:
    b: int
    s: int
    eta: float
    loss: int
    seed: int = 0
    flags: int = 0
    timeout_us: int = 0

    @property
    def S(self) -> int:
        return self.b * self.s

    def c(self) -> _Params:
        return _Params(self.b, self.s, self.eta, self.loss, self.seed, self.flags,
                       self.timeout_us)


class Dataset:
    """BF16 data matrix X (m x ld, device) with n features and FP32 labels y."""

    def __init__(self, X: torch.Tensor, y: torch.Tensor, n: int):
        _need_cuda(X, "X", torch.bfloat16)
        _need_cuda(y, "y", torch.float32)
        if X.dim() != 2 or y.numel() != X.shape[0]:
            raise ValueError("X must be m x ld and y must have m entries")
        self.X, self.y, self.n = X, y, int(n)
        self.m, self.ld = int(X.shape[0]), int(X.shape[1])

    def c(self) -> _Data:
        return _Data(self.m, self.n, self.ld, self.X.data_ptr(), self.y.data_ptr())

    @classmethod
    def from_fp32(cls, X32: torch.Tensor, y: torch.Tensor, stream=None) -> "Dataset":
        """Stores an FP32 device matrix as BF16 (casgd_store_bf16), padded to ld % 8 == 0."""
        X = store_bf16(X32, stream=stream)
        return cls(X, y, X32.shape[1])


def store_bf16(X32: torch.Tensor, ld: int | None = None, stream=None) -> torch.Tensor:
    _need_cuda(X32, "X32", torch.float32)
    m, n = X32.shape
    ld = (n + 7) // 8 * 8 if ld is None else int(ld)
    out = torch.empty((m, ld), dtype=torch.bfloat16, device=X32.device)
    _check(load().casgd_store_bf16(_ptr(X32), m, n, n, _ptr(out), ld, _stream(stream)),
           "casgd_store_bf16")
    return out


def sample_indices(m: int, count: int, seed: int, counter0: int, device="cuda",
                   stream=None, permuted: bool = False) -> torch.Tensor:
    """Row indices for sampler counters counter0 .. counter0+count-1: with replacement,
    or (permuted) without replacement within each epoch of m draws."""
    out = torch.empty(count, dtype=torch.int32, device=device)
    name = "casgd_sample_indices_permuted" if permuted else "casgd_sample_indices"
    _check(getattr(load(), name)(m, count, seed, counter0, _ptr(out), _stream(stream)), name)
    return out


def gram_elems(b: int, s: int, flags: int = 0) -> int:
    return int(load().casgd_gram_elems(b, s, flags))


def workspace_size(data: Dataset, params: Params) -> int:
    nbytes = C.c_size_t(0)
    _check(load().casgd_workspace_size(C.byref(data.c()), C.byref(params.c()), C.byref(nbytes)),
           "casgd_workspace_size")
    return int(nbytes.value)


def workspace(data: Dataset, params: Params, stream=None) -> torch.Tensor:
    """A fresh, initialised device workspace for (data, params)."""
    nbytes = workspace_size(data, params)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=data.X.device)
    _check(load().casgd_workspace_init(_ptr(ws), nbytes, _stream(stream)), "casgd_workspace_init")
    return ws


@dataclass
class Taps:
    idx_in: torch.Tensor | None = None
    idx_out: torch.Tensor | None = None
    G_out: torch.Tensor | None = None
    r_out: torch.Tensor | None = None
    alpha_out: torch.Tensor | None = None

    def c(self) -> _Taps:
        return _Taps(_ptr(self.idx_in), _ptr(self.idx_out), _ptr(self.G_out), _ptr(self.r_out),
                     _ptr(self.alpha_out))

    @classmethod
    def alloc(cls, params: Params, device="cuda", G=True) -> "Taps":
        S = params.S
        return cls(
            idx_out=torch.empty(S, dtype=torch.int32, device=device),
            G_out=(torch.empty(gram_elems(params.b, params.s, params.flags), dtype=torch.float32,
                               device=device) if G else None),
            # BF16 bit patterns, or FP32 values (two int16 each) with FLAG_MARGINS_FP32
            r_out=torch.empty(2 * S if params.flags & FLAG_MARGINS_FP32 else S,
                              dtype=torch.int16, device=device),
            alpha_out=torch.empty(S, dtype=torch.float32, device=device),
        )


def outer_step(data: Dataset, params: Params, w: torch.Tensor, k: int, ws: torch.Tensor,
               taps: Taps | None = None, stream=None) -> None:
    """One outer iteration k on w (FP32[n], updated in place).  Asynchronous."""
    _need_cuda(w, "w", torch.float32)
    t = C.byref(taps.c()) if taps is not None else None
    _check(load().casgd_outer_step(C.byref(data.c()), C.byref(params.c()), _ptr(w), k, _ptr(ws),
                                   ws.numel(), _stream(stream), t), "casgd_outer_step")


def train(data: Dataset, params: Params, w: torch.Tensor, iters: int, ws: torch.Tensor,
          k0: int = 0, loss_every: int = 0, stream=None, stage_events=None):
    """`iters` outer iterations; returns (loss history list, launches, gram_kind).  Blocks."""
    _need_cuda(w, "w", torch.float32)
    nl = iters // loss_every if loss_every > 0 else 0
    hist = (C.c_double * max(nl, 1))()
    prof = _Profile()
    ev_arr = None
    if stage_events is not None:
        ev_arr = (C.c_void_p * len(stage_events))(
            *[e.cuda_event if e is not None else None for e in stage_events])
        prof.stage_events = C.cast(ev_arr, C.POINTER(C.c_void_p))
        prof.n_events = len(stage_events)
    _check(load().casgd_train(C.byref(data.c()), C.byref(params.c()), _ptr(w), k0, iters,
                              _ptr(ws), ws.numel(), _stream(stream), loss_every,
                              hist if nl > 0 else None, C.byref(prof)), "casgd_train")
    return [hist[i] for i in range(nl)], int(prof.launches), int(prof.gram_kind)


def _need_host(t: torch.Tensor, name: str, dtype, numel: int) -> None:
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a CPU tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name} must hold at least {numel} elements, has {t.numel()}")


def train_host(X_host: torch.Tensor, y_host: torch.Tensor, w_host: torch.Tensor,
               data: Dataset, w_dev: torch.Tensor, params: Params, iters: int,
               ws: torch.Tensor, k0: int = 0, loss_every: int = 0, stream=None):
    """casgd_train on host inputs: X_host (CPU BF16, the layout of data.X), y_host and
    w_host (CPU FP32; pin them for full-rate copies) are copied into data's device buffers
    and w_dev, and w_host receives the result.  Returns (loss history, launches,
    gram_kind).  Blocks."""
    _need_host(X_host, "X_host", torch.bfloat16, data.X.numel())
    _need_host(y_host, "y_host", torch.float32, data.m)
    _need_host(w_host, "w_host", torch.float32, data.n)
    _need_cuda(w_dev, "w_dev", torch.float32)
    if w_dev.numel() < data.n:
        raise ValueError(f"w_dev must hold at least {data.n} elements")
    nl = iters // loss_every if loss_every > 0 else 0
    hist = (C.c_double * max(nl, 1))()
    prof = _Profile()
    _check(load().casgd_train_host(_ptr(X_host), _ptr(y_host), _ptr(w_host), C.byref(data.c()),
                                   _ptr(w_dev), C.byref(params.c()), k0, iters, _ptr(ws),
                                   ws.numel(), _stream(stream), loss_every,
                                   hist if nl > 0 else None, C.byref(prof)), "casgd_train_host")
    return [hist[i] for i in range(nl)], int(prof.launches), int(prof.gram_kind)


def loss(data: Dataset, kind: int, w: torch.Tensor, ws: torch.Tensor, stream=None) -> float:
    """Full-data loss f(w) (FP64 result).  Blocks."""
    out = C.c_double(0.0)
    _check(load().casgd_loss(C.byref(data.c()), kind, _ptr(w), _ptr(ws), ws.numel(),
                             _stream(stream), C.byref(out)), "casgd_loss")
    return float(out.value)


def loss_async(data: Dataset, kind: int, w: torch.Tensor, ws: torch.Tensor,
               out_dev: torch.Tensor, stream=None) -> None:
    _need_cuda(out_dev, "out_dev", torch.float64)
    _check(load().casgd_loss_async(C.byref(data.c()), kind, _ptr(w), _ptr(ws), ws.numel(),
                                   _stream(stream), _ptr(out_dev)), "casgd_loss_async")


def get_status(ws: torch.Tensor, stream=None) -> int:
    """Sticky device status of ws (0 = ok); clears it.  Blocks."""
    return int(load().casgd_get_status(_ptr(ws), _stream(stream)))


def chain_trace(data: Dataset, params: Params, ws: torch.Tensor, stream=None) -> list:
    """Chain timeline of the last outer iteration run with FLAG_TRACE_CHAIN: per phase
    j, globaltimer ns (start, loads issued, inputs final, alpha_j stored), then one
    summary row (last tile of G stored, last far sum stored, last update partial
    stored, 0).  Blocks."""
    out = (C.c_uint64 * (4 * params.s + 4))()
    _check(load().casgd_chain_trace(C.byref(data.c()), C.byref(params.c()), _ptr(ws), ws.numel(),
                                    _stream(stream), out), "casgd_chain_trace")
    return [tuple(out[4 * j + e] for e in range(4)) for j in range(params.s + 1)]


def sgd_workspace(b: int, device="cuda") -> torch.Tensor:
    """Zeroed workspace for sgd_fp32 with minibatch size b."""
    nb = C.c_size_t(0)
    _check(load().casgd_sgd_workspace_size(b, C.byref(nb)), "casgd_sgd_workspace_size")
    return torch.zeros(nb.value, dtype=torch.uint8, device=device)


def sgd_fp32(X: torch.Tensor, y: torch.Tensor, params: Params, w: torch.Tensor, steps: int,
             ws: torch.Tensor, q0: int = 0, stream=None) -> None:
    """FP32 plain minibatch SGD (steps q0 .. q0+steps-1) on FP32 X (m x n, row-major,
    contiguous rows), the baseline CA-SGD is compared with.  Asynchronous."""
    _need_cuda(X, "X", torch.float32)
    _need_cuda(y, "y", torch.float32)
    _need_cuda(w, "w", torch.float32)
    m, n = X.shape
    _check(load().casgd_sgd_fp32(_ptr(X), m, n, X.stride(0), _ptr(y), C.byref(params.c()),
                                 _ptr(w), q0, steps, _ptr(ws), ws.numel(), _stream(stream)),
           "casgd_sgd_fp32")


def update_static(Y: torch.Tensor, alpha: torch.Tensor, w: torch.Tensor, n: int,
                  stream=None) -> None:
    """w += Y^T alpha without a workspace and without allocating device memory.

    For callers that cannot allocate where they apply an update; the scratch is a
    fixed array inside the library (see casgd_update_static in include/casgd.h for the
    size limit and the rule that overlapping calls must be serialised).  Y is the BF16
    S x ldY matrix of the gathered rows, alpha FP32[S], w FP32[n] updated in place.
    """
    # The library cannot see buffer lengths: refuse shapes that would let it read or
    # write past a tensor before anything is called.
    if not isinstance(Y, torch.Tensor) or Y.dim() != 2:
        raise ValueError("Y must be a 2-D S x ldY tensor")
    S, ldY = int(Y.shape[0]), int(Y.shape[1])
    n = int(n)
    if not 1 <= n <= ldY:
        raise ValueError(f"n must be in [1, ldY = {ldY}], got {n}")
    if not isinstance(alpha, torch.Tensor) or alpha.numel() < S:
        raise ValueError(f"alpha must hold at least S = {S} values")
    if not isinstance(w, torch.Tensor) or w.numel() < n:
        raise ValueError(f"w must hold at least n = {n} values")
    _need_cuda(Y, "Y", torch.bfloat16)
    _need_cuda(alpha, "alpha", torch.float32)
    _need_cuda(w, "w", torch.float32)
    _check(load().casgd_update_static(_ptr(Y), S, n, ldY, _ptr(alpha), _ptr(w),
                                      _stream(stream)), "casgd_update_static")


# ----------------------------------------------------- feature-sharded outer iteration
def exchange_elems(b: int, s: int, flags: int = 0) -> int:
    """Floats of the exchange buffer: the packed block-lower G, then S margins."""
    v = int(load().casgd_exchange_elems(b, s, flags))
    if v < 0:
        raise ValueError("invalid (b, s, flags)")
    return v


def workspace_sharded(data: Dataset, params: Params, stream=None) -> torch.Tensor:
    """A fresh, initialised workspace for the sharded calls on this process's slice."""
    nbytes = C.c_size_t(0)
    _check(load().casgd_workspace_size_sharded(C.byref(data.c()), C.byref(params.c()),
                                               C.byref(nbytes)), "casgd_workspace_size_sharded")
    ws = torch.empty(int(nbytes.value), dtype=torch.uint8, device=data.X.device)
    _check(load().casgd_workspace_init(_ptr(ws), ws.numel(), _stream(stream)),
           "casgd_workspace_init")
    return ws


def exchange_buffer(params: Params, device="cuda") -> torch.Tensor:
    """The caller-owned FP32 exchange buffer (torch allocations are 256-byte aligned)."""
    return torch.zeros(exchange_elems(params.b, params.s, params.flags), dtype=torch.float32,
                       device=device)


def outer_step_local(data: Dataset, params: Params, w: torch.Tensor, k: int, ws: torch.Tensor,
                     xbuf: torch.Tensor, taps: Taps | None = None, stream=None) -> None:
    """First half of sharded outer iteration k: this slice's partial G and margins into
    xbuf.  Sum xbuf over the processes, then call outer_step_finish.  Asynchronous."""
    _need_cuda(w, "w", torch.float32)
    _need_cuda(xbuf, "xbuf", torch.float32)
    if xbuf.numel() < exchange_elems(params.b, params.s, params.flags):
        raise ValueError("xbuf is smaller than exchange_elems(b, s, flags)")
    t = C.byref(taps.c()) if taps is not None else None
    _check(load().casgd_outer_step_local(C.byref(data.c()), C.byref(params.c()), _ptr(w), k,
                                         _ptr(ws), ws.numel(), _stream(stream), _ptr(xbuf), t),
           "casgd_outer_step_local")


def outer_step_finish(data: Dataset, params: Params, w: torch.Tensor, ws: torch.Tensor,
                      xbuf: torch.Tensor, taps: Taps | None = None, stream=None) -> None:
    """Second half: the recurrence on the summed xbuf and this slice's update of w."""
    _need_cuda(w, "w", torch.float32)
    _need_cuda(xbuf, "xbuf", torch.float32)
    if xbuf.numel() < exchange_elems(params.b, params.s, params.flags):
        raise ValueError("xbuf is smaller than exchange_elems(b, s, flags)")
    t = C.byref(taps.c()) if taps is not None else None
    _check(load().casgd_outer_step_finish(C.byref(data.c()), C.byref(params.c()), _ptr(w),
                                          _ptr(ws), ws.numel(), _stream(stream), _ptr(xbuf), t),
           "casgd_outer_step_finish")


def make_exchange(xbuf: torch.Tensor, all_reduce):
    """The exchange hook the C loop calls once per outer iteration, as a Python callable
    (ctx, buf, count, stream) -> int: it sums xbuf[:count] in place over the processes
    with all_reduce (for example torch.distributed.all_reduce, which on an NCCL process
    group is ncclAllReduce with ncclSum), ordered on the library's stream.  Returns 0, or
    1 when the buffer is not xbuf or all_reduce raised (the loop then stops with
    CASGD_ERR_EXCHANGE)."""
    def hook(ctx, buf, count, stream_ptr):
        try:
            if buf != xbuf.data_ptr() or not 0 <= count <= xbuf.numel():
                return 1
            view = xbuf[:count]
            ctxm = (torch.cuda.stream(torch.cuda.ExternalStream(stream_ptr))
                    if xbuf.is_cuda and stream_ptr else contextlib.nullcontext())
            with ctxm:
                all_reduce(view)
            return 0
        except Exception:  # noqa: BLE001 -- reported to the C loop as a failed exchange
            return 1
    return hook


def train_sharded(data: Dataset, params: Params, w: torch.Tensor, iters: int, ws: torch.Tensor,
                  xbuf: torch.Tensor, all_reduce, k0: int = 0, stream=None, stage_events=None):
    """`iters` feature-sharded outer iterations on this process's slice (data: its columns
    of X and the full y; w: its slice).  all_reduce(t) must sum the FP32 tensor t in
    place over the processes (None: one process, the identity).  Blocks; returns
    (launches, gram_kind)."""
    _need_cuda(w, "w", torch.float32)
    _need_cuda(xbuf, "xbuf", torch.float32)
    if xbuf.numel() < exchange_elems(params.b, params.s, params.flags):
        raise ValueError("xbuf is smaller than exchange_elems(b, s, flags)")
    hook = _ExchangeFn(make_exchange(xbuf, all_reduce if all_reduce is not None
                                     else (lambda t: None)))
    prof = _Profile()
    ev_arr = None
    if stage_events is not None:
        ev_arr = (C.c_void_p * len(stage_events))(
            *[e.cuda_event if e is not None else None for e in stage_events])
        prof.stage_events = C.cast(ev_arr, C.POINTER(C.c_void_p))
        prof.n_events = len(stage_events)
    _check(load().casgd_train_sharded(C.byref(data.c()), C.byref(params.c()), _ptr(w), k0, iters,
                                      _ptr(ws), ws.numel(), _stream(stream), _ptr(xbuf), hook,
                                      None, C.byref(prof)), "casgd_train_sharded")
    return int(prof.launches), int(prof.gram_kind)

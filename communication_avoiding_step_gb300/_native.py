"""ctypes declarations for libcasgd.so (mirrors include/casgd.h)."""
from __future__ import annotations

import ctypes as C
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libcasgd.so")
HEADER = os.path.join(ROOT, "include", "casgd.h")

CASGD_LOGISTIC, CASGD_LSQ, CASGD_POISSON = 0, 1, 2
(CASGD_OK, CASGD_ERR_ARG, CASGD_ERR_WORKSPACE, CASGD_ERR_CUDA, CASGD_ERR_NONFINITE,
 CASGD_ERR_TIMEOUT, CASGD_ERR_BAD_INDEX, CASGD_ERR_UNSUPPORTED, CASGD_ERR_SCRATCH_LIMIT,
 CASGD_ERR_EXCHANGE) = range(10)
FLAG_WRITE_DIAG_BLOCKS = 0x1
FLAG_GRAM_TENSOR = 0x2
FLAG_GRAM_SIMT = 0x4
FLAG_GRAM_NO_CLUSTER = 0x8
FLAG_GRAM_PAIR = 0x20
FLAG_NO_FUSE = 0x40
FLAG_TRACE_CHAIN = 0x100
FLAG_FAR_FROM_GRAM = 0x200
FLAG_FULL_G = 0x400
FLAG_SAMPLE_PERMUTED = 0x800
FLAG_MARGINS_FP32 = 0x1000
FLAG_G_BF16 = 0x2000
FLAG_GATHER_ROWS = 0x4000
FLAG_TEST_STALL = 0x80000000
STAGE_EVENTS = 5


class Data(C.Structure):
    _fields_ = [("m", C.c_int64), ("n", C.c_int64), ("ld", C.c_int64),
                ("X", C.c_void_p), ("y", C.c_void_p)]


class Params(C.Structure):
    _fields_ = [("b", C.c_int32), ("s", C.c_int32), ("eta", C.c_float), ("loss", C.c_int32),
                ("seed", C.c_uint64), ("flags", C.c_uint32), ("timeout_us", C.c_uint32)]


class Taps(C.Structure):
    _fields_ = [("idx_in", C.c_void_p), ("idx_out", C.c_void_p), ("G_out", C.c_void_p),
                ("r_out", C.c_void_p), ("alpha_out", C.c_void_p)]


class Profile(C.Structure):
    _fields_ = [("launches", C.c_int64), ("stage_events", C.POINTER(C.c_void_p)),
                ("n_events", C.c_int32), ("gram_kind", C.c_int32)]


_P = C.POINTER
# int (*casgd_exchange_fn)(void* ctx, float* buf, int64_t count, void* stream)
ExchangeFn = C.CFUNCTYPE(C.c_int, C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p)

SIGNATURES = {
    "casgd_strerror": (C.c_char_p, [C.c_int]),
    "casgd_version": (C.c_int, []),
    "casgd_gram_elems": (C.c_int64, [C.c_int32, C.c_int32, C.c_uint32]),
    "casgd_workspace_size": (C.c_int, [_P(Data), _P(Params), _P(C.c_size_t)]),
    "casgd_workspace_init": (C.c_int, [C.c_void_p, C.c_size_t, C.c_void_p]),
    "casgd_store_bf16": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_int64, C.c_void_p,
                                   C.c_int64, C.c_void_p]),
    "casgd_sample_indices": (C.c_int, [C.c_int64, C.c_int64, C.c_uint64, C.c_uint64,
                                       C.c_void_p, C.c_void_p]),
    "casgd_sample_indices_permuted": (C.c_int, [C.c_int64, C.c_int64, C.c_uint64, C.c_uint64,
                                       C.c_void_p, C.c_void_p]),
    "casgd_outer_step": (C.c_int, [_P(Data), _P(Params), C.c_void_p, C.c_uint64, C.c_void_p,
                                   C.c_size_t, C.c_void_p, _P(Taps)]),
    "casgd_train": (C.c_int, [_P(Data), _P(Params), C.c_void_p, C.c_uint64, C.c_int32,
                              C.c_void_p, C.c_size_t, C.c_void_p, C.c_int32,
                              _P(C.c_double), _P(Profile)]),
    "casgd_train_host": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, _P(Data), C.c_void_p,
                                   _P(Params), C.c_uint64, C.c_int32, C.c_void_p, C.c_size_t,
                                   C.c_void_p, C.c_int32, _P(C.c_double), _P(Profile)]),
    "casgd_loss": (C.c_int, [_P(Data), C.c_int32, C.c_void_p, C.c_void_p, C.c_size_t,
                             C.c_void_p, _P(C.c_double)]),
    "casgd_loss_async": (C.c_int, [_P(Data), C.c_int32, C.c_void_p, C.c_void_p, C.c_size_t,
                                   C.c_void_p, C.c_void_p]),
    "casgd_get_status": (C.c_int, [C.c_void_p, C.c_void_p]),
    "casgd_chain_trace": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p,
                                    C.POINTER(C.c_uint64)]),
    "casgd_sgd_workspace_size": (C.c_int, [C.c_int32, C.POINTER(C.c_size_t)]),
    "casgd_sgd_fp32": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_int64, C.c_void_p,
                                 C.c_void_p, C.c_void_p, C.c_uint64, C.c_int32, C.c_void_p,
                                 C.c_size_t, C.c_void_p]),
    "casgd_update_static": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_int64, C.c_void_p,
                                      C.c_void_p, C.c_void_p]),
    "casgd_exchange_elems": (C.c_int64, [C.c_int32, C.c_int32, C.c_uint32]),
    "casgd_workspace_size_sharded": (C.c_int, [_P(Data), _P(Params), _P(C.c_size_t)]),
    "casgd_outer_step_local": (C.c_int, [_P(Data), _P(Params), C.c_void_p, C.c_uint64,
                                         C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p,
                                         _P(Taps)]),
    "casgd_outer_step_finish": (C.c_int, [_P(Data), _P(Params), C.c_void_p, C.c_void_p,
                                          C.c_size_t, C.c_void_p, C.c_void_p, _P(Taps)]),
    "casgd_train_sharded": (C.c_int, [_P(Data), _P(Params), C.c_void_p, C.c_uint64, C.c_int32,
                                      C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p,
                                      ExchangeFn, C.c_void_p, _P(Profile)]),
}

_lib = None


def header_symbols() -> list[str]:
    """Every function the public header declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(casgd_\w+)\s*\(", txt)))


def load() -> C.CDLL:
    """Load the in-tree libcasgd.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m communication_avoiding_step_gb300.build`")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class CasgdError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = load().casgd_strerror(code).decode()
        super().__init__(f"{where}: casgd error {code} ({msg})")


def check(code: int, where: str) -> None:
    if code != CASGD_OK:
        raise CasgdError(code, where)

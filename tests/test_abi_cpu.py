"""The C-ABI library loads and exports every symbol include/casgd.h declares.

No GPU here: only host-only entry points are called (messages, sizes) and argument
checks that must reject a request before any CUDA call is made.
"""
import ctypes as C
import subprocess

import pytest

import communication_avoiding_step_gb300 as casgd
from communication_avoiding_step_gb300 import _native as nat


@pytest.fixture(scope="module")
def lib():
    return casgd.load()


def test_every_header_symbol_is_exported(lib):
    syms = nat.header_symbols()
    assert len(syms) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", nat.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for s in syms:
        assert s in exported, s
        assert hasattr(lib, s)
    # and the binding declares a prototype for each of them
    assert set(syms) == set(nat.SIGNATURES)


def test_version_and_messages(lib):
    assert lib.casgd_version() == 1
    for code in range(8):
        assert lib.casgd_strerror(code)
    assert b"unknown" in lib.casgd_strerror(99)


def test_gram_elems(lib):
    assert lib.casgd_gram_elems(256, 32, 0) == 32 * 31 // 2 * 256 * 256
    assert lib.casgd_gram_elems(256, 32, nat.FLAG_WRITE_DIAG_BLOCKS) == 32 * 33 // 2 * 256 * 256
    assert lib.casgd_gram_elems(16, 1, 0) == 0
    assert lib.casgd_gram_elems(0, 4, 0) == -1
    assert lib.casgd_gram_elems(4096, 32, 0) == -1        # S over 65536
    assert lib.casgd_gram_elems(1, 65, 0) == -1           # s over 64


def test_workspace_size_host_only(lib):
    d = nat.Data(1000, 2000, 2000, 0, 0)
    p = nat.Params(256, 32, 0.5, 0, 0, 0, 0)
    nbytes = C.c_size_t(0)
    assert lib.casgd_workspace_size(C.byref(d), C.byref(p), C.byref(nbytes)) == 0
    S = 256 * 32
    g = 2 * 90 * 256 * 256 * 4   # two band-layout G buffers of the far-forming default
    assert nbytes.value >= g + 2 * S * 2048 * 2 + S * 14
    assert nbytes.value % 256 == 0
    bad = nat.Params(256, 32, 0.5, 7, 0, 0, 0)
    assert lib.casgd_workspace_size(C.byref(d), C.byref(bad), C.byref(nbytes)) == nat.CASGD_ERR_ARG


def test_unknown_flag_bits_rejected(lib):
    # bit 0x10 named the cluster-multicast Gram, which the library no longer has
    d = nat.Data(1000, 2000, 2000, 0, 0)
    nbytes = C.c_size_t(0)
    for flags in (0x10, 0x8000, 0x40000000):
        p = nat.Params(256, 32, 0.5, 0, 0, flags, 0)
        assert lib.casgd_workspace_size(C.byref(d), C.byref(p), C.byref(nbytes)) == nat.CASGD_ERR_ARG
    known = (nat.FLAG_WRITE_DIAG_BLOCKS | nat.FLAG_GRAM_TENSOR | nat.FLAG_GRAM_PAIR
             | nat.FLAG_FULL_G | nat.FLAG_G_BF16 | nat.FLAG_MARGINS_FP32)
    p = nat.Params(256, 32, 0.5, 0, 0, known, 0)
    assert lib.casgd_workspace_size(C.byref(d), C.byref(p), C.byref(nbytes)) == 0


def _ws_bytes(lib, n, b, s, flags):
    nbytes = C.c_size_t(0)
    d = nat.Data(1000, n, (n + 7) // 8 * 8, 0, 0)
    p = nat.Params(b, s, 0.1, 0, 0, flags, 0)
    assert lib.casgd_workspace_size(C.byref(d), C.byref(p), C.byref(nbytes)) == 0
    return nbytes.value


def _a(x):  # 256-byte sections
    return (x + 255) // 256 * 256


def _band_blocks(s, B):
    return sum(min(j, B) for j in range(s))


def test_workspace_sections_of_the_gram_paths(lib):
    # b = 256, s = 32, n = 2000: the stored-G launch shared with the recurrence (FULL_G)
    # adds a second idx, y_Y, Y and G for casgd_train's iteration-ahead Gram; the
    # far-forming default keeps both G buffers in the band layout (the B = 3 blocks
    # below the diagonal of each block row: 90 of the 496 blocks) and adds the far
    # partials (one column group per block: S x s floats), a third set of row buffers
    # (idx, y_Y, Y: the launch of iteration k gathers iteration k+2's rows) and a second
    # recurrence state (control block, counters area, r, alpha, far sums, far partials:
    # the launches alternate between two)
    n, b, s = 2000, 256, 32
    S, ld = b * s, 2048          # Y rows padded to whole 128-byte lines
    G = s * (s - 1) // 2 * b * b * 4
    Gb = _band_blocks(s, 3) * b * b * 4
    assert _band_blocks(s, 3) == 90
    no_fuse = _ws_bytes(lib, n, b, s, nat.FLAG_NO_FUSE)
    full_g = _ws_bytes(lib, n, b, s, nat.FLAG_FULL_G)
    far = _ws_bytes(lib, n, b, s, 0)
    assert full_g - no_fuse == 2 * _a(S * 4) + _a(S * ld * 2) + _a(G)
    counters = _a((65536 // 256 * 8 + 16384 // 64 + 64 * (16384 // 64)) * 4 + 65 * 4 * 8)
    state2 = _a(32) + counters + 3 * _a(S * 4) + _a(S * s * 1 * 4)
    assert far - full_g == (2 * _a(Gb) - 2 * _a(G) + _a(S * s * 1 * 4)
                            + _a(S * 4) + _a(S * 4) + _a(S * ld * 2) + state2)
    # b = 1024, s = 16, n = 18 (narrow rows, gathered ahead with plain loads: third row
    # buffers and a second state too): the stored G is not shared with the recurrence there
    # (b > 512), so only the far-forming path has second buffers; its band is one block
    # wide; four column groups per block keep a row's far partials within 64
    n, b, s = 18, 1024, 16
    S, ld = b * s, 24
    G = s * (s - 1) // 2 * b * b * 4
    Gb = _band_blocks(s, 1) * b * b * 4
    full_g = _ws_bytes(lib, n, b, s, nat.FLAG_FULL_G)
    far = _ws_bytes(lib, n, b, s, 0)
    state2 = _a(32) + counters + 3 * _a(S * 4) + _a(S * s * 4 * 4)
    assert far - full_g == (2 * _a(S * 4) + _a(S * ld * 2) + 2 * _a(Gb) - _a(G)
                            + _a(S * s * 4 * 4)
                            + 2 * _a(S * 4) + _a(S * ld * 2) + state2)
    # least squares 11,000,000 x 28 at b = 2048, s = 32 (S = 65536): 31 band blocks of
    # 16 MiB per buffer instead of 496 (8.3 GB) in the packed block-lower layout
    far = _ws_bytes(lib, 28, 2048, 32, 0)
    full_g = _ws_bytes(lib, 28, 2048, 32, nat.FLAG_FULL_G)
    assert far < 1.2e9 < 8.3e9 < full_g


def test_argument_errors_before_any_cuda_call(lib):
    p = nat.Params(16, 4, 0.1, 0, 0, 0, 0)
    fake = 1 << 20  # never dereferenced: every case fails validation first
    cases = [
        nat.Data(0, 64, 64, fake, fake),          # m = 0
        nat.Data(100, 64, 60, fake, fake),        # ld < n
        nat.Data(100, 64, 68, fake, fake),        # ld % 8 != 0
        nat.Data(100, 64, 64, fake + 8, fake),    # X not 16-byte aligned
        nat.Data(100, 20000, 20000, fake, fake),  # n over 16384
        nat.Data(100, 64, 64, None, fake),        # null X
    ]
    for d in cases:
        rc = lib.casgd_outer_step(C.byref(d), C.byref(p), C.c_void_p(fake), 0, C.c_void_p(fake),
                                  1 << 30, None, None)
        assert rc == nat.CASGD_ERR_ARG
    good = nat.Data(100, 64, 64, fake, fake)
    for bp in (nat.Params(0, 4, 0.1, 0, 0, 0, 0), nat.Params(16, 0, 0.1, 0, 0, 0, 0),
               nat.Params(16, 65, 0.1, 0, 0, 0, 0), nat.Params(4096, 32, 0.1, 0, 0, 0, 0),
               nat.Params(16, 4, 0.1, 3, 0, 0, 0), nat.Params(16, 4, float("nan"), 0, 0, 0, 0)):
        rc = lib.casgd_outer_step(C.byref(good), C.byref(bp), C.c_void_p(fake), 0,
                                  C.c_void_p(fake), 1 << 30, None, None)
        assert rc == nat.CASGD_ERR_ARG
    rc = lib.casgd_outer_step(C.byref(good), C.byref(p), None, 0, C.c_void_p(fake), 1 << 30,
                              None, None)
    assert rc == nat.CASGD_ERR_ARG
    rc = lib.casgd_store_bf16(C.c_void_p(fake), 10, 9, 9, C.c_void_p(fake + 4), 16, None)
    assert rc == nat.CASGD_ERR_ARG
    rc = lib.casgd_sample_indices(0, 10, 0, 0, C.c_void_p(fake), None)
    assert rc == nat.CASGD_ERR_ARG
    assert lib.casgd_get_status(None, None) == nat.CASGD_ERR_WORKSPACE
    # casgd_train_host: a null host buffer, a null w_dev or bad data, before any copy
    hp = C.c_void_p(fake)
    for args in ((None, hp, hp, good, hp), (hp, None, hp, good, hp), (hp, hp, None, good, hp),
                 (hp, hp, hp, good, None), (hp, hp, hp, cases[0], hp)):
        rc = lib.casgd_train_host(args[0], args[1], args[2], C.byref(args[3]), args[4],
                                  C.byref(p), 0, 1, C.c_void_p(fake), 1 << 30, None, 0, None,
                                  None)
        assert rc == nat.CASGD_ERR_ARG
    # FP32 SGD: bad shapes, params and workspaces are rejected before any CUDA call
    nb = C.c_size_t(0)
    assert lib.casgd_sgd_workspace_size(256, C.byref(nb)) == 0 and nb.value >= 256 * 8
    assert lib.casgd_sgd_workspace_size(0, C.byref(nb)) == nat.CASGD_ERR_ARG
    sp = nat.Params(16, 1, 0.1, 0, 0, 0, 0)
    for args in ((None, 100, 8, 8), (fake, 0, 8, 8), (fake, 100, 8, 4), (fake, 100, 0, 8)):
        rc = lib.casgd_sgd_fp32(C.c_void_p(args[0]) if args[0] else None, args[1], args[2],
                                args[3], C.c_void_p(fake), C.byref(sp), C.c_void_p(fake), 0, 5,
                                C.c_void_p(fake), 1 << 20, None)
        assert rc == nat.CASGD_ERR_ARG
    rc = lib.casgd_sgd_fp32(C.c_void_p(fake), 100, 8, 8, C.c_void_p(fake),
                            C.byref(nat.Params(16, 1, 0.1, 5, 0, 0, 0)), C.c_void_p(fake), 0, 5,
                            C.c_void_p(fake), 1 << 20, None)
    assert rc == nat.CASGD_ERR_ARG
    rc = lib.casgd_sgd_fp32(C.c_void_p(fake), 100, 8, 8, C.c_void_p(fake), C.byref(sp),
                            C.c_void_p(fake), 0, 5, C.c_void_p(fake + 64), 1 << 20, None)
    assert rc == nat.CASGD_ERR_WORKSPACE
    assert lib.casgd_workspace_init(C.c_void_p(fake + 64), 4096, None) == nat.CASGD_ERR_WORKSPACE


def test_product_path_has_no_oracle_dependency():
    """The package and its build never import the oracle or the CPU reference."""
    import os
    import re
    pkg = os.path.dirname(casgd.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(root, f)).read()
                assert not re.search(r"\boracle\b", txt.replace("the oracle", "")), f


def test_update_static_refuses_bad_shapes_before_calling_the_library(monkeypatch):
    """The C side cannot see buffer lengths, so the binding refuses a Y that is not
    2-D, an n outside [1, ldY], a short alpha or a short w before the library is
    touched (checked here with CPU tensors and a library stand-in that fails if used)."""
    import torch

    def no_library():
        raise AssertionError("the library was called")

    monkeypatch.setattr(casgd, "load", no_library)
    Y = torch.zeros((64, 16), dtype=torch.bfloat16)
    a = torch.zeros(64)
    w = torch.zeros(16)
    bad = [
        (torch.zeros(64 * 16, dtype=torch.bfloat16), a, w, 16),   # Y not 2-D
        (Y, a, w, 17),                                             # n > ldY
        (Y, a, w, 0),                                              # n < 1
        (Y, torch.zeros(63), w, 16),                               # alpha shorter than S
        (Y, a, torch.zeros(15), 16),                               # w shorter than n
    ]
    for Yb, ab, wb, n in bad:
        with pytest.raises(ValueError):
            casgd.update_static(Yb, ab, wb, n)
    with pytest.raises(ValueError, match="CUDA"):                  # right shapes, host memory
        casgd.update_static(Y, a, w, 16)

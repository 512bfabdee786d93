"""Planted mistakes in the oracle (CPU only) must each fail one of its pins.

Each case swaps one oracle function for a plausibly wrong version via monkeypatch,
runs the pin that should notice, and expects it to fail.  Nothing here touches the
GPU path.
"""
import numpy as np
import pytest

import oracle
import oracle.casgd as oc
import tests.test_oracle_pins as pins

_orig_gram_block = oc.gram_block
_orig_loss_grad = oc.loss_grad
_orig_splitmix = oc.splitmix64
_orig_bf16 = oc.bf16_round
_orig_feistel = oc.feistel
_orig_epoch_keys = oc.epoch_keys
_orig_outer_step = oc.outer_step


def _drop_first_term(Y, b, j, t, mode="emulate"):
    g = _orig_gram_block(Y, b, j, t, mode)
    return g * 0 if t == 0 else g


def _transposed_block(Y, b, j, t, mode="emulate"):
    return _orig_gram_block(Y, b, t, j, mode)


def _logistic_sign_slip(z, y, kind):
    g = _orig_loss_grad(z, y, kind)
    return -g if kind == oracle.LOGISTIC else g


def _poisson_missing_exp(z, y, kind):
    if kind == oracle.POISSON:
        z = np.asarray(z)
        return z - np.asarray(y, dtype=z.dtype)
    return _orig_loss_grad(z, y, kind)


def _splitmix_off_by_one(seed, counter):
    return _orig_splitmix(seed, np.asarray(counter, dtype=np.uint64) - np.uint64(1))


def _bf16_truncate(x):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def _no_cycle_walk(m, count, seed, counter0):
    d = oc.perm_width(m)
    c = np.arange(count, dtype=np.int64) + int(counter0)
    out = np.empty(count, dtype=np.int64)
    for e in np.unique(c // m):
        sel = (c // m) == e
        out[sel] = oc.feistel(c[sel] % m, d, oc.epoch_keys(seed, int(e))).astype(np.int64)
    return out


def _keys_ignore_epoch(seed, e):
    return _orig_epoch_keys(seed, 0)


def _feistel_no_swap(x, d, keys):
    h = d // 2
    mask = np.uint64((1 << h) - 1)
    x = np.asarray(x, dtype=np.uint64)
    L, R = x >> np.uint64(h), x & mask
    for k in keys:
        L = L ^ (_orig_splitmix(int(k), R) & mask)  # halves never swap: R passes through
    return (L << np.uint64(h)) | R


def _margins_choice_ignored(*args, **kw):
    kw.pop("margins", None)
    return _orig_outer_step(*args, **kw)


def _gram_choice_ignored(*args, **kw):
    kw.pop("gram", None)
    return _orig_outer_step(*args, **kw)


CASES = [
    ("recurrence drops t=0", [("gram_block", _drop_first_term)],
     lambda: pins.test_ca_sgd_equals_s_sgd_steps_fp64(oracle.LSQ)),
    ("transposed Gram block", [("gram_block", _transposed_block)],
     lambda: pins.test_ca_sgd_equals_s_sgd_steps_fp64(oracle.LOGISTIC)),
    ("logistic derivative sign", [("loss_grad", _logistic_sign_slip)],
     lambda: pins.test_loss_grad_matches_finite_differences(oracle.LOGISTIC)),
    ("poisson derivative missing exp", [("loss_grad", _poisson_missing_exp)],
     lambda: pins.test_loss_grad_matches_finite_differences(oracle.POISSON)),
    ("generator counter off by one", [("splitmix64", _splitmix_off_by_one)],
     pins.test_splitmix64_known_answers),
    ("BF16 truncation instead of RNE", [("bf16_round", _bf16_truncate)],
     pins.test_bf16_round_edge_cases),
    ("permutation without cycle walking", [("permuted_indices", _no_cycle_walk)],
     pins.test_permuted_indices_visit_every_row_once_per_epoch),
    ("permutation keys ignore the epoch", [("epoch_keys", _keys_ignore_epoch)],
     pins.test_permuted_epochs_and_seeds_differ),
    ("Feistel halves never swap", [("feistel", _feistel_no_swap)],
     pins.test_permuted_uniform_chi2),
    ("FP32-margin variant still rounds", [("outer_step", _margins_choice_ignored)],
     pins.test_precision_variants_of_the_emulating_mode),
    ("BF16-G variant leaves G in FP32", [("outer_step", _gram_choice_ignored)],
     pins.test_precision_variants_of_the_emulating_mode),
]


@pytest.mark.parametrize("name,patches,pin", CASES, ids=[c[0] for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, patches, pin):
    for attr, fn in patches:
        monkeypatch.setattr(oc, attr, fn)
        monkeypatch.setattr(oracle, attr, fn)
    with pytest.raises(AssertionError):
        pin()


def test_unpatched_pins_pass():
    for _, _, pin in CASES:
        pin()

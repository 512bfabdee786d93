"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one oracle function to published generator outputs, exact rational
arithmetic, a closed form, finite differences, the CA-SGD == s-step SGD identity of
exact arithmetic, or an independent library routine.  A plausible slip in the oracle
(dropped term, wrong sign or index, transposed operand) fails at least one of them;
tests/test_oracle_mutations.py plants such slips and checks that.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth_inputs as si
from oracle import LOGISTIC, LSQ, POISSON

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
M64 = (1 << 64) - 1


# ------------------------------------------------------------------ sampling ----
def _splitmix_py(seed, counter):
    """Independent pure-Python-int statement of SplitMix64 (sequential form)."""
    state = seed & M64
    out = None
    for _ in range(counter + 1):
        state = (state + 0x9E3779B97F4A7C15) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out = z ^ (z >> 31)
    return out


def test_splitmix64_known_answers():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "splitmix64_kat.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) >= 6
    for seed, i, val in rows:
        got = int(oracle.splitmix64(int(seed), int(i)))
        assert got == int(val), (seed, i)


def test_splitmix64_matches_sequential_python():
    rng = np.random.default_rng(5)
    seeds = [0, 1, 2**63, M64, 0x0123456789ABCDEF] + [int(v) for v in rng.integers(0, 2**63, 5)]
    for seed in seeds:
        counters = np.arange(40)
        got = oracle.splitmix64(seed, counters)
        for c in range(40):
            assert int(got[c]) == _splitmix_py(seed, c)


def test_sample_indices_reduction_and_counters():
    m, seed = 1_000_003, 77
    idx = oracle.sample_indices(m, 64, seed, 5 * 64)
    for i in range(64):
        h = _splitmix_py(seed, 5 * 64 + i)
        assert idx[i] == ((h >> 32) * m) >> 32
    # outer iteration k uses counters k*S ...; plain SGD step q uses q*b ...
    b, s, k = 8, 4, 3
    ca = oracle.sample_indices(m, s * b, seed, k * s * b)
    sgd = np.concatenate([oracle.sample_indices(m, b, seed, (k * s + j) * b) for j in range(s)])
    assert np.array_equal(ca, sgd)
    assert idx.min() >= 0 and idx.max() < m


def test_sample_indices_uniform_chi2():
    from scipy import stats
    m = 1000
    idx = oracle.sample_indices(m, 1_000_000, 0, 0)
    counts = np.bincount(idx, minlength=m)
    p = stats.chisquare(counts).pvalue
    assert p > 1e-4
    assert idx.min() == 0 and idx.max() == m - 1


# ---------------------------------------------------------------------- bf16 ----
# --------------------------------------------- sampling without replacement ----
def test_perm_width():
    """d is the smallest even width with 2^d >= m (at least 2)."""
    for m, d in ((1, 2), (4, 2), (5, 4), (16, 4), (17, 6), (64, 6), (65, 8),
                 (4096, 12), (4097, 14), (11_000_000, 24), (2**31 - 1, 32)):
        assert oracle.perm_width(m) == d, m


def test_feistel_is_a_bijection_on_its_domain():
    """Any round keys give a permutation of [0, 2^d) (Luby-Rackoff structure)."""
    for d in (2, 4, 6, 10, 12):
        for seed, e in ((0, 0), (7, 3), (2**64 - 1, 1000)):
            keys = oracle.epoch_keys(seed, e)
            y = oracle.feistel(np.arange(2**d, dtype=np.uint64), d, keys)
            assert np.array_equal(np.sort(y), np.arange(2**d, dtype=np.uint64)), (d, seed, e)
            assert not np.array_equal(y, np.arange(2**d, dtype=np.uint64))


def test_permuted_indices_visit_every_row_once_per_epoch():
    """Brute force: the m draws of each epoch are a permutation of the m rows (cycle
    walking keeps the values below m), at every epoch and for widths that are and are
    not powers of two."""
    for m in (1, 2, 3, 5, 16, 17, 100, 1000, 4097):
        for seed in (0, 7, 2**64 - 1):
            for e in (0, 1, 3):
                idx = oracle.permuted_indices(m, m, seed, e * m)
                assert np.array_equal(np.sort(idx), np.arange(m)), (m, seed, e)
    # a range that starts inside an epoch and spans three more: each whole epoch once
    m = 37
    idx = oracle.permuted_indices(m, 5 * m, 3, 2 * m + 11)
    c = np.arange(5 * m) + 2 * m + 11
    for e in (3, 4, 5):
        assert np.array_equal(np.sort(idx[c // m == e]), np.arange(m))


def test_permuted_indices_are_a_function_of_the_counter():
    m = 1009
    whole = oracle.permuted_indices(m, 3000, 5, 123)
    parts = np.concatenate([oracle.permuted_indices(m, 1000, 5, 123 + 1000 * i)
                            for i in range(3)])
    assert np.array_equal(whole, parts)
    assert whole.min() >= 0 and whole.max() < m


def test_permuted_epochs_and_seeds_differ():
    """Different epochs and seeds give (nearly) unrelated permutations; none is close to
    the identity (a random permutation has one fixed point on average)."""
    m = 1000
    p00 = oracle.permuted_indices(m, m, 0, 0)
    p01 = oracle.permuted_indices(m, m, 0, m)
    p10 = oracle.permuted_indices(m, m, 1, 0)
    for a, b_ in ((p00, p01), (p00, p10), (p01, p10)):
        assert np.mean(a == b_) < 0.02
    for a in (p00, p01, p10):
        assert np.mean(a == np.arange(m)) < 0.02


def test_permuted_uniform_chi2():
    """Over many epochs, the row drawn at a fixed position, and the position at which a
    fixed row is drawn, are uniform (chi-square, 10 rows, 4000 epochs)."""
    scipy_stats = pytest.importorskip("scipy.stats")
    m, E = 10, 4000
    idx = oracle.permuted_indices(m, m * E, 2024, 0).reshape(E, m)
    first = np.bincount(idx[:, 0], minlength=m)
    where0 = np.bincount(np.argmax(idx == 0, axis=1), minlength=m)
    for counts in (first, where0):
        _, pv = scipy_stats.chisquare(counts)
        assert pv > 1e-4, counts


def test_ca_sgd_equals_s_sgd_steps_permuted_fp64():
    """The identity CA-SGD == s SGD steps holds for the permuted rows too (both sides
    draw the same rows for the same counters)."""
    p = si.make_random(120, 8, LSQ, seed=12)
    w0 = si.random_weights(8, seed=5, scale=0.3)
    b, s, eta, seed = 7, 5, 0.2, 3
    w_ca = w0.astype(np.float64)
    for k in range(4):  # 140 draws: past the first epoch of 120 rows
        w_ca = oracle.outer_step(p.X, p.y, w_ca, b, s, eta, LSQ, seed, k, mode="fp64",
                                 permuted=True)
    w_sgd = oracle.plain_sgd(p.X, p.y, b, 4 * s, eta, LSQ, seed, mode="fp64", w0=w0,
                             permuted=True)
    assert np.linalg.norm(w_ca - w_sgd) <= 1e-12 * np.linalg.norm(w_sgd)


def test_bf16_round_edge_cases():
    f = np.float32
    one = 1.0
    cases = {
        1.0: 1.0,
        one + 2.0**-8: 1.0,                       # exact tie, even -> down
        one + 3 * 2.0**-8: one + 2.0**-6,         # tie, odd -> up
        one + 2.0**-8 + 2.0**-20: one + 2.0**-7,  # just above the tie -> up
        -(one + 3 * 2.0**-8): -(one + 2.0**-6),
        2.0**-130: 2.0**-130,                     # subnormal kept
        0.0: 0.0,
    }
    for x, want in cases.items():
        got = oracle.bf16_round(np.array([x], dtype=f))[0]
        assert got == f(want), (x, got, want)
    # largest finite FP32 rounds up to infinity under RNE
    big = np.array([np.finfo(np.float32).max], dtype=f)
    assert np.isinf(oracle.bf16_round(big)[0])
    # -0.0 keeps its sign bit
    assert np.signbit(oracle.bf16_round(np.array([-0.0], dtype=f))[0])


def test_bf16_round_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3.0e38)]
    x = np.concatenate([x, rng.standard_normal(1 << 20).astype(np.float32)])
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float32).numpy()
    got = oracle.bf16_round(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# -------------------------------------------------------------------- losses ----
@pytest.mark.parametrize("kind", [LOGISTIC, LSQ, POISSON])
def test_loss_grad_matches_finite_differences(kind):
    rng = np.random.default_rng(kind)
    z = np.concatenate([rng.normal(0, 2, 200), [0.0, 5.0, -5.0]])
    if kind == LOGISTIC:
        z = np.concatenate([z, [30.0, -30.0, 200.0, -200.0]])
        y = np.where(rng.random(z.size) < 0.5, -1.0, 1.0)
    elif kind == LSQ:
        y = rng.normal(0, 1, z.size)
    else:
        y = rng.poisson(2.0, z.size).astype(np.float64)
    h = 1e-6
    fd = (oracle.loss_value(z + h, y, kind) - oracle.loss_value(z - h, y, kind)) / (2 * h)
    g = oracle.loss_grad(z, y, kind)
    assert np.all(np.isfinite(g))
    scale = 1.0 + np.abs(g)
    if kind == POISSON:
        scale = scale + np.exp(z)          # fd error grows with exp(z)
    assert np.all(np.abs(g - fd) <= 1e-6 * scale)


def test_loss_grad_closed_values():
    # logistic: l'(0, y) = -y/2;  l'(z, y) -> 0 as yz -> +inf, -> -y as yz -> -inf
    y = np.array([1.0, -1.0])
    assert np.allclose(oracle.loss_grad(np.zeros(2), y, LOGISTIC), [-0.5, 0.5], rtol=0, atol=0)
    assert np.allclose(oracle.loss_grad(np.array([800.0, -800.0]), y, LOGISTIC), [0.0, 0.0])
    assert np.allclose(oracle.loss_grad(np.array([-800.0, 800.0]), y, LOGISTIC), [-1.0, 1.0])
    assert oracle.loss_grad(np.array([2.0]), np.array([0.5]), LSQ)[0] == 1.5
    assert np.isclose(oracle.loss_grad(np.array([math.log(3.0)]), np.array([1.0]), POISSON)[0], 2.0)


@pytest.mark.parametrize("kind", [LOGISTIC, LSQ, POISSON])
def test_full_loss_at_zero(kind):
    p = si.make_random(500, 7, kind, seed=3)
    f0 = oracle.full_loss(p.X, p.y, np.zeros(7), kind)
    if kind == LOGISTIC:
        want = math.log(2.0)
    elif kind == LSQ:
        want = float(np.mean(p.y.astype(np.float64) ** 2) / 2)
    else:
        want = 1.0
    assert abs(f0 - want) <= 1e-14 * max(1.0, abs(want))


def test_full_loss_lsq_minimum_at_lstsq():
    p = si.make_random(400, 6, LSQ, seed=4)
    X = p.X.astype(np.float64)
    w_ls = np.linalg.lstsq(X, p.y.astype(np.float64), rcond=None)[0]
    f_ls = oracle.full_loss(p.X, p.y, w_ls, LSQ)
    # closed form: f = ||X w - y||^2 / (2 m)
    assert np.isclose(f_ls, np.sum((X @ w_ls - p.y) ** 2) / (2 * 400), rtol=1e-12)
    rng = np.random.default_rng(0)
    for _ in range(10):
        assert oracle.full_loss(p.X, p.y, w_ls + 1e-3 * rng.standard_normal(6), LSQ) > f_ls


# ---------------------------------------------------------------------- Gram ----
def _grid_bf16(rng, shape):
    """Values k/8 with |k| <= 64: exact in BF16, products and short sums exact in FP32."""
    return (rng.integers(-64, 65, size=shape) / 8.0).astype(np.float32)


def test_gram_exact_on_grid_values():
    rng = np.random.default_rng(2)
    b, s, n = 3, 4, 11
    Y = _grid_bf16(rng, (b * s, n))
    exact = [[sum(Fraction(float(Y[p, c])) * Fraction(float(Y[q, c])) for c in range(n))
              for q in range(b * s)] for p in range(b * s)]
    for mode in ("emulate", "fp64"):
        for diag in (False, True):
            G = oracle.gram_packed(Y, b, s, diag=diag, mode=mode)
            for j in range(s):
                for t in range(j + 1 if diag else j):
                    o = oracle.packed_block_offset(j, t, b, diag)
                    blk = G[o:o + b * b].reshape(b, b)
                    for i in range(b):
                        for c in range(b):
                            assert Fraction(float(blk[i, c])) == exact[j * b + i][t * b + c]
            nblk = s * (s + 1) // 2 if diag else s * (s - 1) // 2
            assert G.size == nblk * b * b


def test_gram_bruteforce_random_bf16():
    rng = np.random.default_rng(3)
    b, s, n = 5, 3, 37
    Y = oracle.bf16_round(rng.standard_normal((b * s, n)).astype(np.float32))
    for j in range(s):
        for t in range(j):
            blk32 = oracle.gram_block(Y, b, j, t, "emulate")
            blk64 = oracle.gram_block(Y, b, j, t, "fp64")
            for i in range(b):
                for c in range(b):
                    p, q = j * b + i, t * b + c
                    ex = sum(Fraction(float(Y[p, e])) * Fraction(float(Y[q, e])) for e in range(n))
                    absum = float(sum(abs(Fraction(float(Y[p, e])) * Fraction(float(Y[q, e])))
                                      for e in range(n)))
                    # FP64 sum of exact products: error <= n u64 sum|prod|
                    assert abs(float(blk64[i, c]) - float(ex)) <= n * 2.0**-53 * absum
                    assert abs(float(blk32[i, c]) - float(ex)) <= n * 2.0**-24 * absum


def test_gram_diagonal_blocks_symmetric_nonnegative():
    rng = np.random.default_rng(4)
    Y = oracle.bf16_round(rng.standard_normal((12, 9)).astype(np.float32))
    for j in range(3):
        blk = oracle.gram_block(Y, 4, j, j, "emulate")
        assert np.array_equal(blk, blk.T)
        assert np.all(np.diag(blk) >= 0)


# ------------------------------------------------------------------- margins ----
def test_margins_zero_at_w0_and_one_ulp():
    p = si.make_random(300, 23, LOGISTIC, seed=5)
    parts = oracle.outer_step(p.X, p.y, np.zeros(23, np.float32), 8, 4, 0.1, LOGISTIC, 0, 0,
                              return_parts=True)
    assert np.all(parts["r"] == 0)
    w = si.random_weights(23, seed=1, scale=1.0)
    parts = oracle.outer_step(p.X, p.y, w, 8, 4, 0.1, LOGISTIC, 0, 0, return_parts=True)
    Y64 = parts["Y"].astype(np.float64)
    r64 = Y64 @ w.astype(np.float64)
    r_near = oracle.bf16_round(r64.astype(np.float32))
    # one BF16 ulp at the magnitude of the value
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r64), 1e-30))) - 7)
    assert np.all(np.abs(parts["r"] - r_near) <= ulp + 1e-30)


# ----------------------------------------------------- recurrence and update ----
@pytest.mark.parametrize("kind", [LOGISTIC, LSQ, POISSON])
def test_ca_sgd_equals_s_sgd_steps_fp64(kind):
    p = si.make_random(301, 13, kind, seed=6)
    w0 = si.random_weights(13, seed=2, scale=0.3)
    b, s, eta, seed = 7, 5, 0.3, 11
    w_ca = w0.astype(np.float64)
    for k in range(2):
        w_ca = oracle.outer_step(p.X, p.y, w_ca, b, s, eta, kind, seed, k, mode="fp64")
    w_sgd = oracle.plain_sgd(p.X, p.y, b, 2 * s, eta, kind, seed, mode="fp64", w0=w0)
    assert np.linalg.norm(w_ca - w_sgd) <= 1e-12 * np.linalg.norm(w_sgd)


def test_s1_is_one_sgd_step():
    p = si.make_random(100, 6, LOGISTIC, seed=7)
    w0 = si.random_weights(6, seed=3)
    for k in range(3):
        w_ca = oracle.outer_step(p.X, p.y, w0, 9, 1, 0.2, LOGISTIC, 4, k, mode="fp64")
        w_sgd = oracle.plain_sgd(p.X, p.y, 9, 1, 0.2, LOGISTIC, 4, mode="fp64", w0=w0, q0=k)
        assert np.allclose(w_ca, w_sgd, rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("kind", [LOGISTIC, LSQ, POISSON])
def test_first_block_alpha_closed_form_from_zero(kind):
    p = si.make_random(200, 5, kind, seed=8)
    b, eta = 6, 0.4
    for mode in ("fp64", "emulate"):
        parts = oracle.outer_step(p.X, p.y, np.zeros(5, np.float32), b, 3, eta, kind, 1, 0,
                                  mode=mode, return_parts=True)
        yb = p.y[parts["idx"][:b]].astype(np.float64)
        if kind == LOGISTIC:
            want = eta * yb / (2 * b)
        elif kind == LSQ:
            want = eta * yb / b
        else:
            want = -eta * (1.0 - yb) / b
        tol = 1e-15 if mode == "fp64" else 2e-7
        assert np.allclose(parts["alpha"][:b], want, rtol=tol, atol=1e-12 if mode == "fp64" else 1e-8)


def test_update_is_w0_plus_Yt_alpha():
    p = si.make_random(150, 9, LSQ, seed=9)
    w0 = si.random_weights(9, seed=4)
    parts = oracle.outer_step(p.X, p.y, w0, 5, 3, 0.1, LSQ, 2, 1, mode="fp64", return_parts=True)
    Y = p.X[parts["idx"]].astype(np.float64)
    direct = w0.astype(np.float64).copy()
    for i in range(Y.shape[0]):
        direct += parts["alpha"][i] * Y[i]
    assert np.allclose(parts["w"], direct, rtol=1e-14, atol=1e-15)


def test_precision_variants_of_the_emulating_mode():
    """margins="fp32": r is the FP32 sum itself, which the recipe's r is the BF16
    rounding of; gram="bf16": the same recurrence fed bf16_round(G), so with one block
    (s = 1: no G) it changes nothing and with G it moves w by less than BF16's relative
    step.  Both variants stay within BF16 rounding of the FP64 iterate on the same
    BF16 data, and FP32 margins are the closer of the two margin choices."""
    p = si.make_random(500, 31, LOGISTIC, seed=13)
    w0 = si.random_weights(31, seed=6, scale=0.5)
    b, s, eta = 8, 6, 0.4
    base = oracle.outer_step(p.X, p.y, w0, b, s, eta, LOGISTIC, 1, 2, return_parts=True)
    m32 = oracle.outer_step(p.X, p.y, w0, b, s, eta, LOGISTIC, 1, 2, return_parts=True,
                            margins="fp32")
    assert np.array_equal(oracle.bf16_round(m32["r"]), base["r"])
    assert not np.array_equal(m32["r"], base["r"])
    ref = oracle.outer_step(p.X, p.y, w0, b, s, eta, LOGISTIC, 1, 2, mode="fp64",
                            storage="bf16")
    e_bf = np.linalg.norm(base["w"] - ref)
    e_32 = np.linalg.norm(m32["w"] - ref)
    assert e_32 < e_bf <= 1e-2 * np.linalg.norm(ref)
    one = oracle.outer_step(p.X, p.y, w0, 48, 1, eta, LOGISTIC, 1, 2)
    assert np.array_equal(one, oracle.outer_step(p.X, p.y, w0, 48, 1, eta, LOGISTIC, 1, 2,
                                                 gram="bf16"))
    gb = oracle.outer_step(p.X, p.y, w0, b, s, eta, LOGISTIC, 1, 2, gram="bf16")
    d = np.linalg.norm(gb - base["w"]) / np.linalg.norm(base["w"])
    assert 0 < d < 2.0**-8


def test_emulate_close_to_fp64_on_bf16_storage():
    p = si.make_problem(1)
    r = p.recipe
    w0 = si.random_weights(r.n, seed=5)
    we = oracle.outer_step(p.X, p.y, w0, r.b, r.s, r.eta, r.loss, 0, 0, mode="emulate")
    wd = oracle.outer_step(p.X, p.y, w0, r.b, r.s, r.eta, r.loss, 0, 0, mode="fp64", storage="bf16")
    assert np.linalg.norm(we - wd) <= 1e-3 * np.linalg.norm(wd)


def test_lsq_sgd_converges_to_lstsq_on_consistent_system():
    p = si.make_random(256, 8, LSQ, seed=10, scale=1.0)
    w_true = np.linspace(-1, 1, 8)
    y = (p.X.astype(np.float64) @ w_true).astype(np.float32)
    w_ls = np.linalg.lstsq(p.X.astype(np.float64), y.astype(np.float64), rcond=None)[0]
    w, _ = oracle.train(p.X, y, 8, 4, 0.05, LSQ, 0, 300, mode="fp64")
    assert np.linalg.norm(w - w_ls) <= 1e-4 * np.linalg.norm(w_ls)


def test_recipe1_loss_decreases():
    p = si.make_problem(1)
    r = p.recipe
    w, losses = oracle.train(p.X, p.y, r.b, r.s, r.eta, r.loss, 0, r.iters, mode="emulate",
                             loss_every=5)
    assert losses[-1] < math.log(2.0) - 0.05
    assert all(np.isfinite(losses))


@pytest.mark.parametrize("kind", [LOGISTIC, LSQ, POISSON])
def test_plain_sgd_fp32_close_to_fp64(kind):
    """The FP32 plain SGD the paper compares against is the FP64 SGD up to FP32
    rounding: after a few steps the two weight vectors agree to ~1e-5 relative (each
    step's sums carry n*u relative error), while a dropped term, a wrong sign or a
    transposed update would differ at order one."""
    p = si.make_random(600, 37, kind, seed=11)
    w64 = oracle.plain_sgd(p.X, p.y, 16, 12, 0.05, kind, 3, mode="fp64")
    w32 = oracle.plain_sgd(p.X, p.y, 16, 12, 0.05, kind, 3, mode="fp32")
    assert w32.dtype == np.float32
    rel = np.linalg.norm(w32 - w64) / np.linalg.norm(w64)
    assert 0.0 < rel < 1e-5
    # and a single FP32 step equals the FP64 step rounded, to FP32 accuracy, at w = 0
    w1 = oracle.plain_sgd(p.X, p.y, 16, 1, 0.05, kind, 3, mode="fp32")
    idx = oracle.sample_indices(p.m, 16, 3, 0)
    g0 = oracle.loss_grad(np.zeros(16), p.y[idx].astype(np.float64), kind)
    ref = p.X[idx].astype(np.float64).T @ (-(0.05 / 16) * g0)
    assert np.allclose(w1, ref, rtol=1e-5, atol=1e-7)

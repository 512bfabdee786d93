"""The seeded input recipes: deterministic, independent of how many rows are drawn, and
with the distributions their docstring states (checked at reduced row counts)."""
import numpy as np

import synth_inputs as si


def test_rows_do_not_depend_on_the_row_count_or_threads():
    # row chunk i of 16384 rows has its own stream, so a longer draw extends a shorter one
    a = si.make_problem(5, m=17000)
    b = si.make_problem(5, m=40000)
    np.testing.assert_array_equal(a.X, b.X[:17000])
    np.testing.assert_array_equal(a.w_star, b.w_star)
    c = si.make_problem(5, m=17000)
    np.testing.assert_array_equal(a.X, c.X)
    np.testing.assert_array_equal(a.y, c.y)
    assert not np.array_equal(a.X, si.make_problem(5, seed=1, m=17000).X)


def test_recipe_shapes_and_dtypes():
    for cid, m in ((1, None), (2, 600), (3, 600), (4, 600), (5, 600)):
        p = si.make_problem(cid, m=m)
        r = si.RECIPES[cid]
        assert p.X.shape == (r.m if m is None else m, r.n)
        assert p.X.dtype == np.float32 and p.y.dtype == np.float32
        assert p.X.flags.c_contiguous


def test_recipe2_scale_and_label_flips():
    p = si.make_problem(2, m=17000)
    assert abs(p.X.std() * np.sqrt(2000) - 1.0) < 0.01
    assert set(np.unique(p.y)) <= {-1.0, 1.0}
    clean = np.where(p.X.astype(np.float64) @ p.w_star >= 0, 1.0, -1.0)
    flips = np.mean(clean != p.y)
    assert abs(flips - 0.05) < 0.007  # binomial sd 0.0017 at this m


def test_recipe3_half_folded_columns_and_logistic_labels():
    p = si.make_problem(3, m=50000)
    assert (p.X[:, 9:] >= 0).all() and (p.X[:, :9] < 0).any()
    assert set(np.unique(p.y)) <= {-1.0, 1.0}
    z = p.X.astype(np.float64) @ p.w_star
    # P(y = +1 | z) = sigmoid(z): compare the mean over rows
    sig = 1.0 / (1.0 + np.exp(-z))
    assert abs(np.mean(p.y > 0) - np.mean(sig)) < 0.01
    for part in (z > 1.0, z < -1.0):  # the labels follow z's sign, not its opposite
        assert part.sum() > 1000
        assert abs(np.mean(p.y[part] > 0) - np.mean(sig[part])) < 0.03


def test_recipe4_noise_level():
    p = si.make_problem(4, m=50000)
    resid = p.y.astype(np.float64) - p.X.astype(np.float64) @ p.w_star
    assert abs(resid.std() - 0.1) < 0.003
    assert abs(resid.mean()) < 0.003


def test_recipe5_poisson_counts():
    p = si.make_problem(5, m=50000)
    assert (p.y >= 0).all() and np.array_equal(p.y, np.round(p.y))
    assert abs(p.X.std() - 0.05) < 0.001
    lam = np.exp(p.X.astype(np.float64) @ p.w_star)
    assert abs(p.y.mean() - lam.mean()) < 4 * np.sqrt(lam.mean() / p.m) + 1e-3

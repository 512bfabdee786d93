"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars (the build's contract, from the method's stated tolerances):
  * sampled row indices, BF16 storage: bit-exact;
  * G within 1e-5 relative Frobenius of the oracle's emulating mode;
  * BF16 margins r: equal, except rare one-ulp flips from a different FP32 summation
    order (each within one BF16 ulp, at most 0.5% of entries);
  * w after one outer iteration within 1e-4 relative L2 of the emulating mode, from
    w = 0 and from a seeded non-zero w;
  * loss kernel within 1e-5 relative of the oracle's FP64 loss on the same BF16 data;
  * after a full run, the final loss (FP64 on the FP32 data) within 0.5% of FP64
    plain minibatch SGD on the same rows.
"""
import math

import numpy as np
import pytest

import oracle
import synth_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GRAM_TOL = 1e-5
W_TOL = 1e-4
LOSS_TOL = 1e-5


def _len_scale(n):
    """The bars above hold for dot products up to 2048 terms (the workloads' n <= 2000).
    Beyond that they grow linearly with n: two valid FP32 summation orders of an n-term
    dot product differ by up to about 2 n u sum|x_k y_k| (u = 2^-24), so the difference
    between the GPU's accumulation order and the oracle's BLAS order grows with n
    (observed 5.4e-5 relative Frobenius for G at n = 16384)."""
    return max(1.0, n / 2048.0)


def _dev(p, casgd):
    X32 = torch.from_numpy(p.X).cuda()
    y = torch.from_numpy(p.y).cuda()
    data = casgd.Dataset.from_fp32(X32, y)
    del X32
    return data


def _run_step(casgd, data, params, w0, k=0, idx_in=None):
    ws = casgd.workspace(data, params)
    taps = casgd.Taps.alloc(params)
    taps.idx_in = idx_in
    w = torch.from_numpy(np.asarray(w0, dtype=np.float32).copy()).cuda()
    casgd.outer_step(data, params, w, k, ws, taps)
    st = casgd.get_status(ws)
    return w.cpu().numpy(), taps, st


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _bf16_ulp(v):
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0**-126)))
    return 2.0 ** (e - 7)


# --------------------------------------------------------------- storage, a1 ----
def test_store_bf16_bitexact(gpu_lib):
    casgd = gpu_lib
    rng = np.random.default_rng(0)
    for m, n in ((1000, 37), (64, 8), (3, 1), (513, 130)):
        X = (rng.standard_normal((m, n)) * 10.0 ** rng.integers(-30, 30, (m, n))).astype(np.float32)
        X[0, 0] = np.float32(1.0 + 2.0**-8)  # a tie
        out = casgd.store_bf16(torch.from_numpy(X).cuda())
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        ld = (n + 7) // 8 * 8
        assert got.shape == (m, ld)
        want = oracle.bf16_round(X).view(np.uint32) >> 16
        assert np.array_equal(got[:, :n].astype(np.uint32), want)
        assert np.all(got[:, n:] == 0)


def test_sample_indices_bitexact(gpu_lib):
    casgd = gpu_lib
    for m, count, seed, c0 in ((4096, 64, 0, 0), (400_000, 8192, 0, 49 * 8192),
                               (2**31 - 1, 100_000, 2**64 - 1, 2**40 + 7), (1, 5, 3, 0),
                               (11_000_000, 16384, 12345, 671 * 16384)):
        got = casgd.sample_indices(m, count, seed, c0).cpu().numpy()
        want = oracle.sample_indices(m, count, seed, c0)
        assert np.array_equal(got, want), (m, count, seed, c0)


def test_sample_indices_permuted_bitexact(gpu_lib):
    """Sampling without replacement: the device's keyed permutation equals the oracle's
    bit for bit, across epoch boundaries and for the largest row count; a whole epoch
    visits every row once."""
    casgd = gpu_lib
    for m, count, seed, c0 in ((4096, 4096, 0, 0), (400_000, 8192, 0, 49 * 8192),
                               (2**31 - 1, 100_000, 2**64 - 1, 2**40 + 7), (1, 5, 3, 0),
                               (11_000_000, 16384, 12345, 671 * 16384), (37, 200, 3, 85),
                               (1000, 3000, 9, 0), (5_000_000, 16384, 0, 305 * 16384)):
        got = casgd.sample_indices(m, count, seed, c0, permuted=True).cpu().numpy()
        want = oracle.permuted_indices(m, count, seed, c0)
        assert np.array_equal(got, want), (m, count, seed, c0)
    whole = casgd.sample_indices(4096, 4096, 11, 4096 * 7, permuted=True).cpu().numpy()
    assert np.array_equal(np.sort(whole), np.arange(4096))


PERM_CASES = [
    ("recipe1", lambda: si.make_problem(1), None),
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), None),
    ("ragged_777x37_b24_s3", lambda: si.make_random(777, 37, si.LOGISTIC, seed=1), (24, 3, 0.3)),
]


@pytest.mark.parametrize("name,factory,override", PERM_CASES, ids=[c[0] for c in PERM_CASES])
def test_outer_step_permuted_sampling(gpu_lib, name, factory, override):
    """CASGD_FLAG_SAMPLE_PERMUTED: the rows of an outer iteration are the oracle's
    permuted draws (bit-exact, an iteration that crosses an epoch boundary included),
    and w matches the oracle on them."""
    casgd = gpu_lib
    p = factory()
    params = _params(casgd, p, override, casgd.FLAG_SAMPLE_PERMUTED)
    b, s = params.b, params.s
    data = _dev(p, casgd)
    w0 = si.random_weights(p.n, seed=7, scale=0.5)
    k = p.m // (b * s)  # counters k*S .. k*S+S-1: past m (across it where S does not divide m)
    w_gpu, taps, st = _run_step(casgd, data, params, w0, k=k)
    assert st == 0
    ref = oracle.outer_step(p.X, p.y, w0, b, s, params.eta, p.recipe.loss, 0, k,
                            mode="emulate", return_parts=True, permuted=True)
    assert np.array_equal(taps.idx_out.cpu().numpy(), ref["idx"])
    assert _rel(w_gpu, ref["w"]) <= W_TOL * _len_scale(p.n)


# ------------------------------------------------------ one outer iteration ----
CASES = [
    # (name, problem factory, b, s, eta, loss)
    ("recipe1", lambda: si.make_problem(1), None),
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), None),
    ("recipe3_m60000", lambda: si.make_problem(3, m=60000), None),
    ("recipe4_m60000", lambda: si.make_problem(4, m=60000), None),
    ("recipe5_m20000", lambda: si.make_problem(5, m=20000), None),
    ("ragged_777x37_b24_s3", lambda: si.make_random(777, 37, si.LOGISTIC, seed=1), (24, 3, 0.3)),
    ("ragged_500x5_b7_s5", lambda: si.make_random(500, 5, si.LSQ, seed=2), (7, 5, 0.05)),
    ("ragged_3000x130_b100_s6", lambda: si.make_random(3000, 130, si.POISSON, seed=3),
     (100, 6, 0.02)),
    ("ragged_2000x200_b136_s1", lambda: si.make_random(2000, 200, si.LOGISTIC, seed=4),
     (136, 1, 0.2)),
    # limits: the widest feature count, and S = 65536 (recipe 4 at s = 32, packed G 8.3 GB)
    ("max_n16384_b64_s4", lambda: si.make_random(3000, 16384, si.LSQ, seed=5), (64, 4, 0.01)),
    ("max_S65536_recipe4_s32", lambda: si.make_problem(4, m=200_000), (2048, 32, 0.01)),
]


def _params(casgd, p, override, flags):
    r = p.recipe
    if override is None:
        b, s, eta = r.b, r.s, r.eta
    else:
        b, s, eta = override
    return casgd.Params(b, s, eta, p.recipe.loss, seed=0, flags=flags)


@pytest.mark.parametrize("gram", ["simt", "tensor", "tensor_1cta", "tensor_pair",
                                  "tensor_pair_nofuse"])
@pytest.mark.parametrize("name,factory,override", CASES, ids=[c[0] for c in CASES])
def test_outer_step_parity(gpu_lib, name, factory, override, gram):
    casgd = gpu_lib
    p = factory()
    flag = {"simt": casgd.FLAG_GRAM_SIMT, "tensor": casgd.FLAG_GRAM_TENSOR,
            "tensor_1cta": casgd.FLAG_GRAM_TENSOR | casgd.FLAG_GRAM_NO_CLUSTER,
            "tensor_pair": casgd.FLAG_GRAM_TENSOR | casgd.FLAG_GRAM_PAIR,
            "tensor_pair_nofuse": casgd.FLAG_GRAM_TENSOR | casgd.FLAG_GRAM_PAIR
            | casgd.FLAG_NO_FUSE}[gram]
    # FULL_G: every block of G is stored (the far-forming Gram has its own test)
    params = _params(casgd, p, override,
                     flag | casgd.FLAG_WRITE_DIAG_BLOCKS | casgd.FLAG_FULL_G)
    b, s = params.b, params.s
    data = _dev(p, casgd)
    for w0 in (np.zeros(p.n, np.float32), si.random_weights(p.n, seed=7, scale=0.5)):
        try:
            w_gpu, taps, st = _run_step(casgd, data, params, w0, k=3)
        except casgd.CasgdError as e:
            if gram != "simt" and e.code == 7:
                pytest.skip("tensor-core Gram does not take this shape")
            raise
        assert st == 0
        ref = oracle.outer_step(p.X, p.y, w0, b, s, params.eta, p.recipe.loss, 0, 3,
                                mode="emulate", return_parts=True)
        # a1: indices bit-exact
        assert np.array_equal(taps.idx_out.cpu().numpy(), ref["idx"])
        # a4: margins
        r_gpu = (taps.r_out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
        diff = r_gpu != ref["r"]
        assert diff.mean() <= 0.005 * _len_scale(p.n)
        assert np.all(np.abs(r_gpu - ref["r"]) <= _bf16_ulp(ref["r"]) + 1e-38)
        # a3: Gram, every block the kernel wrote (diagonal included)
        if taps.G_out.numel() <= 40_000_000:
            G_gpu = taps.G_out.cpu().numpy()
            G_ref = oracle.gram_packed(ref["Y"], b, s, diag=True, mode="emulate")
            assert _rel(G_gpu, G_ref) <= GRAM_TOL * _len_scale(p.n)
        else:  # sampled blocks: first, last, and a few in between
            rng = np.random.default_rng(0)
            blocks = {(s - 1, 0), (s - 1, s - 1), (1, 0), (0, 0)}
            for _ in range(6):
                j = int(rng.integers(0, s))
                blocks.add((j, int(rng.integers(0, j + 1))))
            num = den = 0.0
            for j, t in sorted(blocks):
                o = oracle.packed_block_offset(j, t, b, True)
                g_ref = oracle.gram_block(ref["Y"], b, j, t, "emulate").reshape(-1)
                g_gpu = taps.G_out[o:o + b * b].cpu().numpy().astype(np.float64)
                num += float(np.sum((g_gpu - g_ref) ** 2))
                den += float(np.sum(g_ref.astype(np.float64) ** 2))
            assert math.sqrt(num / den) <= GRAM_TOL * _len_scale(p.n)
        # a6: alpha (diagnostic bound, looser than w because r may flip one ulp)
        assert _rel(taps.alpha_out.cpu().numpy(), ref["alpha"]) <= 2e-3 * _len_scale(p.n)
        # a8: the weights
        assert _rel(w_gpu, ref["w"]) <= W_TOL * _len_scale(p.n)


FUSE_CASES = [
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), None),
    ("recipe5_m20000_pair", lambda: si.make_problem(5, m=20000), None),
    ("ragged_3000x130_b100_s6", lambda: si.make_random(3000, 130, si.POISSON, seed=3),
     (100, 6, 0.02)),
    ("ragged_1500x300_b40_s7", lambda: si.make_random(1500, 300, si.LOGISTIC, seed=6),
     (40, 7, 0.3)),
    ("b1024_s2_recipe3", lambda: si.make_problem(3, m=60000), (1024, 2, 0.05)),
]


@pytest.mark.parametrize("name,factory,override", FUSE_CASES, ids=[c[0] for c in FUSE_CASES])
def test_fused_launch_equals_separate_launches(gpu_lib, name, factory, override):
    """The paired-SM Gram with the recurrence in the same launch computes exactly what the
    two separate launches compute: the MMA order over K, the recurrence's sums and the
    update's partial order are the same, only the timing differs.  Bit-identical G,
    alpha and w, from a non-zero w."""
    casgd = gpu_lib
    p = factory()
    data = _dev(p, casgd)
    w0 = si.random_weights(p.n, seed=3)
    out = []
    for extra in (0, casgd.FLAG_NO_FUSE):
        params = _params(casgd, p, override, casgd.FLAG_GRAM_TENSOR | casgd.FLAG_GRAM_PAIR
                         | casgd.FLAG_FULL_G | extra)
        w, taps, st = _run_step(casgd, data, params, w0, k=3)
        assert st == 0
        G = taps.G_out.cpu().numpy() if taps.G_out.numel() <= 40_000_000 else None
        out.append((w, taps.alpha_out.cpu().numpy(), G))
    (w1, a1, G1), (w2, a2, G2) = out
    if G1 is not None:
        assert np.array_equal(G1.view(np.uint32), G2.view(np.uint32))
    assert np.array_equal(a1.view(np.uint32), a2.view(np.uint32))
    assert np.array_equal(w1.view(np.uint32), w2.view(np.uint32))


PIPE_CASES = [
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), None),
    ("recipe5_m20000", lambda: si.make_problem(5, m=20000), None),
    ("ragged_3000x130_b100_s6", lambda: si.make_random(3000, 130, si.POISSON, seed=3),
     (100, 6, 0.02)),
]


@pytest.mark.parametrize("name,factory,override", PIPE_CASES, ids=[c[0] for c in PIPE_CASES])
def test_train_pipeline_equals_outer_steps(gpu_lib, name, factory, override):
    """casgd_train computes the next iteration's Gram in the launch of the current
    recurrence (stored G); every value must still be exactly what one outer iteration
    at a time computes: bit-identical w after 3 iterations from a non-zero w, and
    after 1."""
    casgd = gpu_lib
    p = factory()
    data = _dev(p, casgd)
    params = _params(casgd, p, override, casgd.FLAG_FULL_G)
    w0 = si.random_weights(p.n, seed=7)
    for iters in (3, 1):
        ws = casgd.workspace(data, params)
        w_step = torch.from_numpy(w0.copy()).cuda()
        for k in range(iters):
            casgd.outer_step(data, params, w_step, 5 + k, ws)
        assert casgd.get_status(ws) == 0
        w_train = torch.from_numpy(w0.copy()).cuda()
        _, _, kind = casgd.train(data, params, w_train, iters, ws, k0=5)
        assert kind == (4 if iters > 1 else 3)
        a = w_step.cpu().numpy()
        b_ = w_train.cpu().numpy()
        assert np.array_equal(a.view(np.uint32), b_.view(np.uint32)), (iters, _rel(b_, a))


# ------------------------------------ far sums formed by the Gram (no far G) ----
def _band_width(b):
    """The recurrence's band width for a block size b (a multiple of 4): the blocks a
    chain lane holds in registers (documented with CASGD_FLAG_FAR_FROM_GRAM)."""
    return 3 if b <= 256 else 2 if b <= 512 else 1


FAR_CASES = [
    # the recipes' own block sizes (b = 256 .. 2048) and feature counts (18 .. 2000)
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), None),
    ("recipe3_m60000", lambda: si.make_problem(3, m=60000), None),
    ("recipe4_m60000", lambda: si.make_problem(4, m=60000), None),
    ("recipe5_m20000", lambda: si.make_problem(5, m=20000), None),
    # a ragged K tail (n = 130) and the fewest blocks with a far block (s = 5, b = 256)
    ("ragged_3000x130_b256_s5", lambda: si.make_random(3000, 130, si.POISSON, seed=3),
     (256, 5, 0.02)),
    ("ragged_2500x70_b512_s3", lambda: si.make_random(2500, 70, si.LOGISTIC, seed=8),
     (512, 3, 0.3)),
    # more than 32 far blocks per row (a chain lane adds two partials)
    ("s40_b256_12000x64", lambda: si.make_random(12000, 64, si.LSQ, seed=9), (256, 40, 0.01)),
    # the largest S (65536) at recipe 4's shape
    ("max_S65536_recipe4_s32", lambda: si.make_problem(4, m=200_000), (2048, 32, 0.01)),
    # one row part per update unit (at least 32 column chunks) with a partial last chunk
    # and s not a multiple of 8: the last block's units add the block sums to w
    ("ragged_3000x2056_b256_s5", lambda: si.make_random(3000, 2056, si.LOGISTIC, seed=5),
     (256, 5, 0.1)),
]


@pytest.mark.parametrize("name,factory,override", FAR_CASES, ids=[c[0] for c in FAR_CASES])
def test_far_from_gram_parity(gpu_lib, name, factory, override):
    """CASGD_FLAG_FAR_FROM_GRAM: the far sums come from the Gram's accumulators and only
    the band and diagonal blocks of G are stored.  Against the oracle: indices, margins,
    every stored block, alpha and w, with the bars of the stored-G path."""
    casgd = gpu_lib
    p = factory()
    params = _params(casgd, p, override,
                     casgd.FLAG_FAR_FROM_GRAM | casgd.FLAG_WRITE_DIAG_BLOCKS)
    b, s = params.b, params.s
    B = _band_width(b)
    data = _dev(p, casgd)
    for w0 in (np.zeros(p.n, np.float32), si.random_weights(p.n, seed=7, scale=0.5)):
        w_gpu, taps, st = _run_step(casgd, data, params, w0, k=3)
        assert st == 0
        ref = oracle.outer_step(p.X, p.y, w0, b, s, params.eta, p.recipe.loss, 0, 3,
                                mode="emulate", return_parts=True)
        assert np.array_equal(taps.idx_out.cpu().numpy(), ref["idx"])
        r_gpu = (taps.r_out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
        assert (r_gpu != ref["r"]).mean() <= 0.005 * _len_scale(p.n)
        assert np.all(np.abs(r_gpu - ref["r"]) <= _bf16_ulp(ref["r"]) + 1e-38)
        stored = [(j, t) for j in range(s) for t in range(max(0, j - B), j + 1)]
        if len(stored) * b * b > 20_000_000:  # sampled: first, last and a few between
            rng = np.random.default_rng(1)
            keep = {stored[0], stored[-1], (1, 0)}
            for i in rng.choice(len(stored), 6, replace=False):
                keep.add(stored[int(i)])
            stored = sorted(keep)
        num = den = 0.0
        for j, t in stored:
            o = oracle.packed_block_offset(j, t, b, True)
            g_ref = oracle.gram_block(ref["Y"], b, j, t, "emulate").reshape(-1)
            g_gpu = taps.G_out[o:o + b * b].cpu().numpy().astype(np.float64)
            num += float(np.sum((g_gpu - g_ref) ** 2))
            den += float(np.sum(g_ref.astype(np.float64) ** 2))
        assert math.sqrt(num / den) <= GRAM_TOL * _len_scale(p.n)
        assert _rel(taps.alpha_out.cpu().numpy(), ref["alpha"]) <= 2e-3 * _len_scale(p.n)
        assert _rel(w_gpu, ref["w"]) <= W_TOL * _len_scale(p.n)


FAR_PIPE_CASES = [
    # rows of n % 8 == 0 columns (at least 256) are gathered two iterations ahead inside
    # the far-forming launch; the others by a launch of their own
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), None),
    ("recipe5_m20000", lambda: si.make_problem(5, m=20000), None),
    ("recipe3_m60000", lambda: si.make_problem(3, m=60000), None),
    ("ragged_3000x130_b256_s5", lambda: si.make_random(3000, 130, si.POISSON, seed=3),
     (256, 5, 0.02)),
    ("ragged_3000x264_b256_s3", lambda: si.make_random(3000, 264, si.LOGISTIC, seed=4),
     (256, 3, 0.1)),
    ("ragged_3000x2056_b256_s5", lambda: si.make_random(3000, 2056, si.LOGISTIC, seed=5),
     (256, 5, 0.1)),
]


@pytest.mark.parametrize("name,factory,override", FAR_PIPE_CASES,
                         ids=[c[0] for c in FAR_PIPE_CASES])
def test_far_from_gram_train_equals_outer_steps(gpu_lib, name, factory, override):
    """casgd_train with the far-forming Gram stores the next iteration's band in the
    launch of this iteration's recurrence, and gathers the rows two iterations ahead
    there too (three row buffers in turn) or the next iteration's rows in a launch of
    their own; the values are those of one outer iteration at a time: bit-identical w
    after 5 iterations (every row buffer reused), after 2 and after 1, and the same again
    on a second run (the far sums are taken in a fixed order)."""
    casgd = gpu_lib
    p = factory()
    data = _dev(p, casgd)
    params = _params(casgd, p, override, casgd.FLAG_FAR_FROM_GRAM)
    w0 = si.random_weights(p.n, seed=7)
    for iters in (5, 2, 1):
        ws = casgd.workspace(data, params)
        w_step = torch.from_numpy(w0.copy()).cuda()
        for k in range(iters):
            casgd.outer_step(data, params, w_step, 5 + k, ws)
        assert casgd.get_status(ws) == 0
        a = w_step.cpu().numpy()
        for _ in range(2):
            w_train = torch.from_numpy(w0.copy()).cuda()
            _, _, kind = casgd.train(data, params, w_train, iters, ws, k0=5)
            assert kind == (6 if iters > 1 else 5)
            b_ = w_train.cpu().numpy()
            assert np.array_equal(a.view(np.uint32), b_.view(np.uint32)), (iters, _rel(b_, a))


@pytest.mark.parametrize("name,factory,override,per_iter", [
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), None, 1),
    ("recipe3_m60000", lambda: si.make_problem(3, m=60000), None, 1),
    ("ragged_3000x130_b256_s5", lambda: si.make_random(3000, 130, si.POISSON, seed=3),
     (256, 5, 0.02), 2),
], ids=lambda v: v if isinstance(v, str) else "")
def test_far_train_launches_per_iteration(gpu_lib, name, factory, override, per_iter):
    """The far-forming casgd_train: a prologue (the first rows, the first band, the
    second rows and the reset: four launches with the first shared launch), then one
    launch per outer iteration where the launch gathers the rows two ahead itself (rows
    of n % 8 == 0 and at least 512 bytes, or of at most 64 columns), else two."""
    casgd = gpu_lib
    p = factory()
    data = _dev(p, casgd)
    params = _params(casgd, p, override, 0)
    ws = casgd.workspace(data, params)
    w = torch.zeros(p.n, device="cuda")
    iters = 6
    _, launches, kind = casgd.train(data, params, w, iters, ws)
    assert kind == 6 and casgd.get_status(ws) == 0
    assert launches == 4 + per_iter * (iters - 1)


def test_train_host_equals_train_on_device_data(gpu_lib):
    """casgd_train_host copies X, y and w0 from (pinned) host buffers into the caller's
    device buffers, trains, and copies w back: bit-identical to casgd_train on the same
    data already on the device, loss history included."""
    casgd = gpu_lib
    p = si.make_problem(5, m=20000)
    r = p.recipe
    data = _dev(p, casgd)
    params = casgd.Params(r.b, r.s, r.eta, r.loss, seed=1)
    Xh = data.X.cpu().pin_memory()
    yh = data.y.cpu().pin_memory()
    dset = casgd.Dataset(torch.empty_like(data.X), torch.empty_like(data.y), p.n)
    w0 = si.random_weights(p.n, seed=12)
    wh = torch.from_numpy(w0.copy()).pin_memory()
    wdev = torch.empty(p.n, device="cuda")
    hist, _, kind = casgd.train_host(Xh, yh, wh, dset, wdev, params, 3,
                                     casgd.workspace(dset, params), k0=2, loss_every=3)
    w_ref = torch.from_numpy(w0.copy()).cuda()
    hist_ref, _, kind_ref = casgd.train(data, params, w_ref, 3, casgd.workspace(data, params),
                                        k0=2, loss_every=3)
    assert kind == kind_ref == 6
    assert np.array_equal(wh.numpy().view(np.uint32), w_ref.cpu().numpy().view(np.uint32))
    assert hist == hist_ref
    with pytest.raises(ValueError):  # device tensors are not host buffers
        casgd.train_host(data.X, yh, wh, dset, wdev, params, 1, casgd.workspace(dset, params))


def test_far_train_rows_ahead_permuted_sampling(gpu_lib):
    """The rows gathered two iterations ahead follow CASGD_FLAG_SAMPLE_PERMUTED's
    sampler too: casgd_train over 4 iterations (crossing an epoch of the 20000 rows at
    S = 8192) is bit-identical to 4 outer iterations one at a time."""
    casgd = gpu_lib
    p = si.make_problem(5, m=20000)
    r = p.recipe
    data = _dev(p, casgd)
    params = casgd.Params(r.b, r.s, r.eta, r.loss, seed=3, flags=casgd.FLAG_SAMPLE_PERMUTED)
    w0 = si.random_weights(p.n, seed=8)
    ws = casgd.workspace(data, params)
    w_step = torch.from_numpy(w0.copy()).cuda()
    for k in range(4):
        casgd.outer_step(data, params, w_step, 1 + k, ws)
    w_train = torch.from_numpy(w0.copy()).cuda()
    _, _, kind = casgd.train(data, params, w_train, 4, ws, k0=1)
    assert kind == 6 and casgd.get_status(ws) == 0
    a, b_ = w_step.cpu().numpy(), w_train.cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b_.view(np.uint32)), _rel(b_, a)


def test_far_from_gram_is_the_default(gpu_lib):
    """Without variant flags the far-forming Gram runs wherever it applies (b a multiple
    of 256), bit-identical to forcing it; FULL_G runs the stored-G launches instead."""
    casgd = gpu_lib
    p = si.make_random(3000, 130, si.POISSON, seed=3)
    data = _dev(p, casgd)
    w0 = si.random_weights(p.n, seed=7)
    out = {}
    for name, fl in (("default", 0), ("forced", casgd.FLAG_FAR_FROM_GRAM),
                     ("full", casgd.FLAG_FULL_G)):
        params = casgd.Params(256, 5, 0.02, si.POISSON, flags=fl)
        ws = casgd.workspace(data, params)
        w = torch.from_numpy(w0.copy()).cuda()
        _, _, kind = casgd.train(data, params, w, 2, ws, k0=1)
        out[name] = (kind, w.cpu().numpy())
    assert out["default"][0] == 6 and out["forced"][0] == 6 and out["full"][0] == 4
    assert np.array_equal(out["default"][1].view(np.uint32), out["forced"][1].view(np.uint32))
    assert _rel(out["full"][1], out["default"][1]) <= 1e-5


@pytest.mark.parametrize("cid,m,flags", [(2, 20000, 0), (5, 20000, 0),
                                         (5, 20000, "permuted"), (3, 60000, 0)])
def test_far_gram_gathers_rows_like_copied_rows(gpu_lib, cid, m, flags):
    """With CASGD_FLAG_GATHER_ROWS the far-forming launch reads its rows straight from X
    (the Gram's producer draws the sampled indices and gathers four rows per TMA copy; the
    margin and update units read X the same way).  By default, and with the indices given,
    the rows are first copied into Y and read from there.  All three are the same
    arithmetic on the same values, so one outer iteration agrees bit for bit (indices,
    alpha and w), and so does a pipelined casgd_train of three iterations."""
    casgd = gpu_lib
    p = si.make_problem(cid, m=m)
    r = p.recipe
    fl = casgd.FLAG_SAMPLE_PERMUTED if flags == "permuted" else 0
    pg = casgd.Params(r.b, r.s, r.eta, r.loss, seed=5, flags=fl | casgd.FLAG_GATHER_ROWS)
    pc = casgd.Params(r.b, r.s, r.eta, r.loss, seed=5, flags=fl)
    data = _dev(p, casgd)
    w0 = si.random_weights(p.n, seed=8, scale=0.3)
    w_g, taps_g, st = _run_step(casgd, data, pg, w0, k=2)            # rows from X
    assert st == 0
    w_c, taps_c, st = _run_step(casgd, data, pc, w0, k=2)            # rows copied into Y
    assert st == 0
    w_i, taps_i, st = _run_step(casgd, data, pg, w0, k=2, idx_in=taps_g.idx_out)  # given
    assert st == 0
    for w_, t_ in ((w_c, taps_c), (w_i, taps_i)):
        assert np.array_equal(t_.idx_out.cpu().numpy(), taps_g.idx_out.cpu().numpy())
        assert np.array_equal(t_.alpha_out.cpu().numpy().view(np.uint32),
                              taps_g.alpha_out.cpu().numpy().view(np.uint32))
        assert np.array_equal(w_.view(np.uint32), w_g.view(np.uint32))
    ref = oracle.outer_step(p.X, p.y, w0, r.b, r.s, r.eta, r.loss, 5, 2, mode="emulate",
                            permuted=bool(fl))
    assert _rel(w_g, ref) <= W_TOL
    out = []
    for params in (pg, pc):
        ws = casgd.workspace(data, params)
        w = torch.from_numpy(w0.copy()).cuda()
        _, _, kind = casgd.train(data, params, w, 3, ws, k0=1)
        assert kind == 6 and casgd.get_status(ws) == 0
        out.append(w.cpu().numpy())
    assert np.array_equal(out[0].view(np.uint32), out[1].view(np.uint32))


def test_far_from_gram_unsupported_shapes(gpu_lib):
    """The flag needs b a multiple of 256, s >= 2 and the paired kernel in the same
    launch; anything else is CASGD_ERR_UNSUPPORTED and launches nothing."""
    casgd = gpu_lib
    p = si.make_random(3000, 130, si.LOGISTIC, seed=3)
    data = _dev(p, casgd)
    for b, s, extra in ((100, 6, 0), (256, 1, 0), (256, 4, casgd.FLAG_NO_FUSE),
                        (256, 4, casgd.FLAG_GRAM_SIMT), (256, 4, casgd.FLAG_GRAM_NO_CLUSTER),
                        (256, 4, casgd.FLAG_FULL_G)):
        params = casgd.Params(b, s, 0.1, si.LOGISTIC, flags=casgd.FLAG_FAR_FROM_GRAM | extra)
        ws = casgd.workspace(data, params)
        w = torch.zeros(p.n, device="cuda")
        with pytest.raises(casgd.CasgdError) as e:
            casgd.outer_step(data, params, w, 0, ws)
        assert e.value.code == 7
        torch.cuda.synchronize()
        assert torch.count_nonzero(w).item() == 0


# ------------------------------------------------- precision variants (f3) ----
PREC_CASES = [
    # far-forming Gram (b = 256), stored-G pair launch (b = 100), CUDA-core Gram
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), None, 0),
    ("ragged_3000x130_b100_s6", lambda: si.make_random(3000, 130, si.POISSON, seed=3),
     (100, 6, 0.02), 0),
    ("ragged_777x37_b24_s3_simt", lambda: si.make_random(777, 37, si.LOGISTIC, seed=1),
     (24, 3, 0.3), "simt"),
]


@pytest.mark.parametrize("variant", ["margins_fp32", "g_bf16", "both"])
@pytest.mark.parametrize("name,factory,override,gram", PREC_CASES,
                         ids=[c[0] for c in PREC_CASES])
def test_precision_variants_parity(gpu_lib, name, factory, override, gram, variant):
    """CASGD_FLAG_MARGINS_FP32 / CASGD_FLAG_G_BF16 against the oracle's emulating mode
    with the same choice: FP32 margins within FP32 summation order, G blocks the BF16
    rounding of the oracle's (one-ulp flips where the FP32 sums straddle a rounding
    boundary), alpha and w with the recipe's bars; and each variant changes w."""
    casgd = gpu_lib
    p = factory()
    fl = casgd.FLAG_WRITE_DIAG_BLOCKS | (casgd.FLAG_GRAM_SIMT if gram == "simt" else 0)
    m32 = variant in ("margins_fp32", "both")
    gbf = variant in ("g_bf16", "both")
    vfl = (casgd.FLAG_MARGINS_FP32 if m32 else 0) | (casgd.FLAG_G_BF16 if gbf else 0)
    params = _params(casgd, p, override, fl | vfl)
    b, s = params.b, params.s
    data = _dev(p, casgd)
    w0 = si.random_weights(p.n, seed=7, scale=0.5)
    w_gpu, taps, st = _run_step(casgd, data, params, w0, k=3)
    assert st == 0
    ref = oracle.outer_step(p.X, p.y, w0, b, s, params.eta, p.recipe.loss, 0, 3,
                            mode="emulate", return_parts=True,
                            margins="fp32" if m32 else "bf16", gram="bf16" if gbf else "fp32")
    assert np.array_equal(taps.idx_out.cpu().numpy(), ref["idx"])
    if m32:
        r_gpu = taps.r_out.cpu().numpy().view(np.float32)
        assert r_gpu.shape == ref["r"].shape
        assert np.all(np.abs(r_gpu - ref["r"]) <= 1e-5 * np.abs(ref["r"]) + 1e-6)
    else:
        r_gpu = (taps.r_out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
        assert np.all(np.abs(r_gpu - ref["r"]) <= _bf16_ulp(ref["r"]) + 1e-38)
    # blocks every path stores: the diagonal and the first band block
    for j in range(s):
        for t in ([j - 1, j] if j > 0 else [j]):
            o = oracle.packed_block_offset(j, t, b, True)
            g_ref = oracle.gram_block(ref["Y"], b, j, t, "emulate").reshape(-1)
            g_gpu = taps.G_out[o:o + b * b].cpu().numpy()
            if gbf:
                # the GPU rounds its own FP32 sum, within the summation-order bound
                # d = 2 n u sum_k |y_ik y_tk| of the oracle's: |g - g_ref| <= d + ulp/2
                Yj = np.abs(ref["Y"][j * b:(j + 1) * b].astype(np.float64))
                Yt = np.abs(ref["Y"][t * b:(t + 1) * b].astype(np.float64))
                d = (2.0 * p.n * 2.0**-24) * (Yj @ Yt.T).reshape(-1)
                g64 = g_ref.astype(np.float64)
                assert np.all(np.abs(g_gpu - g64) <= d + 0.5 * _bf16_ulp(np.abs(g64) + d) + 1e-30)
                assert np.mean(g_gpu != oracle.bf16_round(g_ref)) <= 0.01
                assert np.array_equal(oracle.bf16_round(g_gpu), g_gpu)  # BF16 values
            else:
                assert _rel(g_gpu, g_ref) <= GRAM_TOL * _len_scale(p.n)
    assert _rel(taps.alpha_out.cpu().numpy(), ref["alpha"]) <= 2e-3 * _len_scale(p.n)
    assert _rel(w_gpu, ref["w"]) <= W_TOL * _len_scale(p.n)
    w_rec, _, st = _run_step(casgd, data, _params(casgd, p, override, fl), w0, k=3)
    assert st == 0 and not np.array_equal(w_rec, w_gpu)


def test_outer_step_given_indices_and_bad_index(gpu_lib):
    casgd = gpu_lib
    p = si.make_problem(1)
    params = casgd.Params(16, 4, 0.1, si.LOGISTIC)
    data = _dev(p, casgd)
    idx = np.arange(64, dtype=np.int32) * 7 % p.m
    w0 = si.random_weights(p.n, seed=3)
    w_gpu, taps, st = _run_step(casgd, data, params, w0, idx_in=torch.from_numpy(idx).cuda())
    assert st == 0
    ref = oracle.outer_step(p.X, p.y, w0, 16, 4, 0.1, si.LOGISTIC, 0, 0, idx=idx)
    assert _rel(w_gpu, ref) <= W_TOL
    bad = idx.copy()
    bad[5] = p.m          # one past the end
    bad[9] = -1
    _, _, st = _run_step(casgd, data, params, w0, idx_in=torch.from_numpy(bad).cuda())
    assert st == 6        # CASGD_ERR_BAD_INDEX


def test_deterministic(gpu_lib):
    casgd = gpu_lib
    p = si.make_problem(5, m=30000)
    r = p.recipe
    data = _dev(p, casgd)
    params = casgd.Params(r.b, r.s, r.eta, r.loss)
    outs = []
    for _ in range(2):
        ws = casgd.workspace(data, params)
        w = torch.zeros(p.n, device="cuda")
        casgd.train(data, params, w, 3, ws)
        outs.append(w.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


# ---------------------------------------------------------------------- loss ----
@pytest.mark.parametrize("kind,m,n", [(si.LOGISTIC, 10_001, 64), (si.LSQ, 5000, 28),
                                      (si.POISSON, 3001, 512), (si.LOGISTIC, 777, 2000),
                                      (si.LSQ, 1, 3), (si.LSQ, 300, 4100),
                                      (si.LOGISTIC, 4099, 12)])
def test_loss_kernel_parity(gpu_lib, kind, m, n):
    casgd = gpu_lib
    p = si.make_random(m, n, kind, seed=11)
    data = _dev(p, casgd)
    params = casgd.Params(1, 1, 0.1, kind)
    ws = casgd.workspace(data, params)
    for w in (np.zeros(n, np.float32), si.random_weights(n, seed=2, scale=1.0)):
        got = casgd.loss(data, kind, torch.from_numpy(w).cuda(), ws)
        want = oracle.full_loss(oracle.bf16_round(p.X), p.y, w, kind)
        assert abs(got - want) <= LOSS_TOL * abs(want)


# ------------------------------------------------------------ full training ----
@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_final_loss_within_half_percent_of_fp64_sgd(gpu_lib, cid):
    casgd = gpu_lib
    p = si.make_problem(cid)
    r = p.recipe
    iters = r.outer_iters()
    data = _dev(p, casgd)
    params = casgd.Params(r.b, r.s, r.eta, r.loss)
    ws = casgd.workspace(data, params)
    w = torch.zeros(p.n, device="cuda")
    hist, launches, _ = casgd.train(data, params, w, iters, ws, loss_every=iters)
    assert len(hist) == 1
    assert launches >= iters
    w_gpu = w.cpu().numpy()
    assert np.all(np.isfinite(w_gpu))
    f_gpu = oracle.full_loss(p.X, p.y, w_gpu, r.loss)
    w_sgd = oracle.plain_sgd(p.X, p.y, r.b, iters * r.s, r.eta, r.loss, 0, mode="fp64")
    f_ref = oracle.full_loss(p.X, p.y, w_sgd, r.loss)
    assert abs(f_gpu - f_ref) / f_ref < 0.005
    # the device loss kernel agrees with the oracle on the BF16 data at the final w
    assert abs(hist[-1] - oracle.full_loss(oracle.bf16_round(p.X), p.y, w_gpu, r.loss)) \
        <= LOSS_TOL * abs(hist[-1])


def test_chain_trace_timeline(gpu_lib):
    """The opt-in chain timeline (CASGD_FLAG_TRACE_CHAIN, casgd_chain_trace): per phase,
    start <= loads issued <= inputs final <= alpha stored, phases in order, and the
    summary row records the Gram's last tile, the last far sum and the last update
    partial of a launch shared with the Gram (recipe 2 shape, one outer iteration)."""
    casgd = gpu_lib
    p = si.make_problem(2, m=20000)
    r = p.recipe
    data = _dev(p, casgd)
    params = casgd.Params(r.b, r.s, r.eta, r.loss, flags=casgd.FLAG_TRACE_CHAIN)
    ws = casgd.workspace(data, params)
    w = torch.zeros(p.n, device="cuda")
    casgd.outer_step(data, params, w, 0, ws)
    assert casgd.get_status(ws) == 0
    tr = np.array(casgd.chain_trace(data, params, ws), dtype=np.uint64).astype(np.int64)
    assert tr.shape == (r.s + 1, 4)
    ph = tr[: r.s]
    assert np.all(ph > 0)
    assert np.all(np.diff(ph, axis=1) >= 0)               # within a phase
    assert np.all(ph[1:, 0] >= ph[:-1, 3])                # phases in order
    gram_end, far_end, upd_end, zero = tr[r.s]
    assert zero == 0 and gram_end > ph[0, 0] and far_end > ph[0, 0]
    assert upd_end >= ph[r.s - 1, 3]                      # the last block's update follows it
    span_us = (upd_end - ph[0, 0]) / 1e3
    assert 1.0 < span_us < 1e5


SGD_CASES = [
    # (name, factory, b, steps, eta)
    ("recipe1", lambda: si.make_problem(1), 16, 40, 0.1),
    ("recipe2_m20000", lambda: si.make_problem(2, m=20000), 256, 24, 0.5),
    ("recipe5_m20000", lambda: si.make_problem(5, m=20000), 512, 10, 0.01),
    ("ragged_777x37_b24", lambda: si.make_random(777, 37, si.LOGISTIC, seed=1), 24, 30, 0.3),
    ("ragged_500x5_b7_lsq", lambda: si.make_random(500, 5, si.LSQ, seed=2), 7, 50, 0.05),
]


@pytest.mark.parametrize("name,factory,b,steps,eta", SGD_CASES, ids=[c[0] for c in SGD_CASES])
def test_sgd_fp32_matches_oracle(gpu_lib, name, factory, b, steps, eta):
    """FP32 plain minibatch SGD on the GPU against the oracle's FP32 plain SGD on the
    same rows (sampled with the same counters), from a non-zero w, and continued from
    a later step (q0)."""
    casgd = gpu_lib
    p = factory()
    X = torch.from_numpy(p.X).cuda()
    y = torch.from_numpy(p.y).cuda()
    w0 = si.random_weights(p.n, seed=5)
    params = casgd.Params(b, 1, eta, p.recipe.loss, seed=2)
    ws = casgd.sgd_workspace(b)
    w = torch.from_numpy(w0.copy()).cuda()
    casgd.sgd_fp32(X, y, params, w, steps, ws, q0=3)
    assert casgd.get_status(ws) == 0
    want = oracle.plain_sgd(p.X, p.y, b, steps, eta, p.recipe.loss, 2, mode="fp32", w0=w0, q0=3)
    assert _rel(w.cpu().numpy(), want) <= W_TOL * _len_scale(p.n)


def test_sgd_fp32_permuted_sampling(gpu_lib):
    """The FP32 SGD baseline draws the same permuted rows as CA-SGD."""
    casgd = gpu_lib
    p = si.make_random(777, 37, si.LOGISTIC, seed=1)
    X = torch.from_numpy(p.X).cuda()
    y = torch.from_numpy(p.y).cuda()
    w0 = si.random_weights(p.n, seed=5)
    params = casgd.Params(24, 1, 0.3, p.recipe.loss, seed=2, flags=casgd.FLAG_SAMPLE_PERMUTED)
    ws = casgd.sgd_workspace(24)
    w = torch.from_numpy(w0.copy()).cuda()
    casgd.sgd_fp32(X, y, params, w, 70, ws, q0=3)  # 1680 draws: past two epochs
    assert casgd.get_status(ws) == 0
    want = oracle.plain_sgd(p.X, p.y, 24, 70, 0.3, p.recipe.loss, 2, mode="fp32", w0=w0, q0=3,
                            permuted=True)
    assert _rel(w.cpu().numpy(), want) <= W_TOL * _len_scale(p.n)

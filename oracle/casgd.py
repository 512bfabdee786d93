"""Plain, slow CPU statement of one CA-SGD outer iteration and its pieces.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
GPUs, abstract.  It fixes the method in prose:
  * s minibatch steps of b rows are batched into one outer iteration whose only
    collective is the sum of one sb x sb Gram matrix (CA-SGD);
  * the recipe stores the input matrix and the margin vector in low precision
    (BF16), forms the Gram matrix from BF16 inputs with high-precision (FP32)
    accumulation, and runs the inner recurrence and the weight update in high
    precision (FP32);
  * the models are logistic, linear (least-squares) and Poisson regression.

Two arithmetic modes:
  mode="fp64"     everything in FP64 from the FP32 data (storage="fp32"), or from
                  the BF16-rounded data (storage="bf16"); margins not rounded.
  mode="emulate"  the recipe: BF16 storage of X, FP32 Gram and margin sums, margins
                  rounded once to BF16, FP32 recurrence and update.
Sums use NumPy matmul (a library primitive) in the mode's precision.

Readings of points the abstract leaves open (each is listed in the design notes):
  sampling     rows drawn with replacement; the row of slot i of block j in outer
               iteration k uses generator counter c = k*s*b + j*b + i, i.e. the c-th
               output h of SplitMix64 seeded with `seed`, reduced to [0, m) as
               ((h >> 32) * m) >> 32.  Step q of plain SGD uses counters q*b .. q*b+b-1,
               so CA-SGD and plain SGD see the same rows.  Variant (without
               replacement): counter c is position c mod m of epoch c div m of a keyed
               pseudorandom permutation of the rows (permuted_indices).
  losses       logistic l = log(1 + exp(-y z)), y in {-1, +1}; least squares
               l = (z - y)^2 / 2; Poisson (log link) l = exp(z) - y z, the log(y!)
               constant left out.  No regulariser, no intercept; f = mean over rows.
  step         alpha_j = -(eta / b) * l'(z_j, y_j) with -(eta/b) formed in the mode's
               precision; constant eta; w0 = 0 unless given.
  BF16         round to nearest, ties to even, subnormals kept.
"""
from __future__ import annotations

import numpy as np

LOGISTIC, LSQ, POISSON = 0, 1, 2

_U64 = np.uint64
_GAMMA = _U64(0x9E3779B97F4A7C15)   # SplitMix64 increment (golden ratio * 2^64, odd)
_MIX1 = _U64(0xBF58476D1CE4E5B9)
_MIX2 = _U64(0x94D049BB133111EB)


# ----------------------------------------------------------------------------------
# Sampling (the abstract: s minibatches of b rows; scheme not stated -> reading above)
# ----------------------------------------------------------------------------------
def splitmix64(seed: int, counter) -> np.ndarray:
    """The `counter`-th (0-based) output of SplitMix64 started from state `seed`.

    SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014; variant 13 mixing constants): the state advances by
    the odd constant gamma, and each output is the state passed through two
    xor-shift-multiply rounds and a final xor-shift.  Being a pure function of
    state = seed + (counter + 1) * gamma (mod 2^64), it can be evaluated at any
    counter directly.
    """
    c = np.asarray(counter, dtype=_U64)
    with np.errstate(over="ignore"):
        z = _U64(seed) + (c + _U64(1)) * _GAMMA
        z = (z ^ (z >> _U64(30))) * _MIX1
        z = (z ^ (z >> _U64(27))) * _MIX2
        return z ^ (z >> _U64(31))


def sample_indices(m: int, count: int, seed: int, counter0: int) -> np.ndarray:
    """Row indices for generator counters counter0 .. counter0+count-1, in [0, m).

    Outer iteration k uses counter0 = k*s*b.  The top 32 bits of each output are
    mapped to [0, m) by a multiply and a shift (Lemire's multiply-shift reduction).
    """
    if not (0 < m < 2**31):
        raise ValueError("m must be in [1, 2^31)")
    h = splitmix64(seed, np.arange(count, dtype=_U64) + _U64(counter0))
    return ((h >> _U64(32)) * _U64(m) >> _U64(32)).astype(np.int64)


# Sampling without replacement (a variant: every row once per epoch of m draws).
# A keyed pseudorandom permutation of [0, m) built from published pieces:
#   * a balanced Feistel network (Luby & Rackoff, "How to construct pseudorandom
#     permutations from pseudorandom functions", SIAM J. Comput. 1988) on d-bit values,
#     d the smallest even width with 2^d >= m (at least 2): halves of h = d/2 bits,
#     four rounds (L, R) -> (R, L xor F_r(R));
#   * round function F_r(R) = the low h bits of SplitMix64 output number R of the stream
#     started at state K_{e,r}, the round key K_{e,r} = SplitMix64 output number 4e + r
#     of the stream started at seed xor 0x6A09E667F3BCC908 (a fixed constant that keeps
#     the keys apart from the with-replacement stream);
#   * cycle walking (Black & Rogaway, "Ciphers with arbitrary finite domains", CT-RSA
#     2002): apply the d-bit permutation until the value falls in [0, m); this is a
#     permutation of [0, m) because the walk stays on the cycle of its start.
_PERM_SEED_XOR = 0x6A09E667F3BCC908
_PERM_ROUNDS = 4


def perm_width(m: int) -> int:
    """d: the smallest even bit width with 2^d >= m, at least 2."""
    d = 2
    while (1 << d) < m:
        d += 2
    return d


def feistel(x, d: int, keys) -> np.ndarray:
    """The d-bit Feistel permutation with the given round keys, on uint64 values."""
    h = d // 2
    mask = _U64((1 << h) - 1)
    x = np.asarray(x, dtype=_U64)
    L, R = x >> _U64(h), x & mask
    for k in keys:
        L, R = R, L ^ (splitmix64(int(k), R) & mask)
    return (L << _U64(h)) | R


def epoch_keys(seed: int, e: int) -> list:
    """Round keys K_{e,0..3} of epoch e."""
    base = (seed ^ _PERM_SEED_XOR) & 0xFFFFFFFFFFFFFFFF
    return [int(splitmix64(base, _PERM_ROUNDS * e + r)) for r in range(_PERM_ROUNDS)]


def permuted_indices(m: int, count: int, seed: int, counter0: int) -> np.ndarray:
    """Row indices for counters counter0 .. counter0+count-1 without replacement within
    each epoch: counter c is position c mod m of the permutation of epoch c div m."""
    if not (0 < m < 2**31):
        raise ValueError("m must be in [1, 2^31)")
    d = perm_width(m)
    c = np.arange(count, dtype=np.int64) + int(counter0)
    out = np.empty(count, dtype=np.int64)
    for e in np.unique(c // m):
        sel = (c // m) == e
        keys = epoch_keys(seed, int(e))
        y = feistel(c[sel] % m, d, keys)
        while True:  # cycle walking
            over = y >= _U64(m)
            if not over.any():
                break
            y[over] = feistel(y[over], d, keys)
        out[sel] = y.astype(np.int64)
    return out


def draw_indices(m: int, count: int, seed: int, counter0: int, permuted: bool = False):
    """sample_indices (with replacement) or permuted_indices (without)."""
    if permuted:
        return permuted_indices(m, count, seed, counter0)
    return sample_indices(m, count, seed, counter0)


# ----------------------------------------------------------------------------------
# Low-precision storage (the abstract: input matrix and margins stored in BF16)
# ----------------------------------------------------------------------------------
def bf16_round(x) -> np.ndarray:
    """Round FP32 values to the nearest BF16 value, ties to even; returns FP32.

    BF16 keeps the top 16 bits of an IEEE binary32.  Round to nearest even: add
    0x7FFF plus the lowest kept bit, then clear the low 16 bits (a carry into the
    exponent is the correct rounding up, up to infinity).  Finite inputs only.
    """
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> _U64(16)) & _U64(1)
    u = ((u + _U64(0x7FFF) + keep_lsb) >> _U64(16)) << _U64(16)
    return (u & _U64(0xFFFFFFFF)).astype(np.uint32).view(np.float32).reshape(a.shape)


# ----------------------------------------------------------------------------------
# GLM losses (the abstract: logistic, linear and Poisson problems)
# ----------------------------------------------------------------------------------
def loss_value(z, y, kind: int):
    """Per-row loss l(z, y) in the dtype of z (forms in the module docstring)."""
    z = np.asarray(z)
    y = np.asarray(y, dtype=z.dtype)
    with np.errstate(over="ignore"):
        if kind == LOGISTIC:
            return np.logaddexp(z.dtype.type(0), -y * z)
        if kind == LSQ:
            d = z - y
            return z.dtype.type(0.5) * d * d
        if kind == POISSON:
            return np.exp(z) - y * z
    raise ValueError(kind)


def loss_grad(z, y, kind: int):
    """dl/dz in the dtype of z.

    logistic: -y / (1 + exp(y z)) (finite for every z: 1/(1+inf) = 0);
    least squares: z - y;  Poisson: exp(z) - y.
    """
    z = np.asarray(z)
    y = np.asarray(y, dtype=z.dtype)
    one = z.dtype.type(1)
    with np.errstate(over="ignore"):
        if kind == LOGISTIC:
            return -y / (one + np.exp(y * z))
        if kind == LSQ:
            return z - y
        if kind == POISSON:
            return np.exp(z) - y
    raise ValueError(kind)


def full_loss(X, y, w, kind: int, chunk_elems: int = 1 << 22) -> float:
    """f(w) = (1/m) sum_i l(x_i . w, y_i), evaluated in FP64 (X taken as given)."""
    X = np.asarray(X)
    m = X.shape[0]
    w64 = np.asarray(w, dtype=np.float64)
    y64 = np.asarray(y, dtype=np.float64)
    rows = max(1, chunk_elems // max(1, X.shape[1]))
    total = 0.0
    for a in range(0, m, rows):
        z = X[a:a + rows].astype(np.float64) @ w64
        total += float(np.sum(loss_value(z, y64[a:a + rows], kind)))
    return total / m


# ----------------------------------------------------------------------------------
# Gram matrix (the abstract: one sb x sb Gram matrix per outer iteration)
# ----------------------------------------------------------------------------------
def _mode_dtype(mode: str):
    if mode == "emulate":
        return np.float32
    if mode == "fp64":
        return np.float64
    raise ValueError(mode)


def gram_block(Y, b: int, j: int, t: int, mode: str = "emulate") -> np.ndarray:
    """G_{j,t} = Y_j Y_t^T (b x b) where Y_j = rows j*b .. j*b+b-1 of Y.

    In emulate mode the products of two BF16 values are exact in FP32 and are
    summed in FP32; in fp64 mode everything is FP64.
    """
    ft = _mode_dtype(mode)
    Yj = np.asarray(Y[j * b:(j + 1) * b], dtype=ft)
    Yt = np.asarray(Y[t * b:(t + 1) * b], dtype=ft)
    return Yj @ Yt.T


def packed_block_offset(j: int, t: int, b: int, diag: bool) -> int:
    """Element offset of block (j, t) in the packed block-lower layout.

    Blocks are stored row-major (b x b each) in the order j ascending, then t
    ascending, for t < j (strict) or t <= j (diag=True).
    """
    if diag:
        return (j * (j + 1) // 2 + t) * b * b
    return (j * (j - 1) // 2 + t) * b * b


def gram_packed(Y, b: int, s: int, diag: bool = False, mode: str = "emulate") -> np.ndarray:
    """All blocks the recurrence can read (t < j), plus the diagonal if asked,
    in the packed block-lower layout (small cases only)."""
    ft = _mode_dtype(mode)
    nblk = s * (s + 1) // 2 if diag else s * (s - 1) // 2
    out = np.zeros(nblk * b * b, dtype=ft)
    for j in range(s):
        for t in range(j + 1 if diag else j):
            o = packed_block_offset(j, t, b, diag)
            out[o:o + b * b] = gram_block(Y, b, j, t, mode).reshape(-1)
    return out


# ----------------------------------------------------------------------------------
# One outer iteration
# ----------------------------------------------------------------------------------
def gather_rows(X, idx, mode: str, storage: str | None = None) -> np.ndarray:
    """Y = rows idx of the stored matrix, as values of the mode's dtype.

    emulate: storage is BF16 (always).  fp64: storage 'fp32' (default) or 'bf16'.
    """
    rows = np.asarray(X)[np.asarray(idx)]
    if mode == "emulate":
        return bf16_round(rows.astype(np.float32))
    st = storage or "fp32"
    if st == "bf16":
        return bf16_round(rows.astype(np.float32)).astype(np.float64)
    return rows.astype(np.float64)


def outer_step(X, y, w, b: int, s: int, eta: float, kind: int, seed: int, k: int,
               mode: str = "emulate", storage: str | None = None, idx=None,
               return_parts: bool = False, permuted: bool = False,
               margins: str = "bf16", gram: str = "fp32"):
    """One CA-SGD outer iteration: s minibatch SGD steps of b rows, batched.

    Derivation (pins the recurrence).  Minibatch SGD on f(w) = (1/m) sum l(x.w, y)
    with batch Y_j is w_{j+1} = w_j - (eta/b) Y_j^T l'(Y_j w_j, y_j) = w_j + Y_j^T a_j.
    Unrolled, w_j = w_0 + sum_{t<j} Y_t^T a_t, hence
        Y_j w_j = Y_j w_0 + sum_{t<j} (Y_j Y_t^T) a_t = r_j + sum_{t<j} G_{j,t} a_t,
    and after s steps w_s = w_0 + Y^T a.  Steps, in order:
      1. idx: S = s*b row indices for counters k*S .. k*S+S-1;
      2. Y = X[idx] (BF16 storage in emulate mode), y_Y = y[idx];
      3. r = Y w_0 (FP32 sum then one BF16 rounding in emulate mode);
      4. for j = 0..s-1:  z_j = r_j + sum_{t<j} G_{j,t} a_t,  a_j = -(eta/b) l'(z_j, y_j)
         with G_{j,t} = Y_j Y_t^T;
      5. w = w_0 + Y^T a.
    Returns w (mode dtype), or a dict with idx, Y, r, alpha, w when return_parts.

    Two other precision choices of the emulating mode (the abstract studies several
    and lists none; these vary one each): margins="fp32" keeps r as its FP32 sum (no
    BF16 rounding); gram="bf16" rounds every entry of G to BF16 (nearest even) before
    the recurrence uses it, as when G is summed across processes in BF16.
    """
    ft = _mode_dtype(mode)
    X = np.asarray(X)
    m = X.shape[0]
    S = s * b
    if idx is None:
        idx = draw_indices(m, S, seed, k * S, permuted)
    idx = np.asarray(idx, dtype=np.int64)
    Y = gather_rows(X, idx, mode, storage)
    yY = np.asarray(y, dtype=np.float32)[idx].astype(ft)
    # the weights stay FP32 in the recipe; fp64 mode takes them as given
    w0 = np.asarray(w).astype(np.float32).astype(ft) if mode == "emulate" \
        else np.asarray(w, dtype=np.float64)

    r = Y @ w0
    if mode == "emulate" and margins == "bf16":
        r = bf16_round(r)                       # margins stored in low precision

    coef = -(ft(eta) / ft(b))
    alpha = np.zeros(S, dtype=ft)
    for j in range(s):
        rows = slice(j * b, (j + 1) * b)
        z = r[rows].astype(ft)
        for t in range(j):
            cols = slice(t * b, (t + 1) * b)
            G_jt = gram_block(Y, b, j, t, mode)
            if mode == "emulate" and gram == "bf16":
                G_jt = bf16_round(G_jt)
            z = z + G_jt @ alpha[cols]
        alpha[rows] = coef * loss_grad(z, yY[rows], kind)

    w_new = w0 + Y.T @ alpha
    if return_parts:
        return {"idx": idx, "Y": Y, "r": r, "alpha": alpha, "w": w_new}
    return w_new


def train(X, y, b: int, s: int, eta: float, kind: int, seed: int, iters: int,
          mode: str = "emulate", storage: str | None = None, w0=None, k0: int = 0,
          loss_every: int = 0, loss_X=None, permuted: bool = False):
    """`iters` outer iterations k = k0 .. k0+iters-1 from w0 (zeros by default).

    Returns (w, losses) where losses holds f(w) (FP64, on `loss_X` or X) after every
    `loss_every`-th iteration when loss_every > 0.
    """
    X = np.asarray(X)
    w = np.zeros(X.shape[1], dtype=np.float32) if w0 is None else np.asarray(w0)
    losses = []
    for it in range(iters):
        w = outer_step(X, y, w, b, s, eta, kind, seed, k0 + it, mode=mode, storage=storage,
                       permuted=permuted)
        if mode == "emulate":
            w = np.asarray(w, dtype=np.float32)
        if loss_every and (it + 1) % loss_every == 0:
            losses.append(full_loss(X if loss_X is None else loss_X, y, w, kind))
    return w, losses


def plain_sgd(X, y, b: int, steps: int, eta: float, kind: int, seed: int,
              mode: str = "fp64", w0=None, q0: int = 0, permuted: bool = False):
    """Plain minibatch SGD, one step per minibatch, on the same rows as CA-SGD.

    Step q (q = q0 .. q0+steps-1) uses counters q*b .. q*b+b-1 and does
    w <- w - (eta/b) Y_q^T l'(Y_q w, y_q).  mode "fp64": FP64 on the FP32 data;
    "fp32": FP32 on the FP32 data (the FP32 SGD the paper compares against).
    """
    ft = np.float64 if mode == "fp64" else np.float32
    X = np.asarray(X)
    m = X.shape[0]
    w = (np.zeros(X.shape[1]) if w0 is None else np.asarray(w0)).astype(ft)
    coef = -(ft(eta) / ft(b))
    yv = np.asarray(y, dtype=np.float32)
    for q in range(q0, q0 + steps):
        idx = draw_indices(m, b, seed, q * b, permuted)
        Yq = X[idx].astype(ft)
        g = loss_grad(Yq @ w, yv[idx].astype(ft), kind)
        w = w + Yq.T @ (coef * g)
    return w

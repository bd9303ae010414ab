"""CPU check of the accuracy argument behind the f16 tensor-core routes.

The 4-bit prefill GEMM, MUL_MAT_ID and the Q8 GEMM above the decode sizes form
each weight once in f16 (round to nearest even) and convert each activation
row to f16 after a power-of-two scale that puts the row's largest magnitude
in [2^14, 2^15).  The claim: for weights in f16's normal range the weight
rounding costs at most 2^-11 of sum_k |x||w|, and the activation conversion
costs nothing for elements within 2^31 of their row's largest.

This file emulates that arithmetic with numpy's float16 (exact products and
sums in fp64, so only the two roundings remain) and checks the claim against
the oracle on random and on adversarial inputs.  It also shows that the
adversarial inputs defeat one bf16 rounding per weight, which the earlier
route took, so the GPU tests built on them have teeth."""
import numpy as np

import oracle.qmm_oracle as O


def f16_weights(tiles, N, K):
    q, s, m = O.q4_blocks_from_tiles(tiles, N, K)
    w = q.astype(np.float64) * np.repeat(s, 32, axis=1) + np.repeat(m, 32, axis=1)   # exact in fp64
    return w.astype(np.float16).astype(np.float64)


def f16_rows(X):
    """Each row times 2^sh, sh = min(14 - floor(log2 amax), 126), to f16, and 2^-sh."""
    X = np.asarray(X, np.float64)
    out = np.empty_like(X)
    up = np.ones(X.shape[0])
    for r, row in enumerate(X):
        amax = np.abs(row).max()
        sh = 0 if amax == 0 else min(14 - int(np.floor(np.log2(amax))), 126)
        out[r] = (row * 2.0 ** sh).astype(np.float16).astype(np.float64)
        up[r] = 2.0 ** -sh
    return out, up


def emulate(tiles, N, K, X):
    W16 = f16_weights(tiles, N, K)
    X16, up = f16_rows(X)
    return (X16 @ W16.T) * up[:, None]


def bf16_weight_product(tiles, N, K, X):
    return np.asarray(X, np.float64) @ O.bf16_rne(O.q4_decode(tiles, N, K)).T


def two_valued(seed, N, K, lo=1.0, hi=1.0039):
    rng = np.random.default_rng(seed)
    pat = rng.random(K) < 0.5
    pat[0::32], pat[1::32] = False, True
    W = np.where(pat, hi, lo)[None, :] * (2.0 ** rng.integers(-8, 9, N))[:, None]
    return W.astype(np.float32), pat


def bf16_values(a):
    return O.bf16_rne(np.asarray(a, np.float32))


def test_activation_rows_convert_exactly():
    rng = np.random.default_rng(1)
    K = 512
    X = rng.standard_normal((6, K))
    X[0] *= 2.0 ** 100
    X[1] *= 2.0 ** -100
    # magnitudes in [2^-14, 2^15): every element within 2^31 of the row's largest
    X[2] = rng.choice([-1.0, 1.0], K) * rng.uniform(1.0, 2.0, K) * 2.0 ** rng.integers(-14, 15, K)
    X[3, 5] = 3.0e4
    X[4] *= 1.0e-38                           # bf16 subnormals
    X[5] = 0.0
    X = bf16_values(X)
    X16, up = f16_rows(X)
    assert np.array_equal(X16 * up[:, None], X)
    assert np.all(np.abs(X16).max(axis=1)[:5] < 2.0 ** 15)


def test_same_sign_case_defeats_bf16_and_meets_f16_bound():
    N, K, M = 64, 1024, 4
    W, pat = two_valued(2, N, K)
    tiles = O.pack_q4(W)
    X = bf16_values(np.random.default_rng(3).uniform(0.5, 2.0, (M, K)) * pat[None, :])
    y, norm = O.q4_gemm(tiles, N, K, X)
    e_bf16 = O.normalized_error(bf16_weight_product(tiles, N, K, X), y, norm)
    e_f16 = O.normalized_error(emulate(tiles, N, K, X), y, norm)
    assert e_bf16 > 3.8e-3           # one bf16 rounding per weight misses the 2e-3 gate
    assert e_f16 <= 2.0 ** -11       # one f16 rounding stays within its bound


def test_f16_bound_on_random_weights_and_wide_activations():
    rng = np.random.default_rng(4)
    N, K, M = 96, 768, 8
    W = (rng.standard_normal((N, K)) * 0.02 * 2.0 ** rng.integers(-4, 5, (N, 1))).astype(np.float32)
    tiles = O.pack_q4(W)
    X = rng.standard_normal((M, K)) * 2.0 ** rng.integers(-60, 61, (M, 1))
    X = bf16_values(X)
    y, norm = O.q4_gemm(tiles, N, K, X)
    assert O.normalized_error(emulate(tiles, N, K, X), y, norm) <= 2.0 ** -11


def test_planted_coarser_weight_rounding_is_caught():
    # the bound is tight enough to reject a route that rounded to 10 significant bits
    N, K = 32, 512
    W, pat = two_valued(5, N, K, lo=1.0, hi=1.000976)   # code 15 decodes to 1.00097275
    tiles = O.pack_q4(W)
    X = bf16_values(pat[None, :].astype(np.float64))
    y, norm = O.q4_gemm(tiles, N, K, X)
    Wd = O.q4_decode(tiles, N, K)
    mant, e = np.frexp(Wd)
    w10 = np.ldexp(np.round(mant * 2 ** 10) / 2 ** 10, e)   # 10 significant bits
    assert O.normalized_error(X @ w10.T, y, norm) > 2.0 ** -11
    assert O.normalized_error(emulate(tiles, N, K, X), y, norm) <= 2.0 ** -11

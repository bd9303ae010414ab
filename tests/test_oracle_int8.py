"""Pins for the int8 half of the oracle (CPU only).

Each test checks the oracle against something it does not compute itself:
pure-Python brute force, an fp64 BLAS product, numpy's own float32 arithmetic,
or constants printed on the pages.
"""
import itertools

import numpy as np
import pytest

import oracle.qmm_oracle as O


def brute_y(A, zA, B, zB):
    """sum_k (A - zA)(B - zB) with Python ints, the definition on the pages."""
    M, K = len(A), len(A[0])
    N = len(B[0])
    return [[sum((int(A[m][k]) - zA) * (int(B[k][n]) - zB) for k in range(K)) for n in range(N)]
            for m in range(M)]


def brute_s(A, a_type, B, b_type):
    sh = lambda v, t: int(v) - 128 if t == "u8" else int(v)
    M, K, N = len(A), len(A[0]), len(B[0])
    return [[sum(sh(A[m][k], a_type) * sh(B[k][n], b_type) for k in range(K)) for n in range(N)]
            for m in range(M)]


def rand_codes(rng, t, shape):
    return rng.integers(0, 256, shape) if t == "u8" else rng.integers(-128, 128, shape)


@pytest.mark.parametrize("a_type,b_type", list(itertools.product(["u8", "s8"], repeat=2)))
def test_brute_force_tiny(a_type, b_type):
    rng = np.random.default_rng(1)
    lo = {"u8": 0, "s8": -128}
    hi = {"u8": 255, "s8": 127}
    for M, K, N in [(1, 1, 1), (2, 3, 4), (4, 4, 4), (3, 1, 2), (1, 4, 3)]:
        for zA, zB in [(0, 0), (lo[a_type], hi[b_type]), (hi[a_type], lo[b_type]),
                       (int(rng.integers(lo[a_type], hi[a_type] + 1)),
                        int(rng.integers(lo[b_type], hi[b_type] + 1)))]:
            A = rand_codes(rng, a_type, (M, K))
            B = rand_codes(rng, b_type, (K, N))
            r = O.int8_gemm_y(A, a_type, zA, B, b_type, zB)
            assert r["Y"].tolist() == brute_y(A.tolist(), zA, B.tolist(), zB)
            assert r["S"].tolist() == brute_s(A.tolist(), a_type, B.tolist(), b_type)


def test_extreme_codes_brute_force():
    # all -128 * -128 products (the largest magnitude per product) and sign flips
    A = np.full((2, 4), -128)
    B = np.array([[-128, 127], [-128, -128], [-128, 127], [-128, -128]])
    r = O.int8_gemm_y(A, "s8", 0, B, "s8", 0)
    assert r["S"].tolist() == brute_s(A.tolist(), "s8", B.tolist(), "s8")
    assert r["S"][0, 0] == 4 * 16384


def test_s_against_fp64_blas():
    # int8 products summed over K=300 stay far below 2^53: the fp64 BLAS product is exact
    rng = np.random.default_rng(2)
    A = rng.integers(0, 256, (64, 300))
    B = rng.integers(-128, 128, (300, 50))
    r = O.int8_gemm_y(A, "u8", 17, B, "s8", -3)
    S64 = (A - 128).astype(np.float64) @ B.astype(np.float64)
    assert np.array_equal(r["S"], S64.astype(np.int64))
    Yd = (A - 17).astype(np.float64) @ (B + 3).astype(np.float64)
    assert np.array_equal(r["Y"], Yd.astype(np.int64))


def test_planted_shift_error_is_caught(monkeypatch):
    # a plausible mistake (shifting uint8 by 127) must break the brute-force pin
    real = O.shift

    def bad_shift(x, t):
        return real(x, t) + (1 if t == "u8" else 0)

    monkeypatch.setattr(O, "shift", bad_shift)
    rng = np.random.default_rng(3)
    A = rng.integers(0, 256, (2, 3))
    B = rng.integers(-128, 128, (3, 2))
    with pytest.raises(AssertionError):
        # the identity check inside the oracle fires, or the S pin fails
        r = O.int8_gemm_y(A, "u8", 5, B, "s8", 0)
        assert r["S"].tolist() == brute_s(A.tolist(), "u8", B.tolist(), "s8")


def test_planted_sign_error_is_caught():
    # flipping the sign of the zB' term must disagree with the direct definition
    rng = np.random.default_rng(4)
    A = rng.integers(0, 256, (3, 5))
    B = rng.integers(-128, 128, (5, 4))
    r = O.int8_gemm_y(A, "u8", 100, B, "s8", 7)
    K = 5
    bad = r["S"] - r["zAp"] * r["colSum"][None, :] + r["zBp"] * (r["rowSum"][:, None] - K * r["zAp"])
    assert not np.array_equal(bad, np.array(brute_y(A.tolist(), 100, B.tolist(), 7)))


def test_k_bound(golden):
    g = golden("int8_inference_bounds.txt")
    assert g["bound_factor"] == 255 * 128
    kmax = max(k for k in range(60000, 70000) if O.check_k_bound(k))
    assert kmax * g["bound_factor"] < g["bound_limit"] <= (kmax + 1) * g["bound_factor"]
    assert abs(kmax - g["k_about"]) < 1000           # "K up to about 65,000"
    assert O.check_k_bound(g["largest_model_k"])


def test_requant_ties_to_even_and_zp_after_round():
    # Mq = fl(fl(1*0.5)/1) = 0.5 exactly, so odd Yb gives exact .5 ties
    Yb = np.array([[5, -7, 3, -3, 1, -1]])
    q = O.int8_epilogue(Yb, "s8", s_x=1.0, s_w=np.full(6, 0.5), s_y=1.0, zp_y=0)
    assert q.tolist() == [[2, -4, 2, -2, 0, 0]]
    q1 = O.int8_epilogue(Yb, "s8", s_x=1.0, s_w=np.full(6, 0.5), s_y=1.0, zp_y=1)
    # zero point added after rounding: 2.5 -> 2 -> 3 (rounding 3.5 would give 4)
    assert q1.tolist() == [[3, -3, 3, -1, 1, 1]]


def test_rounding_boundary_example(golden):
    g = golden("onnx_pack_rounding_boundary.txt")
    acc = g["accumulator"]
    s_w = np.float32(g["exact_scaled"] / acc)
    r = float(np.float32(np.float32(acc) * s_w))
    assert abs(r - g["exact_scaled"]) < 1e-6
    q = O.int8_epilogue(np.array([[acc]]), "s8", s_x=1.0, s_w=np.array([s_w]), s_y=1.0)
    assert int(q[0, 0]) == g["expected_q"]
    # the float32-accumulation value of the page rounds half to even the other way
    assert int(np.rint(g["float_path_scaled"])) == g["float_path_q"]


def test_clamps():
    Yb = np.array([[2 ** 30, -2 ** 30, 0]])
    assert O.int8_epilogue(Yb, "s8").tolist() == [[127, -128, 0]]
    assert O.int8_epilogue(Yb, "u8").tolist() == [[255, 0, 0]]
    assert O.int8_epilogue(Yb, "u8", zp_y=128).tolist() == [[255, 0, 128]]


def test_f32_and_requant_match_numpy_float32():
    # numpy float32 arithmetic is IEEE single precision; the oracle emulates it in fp64
    rng = np.random.default_rng(5)
    M, N = 8, 6
    Y = rng.integers(-2 ** 24, 2 ** 24, (M, N))
    sx = rng.uniform(1e-3, 1e-1, M).astype(np.float32)
    sw = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    sy = np.float32(0.37)
    f = O.int8_epilogue(Y, "f32", s_x=sx, s_w=sw)
    ref = (Y.astype(np.float32) * sx[:, None]) * sw[None, :]
    assert np.array_equal(f.astype(np.float32), ref)
    q = O.int8_epilogue(Y // 2 ** 12, "s8", s_x=sx, s_w=sw, s_y=float(sy), zp_y=-7)
    mq = (sx[:, None] * sw[None, :]) / sy
    refq = np.clip(np.rint((Y // 2 ** 12).astype(np.float32) * mq).astype(np.int64) - 7, -128, 127)
    assert np.array_equal(q, refq)


def test_page_zero_points_proof_shapes(golden):
    g = golden("onnx_pack_qdq_constants.txt")
    rng = np.random.default_rng(6)
    for (M, K, N) in (g["proof_shape"], g["large_shape"]):
        A = rng.integers(-128, 128, (M, K))
        B = rng.integers(-128, 128, (K, N))
        r = O.int8_gemm_y(A, "s8", g["zp_x"], B, "s8", g["zp_w"])
        direct = (A - g["zp_x"]).astype(np.float64) @ (B - g["zp_w"]).astype(np.float64)
        assert np.array_equal(r["Y"], direct.astype(np.int64))
        if M * N <= 100:
            assert r["Y"].tolist() == brute_y(A.tolist(), g["zp_x"], B.tolist(), g["zp_w"])
        sx = np.float32(0.02)
        sw = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
        sy = np.float32(float(np.abs(r["Y"]).mean()) * 0.02 * 5e-3 / 40)
        q = O.int8_epilogue(r["Y"], "s8", s_x=float(sx), s_w=sw, s_y=float(sy), zp_y=g["zp_y"])
        mq = (sx * sw) / sy
        ref = np.clip(np.rint(r["Y"].astype(np.float32) * mq[None, :]).astype(np.int64) + g["zp_y"],
                      -128, 127)
        assert np.array_equal(q, ref)


def test_per_axis_scales(golden):
    g = golden("onnx_pack_qdq_constants.txt")
    M, N = g["per_axis_rows"], g["per_axis_cols"]
    rng = np.random.default_rng(7)
    A = rng.integers(0, 256, (M, 40))
    B = rng.integers(-127, 128, (40, N))
    r = O.int8_gemm_y(A, "u8", 131, B, "s8", 0)
    sx = rng.uniform(0.01, 0.03, M).astype(np.float32)
    sw = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    q = O.int8_epilogue(r["Y"], "u8", s_x=sx, s_w=sw, s_y=0.5, zp_y=128)
    mq = (sx[:, None] * sw[None, :]) / np.float32(0.5)
    ref = np.clip(np.rint(r["Y"].astype(np.float32) * mq).astype(np.int64) + 128, 0, 255)
    assert np.array_equal(q, ref)


def test_packb_from_f32():
    rng = np.random.default_rng(8)
    K, N = 100, 7
    W = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    W[:, 3] = 0.0                                   # amax == 0 column
    p = O.pack_b_int8(W, "f32")
    q, s = p["codes"], p["col_scale"]
    assert p["packed"].shape == (N, O.padded_k(K)) and O.padded_k(K) == 128
    assert np.all(p["packed"][:, K:] == 0)
    assert np.array_equal(p["packed"][:, :K].T.astype(np.int64), q)
    assert s[3] == 0 and np.all(q[:, 3] == 0)
    for n in range(N):
        if n == 3:
            continue
        amax = np.abs(W[:, n]).max()
        assert s[n] == np.float32(amax / np.float32(127))
        kk = int(np.abs(W[:, n]).argmax())
        assert abs(q[kk, n]) == 127
        err = np.abs(W[:, n].astype(np.float64) - q[:, n] * s[n])
        assert err.max() <= s[n] / 2 * (1 + 2 ** -20)
    # independent route: numpy float32 division then half-even rounding
    ref = np.clip(np.rint(W / np.where(s > 0, s, 1).astype(np.float32)), -127, 127)
    ref[:, 3] = 0
    assert np.array_equal(q, ref.astype(np.int64))
    assert np.array_equal(p["col_sum"], q.sum(axis=0))


def test_packb_from_u8_shifts():
    rng = np.random.default_rng(9)
    B = rng.integers(0, 256, (33, 5))
    p = O.pack_b_int8(B, "u8")
    assert np.array_equal(p["packed"][:, :33].T.astype(np.int64), B - 128)
    assert p["col_sum"].tolist() == [sum(int(B[k, n]) - 128 for k in range(33)) for n in range(5)]


# ---------------------------------------------------------------------------
# activation quantisation (s = amax/127 per row or per tensor, packB rounding)
# ---------------------------------------------------------------------------

def test_activation_quant_amax_maps_to_127_and_ties_to_even():
    # amax = 127 gives s = 1 exactly, so the codes are the rounded values
    X = np.array([[127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -126.4, -0.49],
                  [-127.0, 0.0, 63.5, -63.5, 64.5, 1e-8, 5.5, -5.5]], dtype=np.float32)
    q, s = O.quantize_activations_f32(X, per_row=True)
    assert list(s) == [1.0, 1.0]
    assert q[0].tolist() == [127, 2, 4, -2, 0, 2, -126, 0]
    assert q[1].tolist() == [-127, 0, 64, -64, 64, 0, 6, -6]


def test_activation_quant_zero_row_and_bound():
    g = np.random.default_rng(3)
    X = (g.standard_normal((6, 257)) * np.array([[1e-3], [0.0], [1.0], [40.0], [1e4], [0.02]])).astype(np.float32)
    q, s = O.quantize_activations_f32(X, per_row=True)
    assert s[1] == 0.0 and not q[1].any()
    for m in range(6):
        assert np.abs(q[m]).max() <= 127
        if s[m] > 0:
            i = np.argmax(np.abs(X[m]))
            assert abs(q[m, i]) == 127 and np.sign(q[m, i]) == np.sign(X[m, i])
            # packB's rounding bound: |x - q s| <= s/2 (one fp32 rounding of x/s on top)
            assert np.all(np.abs(X[m].astype(np.float64) - q[m] * s[m]) <= s[m] * 0.5 * (1 + 2.0 ** -22))


def test_activation_quant_rows_are_packb_columns():
    # the row rule is packB's column rule on the transpose (checked separately above)
    g = np.random.default_rng(4)
    X = (g.standard_normal((9, 130)) * 3).astype(np.float32)
    q, s = O.quantize_activations_f32(X, per_row=True)
    qc, sc = O.quantize_columns_f32(X.T)
    assert np.array_equal(q, qc.T) and np.array_equal(s, sc)


def test_activation_quant_per_tensor():
    g = np.random.default_rng(5)
    X = (g.standard_normal((7, 100)) * np.arange(1, 8)[:, None]).astype(np.float32)
    q, s = O.quantize_activations_f32(X, per_row=False)
    qr, sr = O.quantize_activations_f32(X, per_row=True)
    assert s.shape == (1,) and s[0] == sr.max()                # one scale: the largest row's
    assert np.array_equal(q[np.argmax(sr)], qr[np.argmax(sr)])  # that row is coded as per row
    q1, s1 = O.quantize_activations_f32(X[2:3], per_row=False)
    assert np.array_equal(q1, qr[2:3]) and s1[0] == sr[2]       # one row: the two modes agree


# --------------------------------------------------------------------------
# per-axis zero points (ONNX pack page, "What works today": per-axis along the
# same axes as the scales; the fully per-axis proof uses 8 row scales and zero
# points and 6 column scales and zero points)
# --------------------------------------------------------------------------

def brute_y_axis(A, zA, B, zB):
    M, K, N = len(A), len(A[0]), len(B[0])
    return [[sum((int(A[m][k]) - int(zA[m])) * (int(B[k][n]) - int(zB[n])) for k in range(K)) for n in range(N)]
            for m in range(M)]


@pytest.mark.parametrize("a_type,b_type", list(itertools.product(["u8", "s8"], repeat=2)))
def test_axis_zp_brute_force_tiny(a_type, b_type):
    rng = np.random.default_rng(21)
    for M, K, N in [(1, 1, 1), (2, 3, 4), (4, 4, 4), (3, 1, 2), (1, 5, 3)]:
        A = rand_codes(rng, a_type, (M, K))
        B = rand_codes(rng, b_type, (K, N))
        zA = rand_codes(rng, a_type, (M,))
        zB = rand_codes(rng, b_type, (N,))
        r = O.int8_gemm_y_axis(A, a_type, zA, B, b_type, zB)
        assert r["Y"].tolist() == brute_y_axis(A.tolist(), zA.tolist(), B.tolist(), zB.tolist())


def test_axis_zp_equal_entries_reduce_to_per_tensor():
    rng = np.random.default_rng(22)
    for a_type, b_type in itertools.product(["u8", "s8"], repeat=2):
        A = rand_codes(rng, a_type, (7, 33))
        B = rand_codes(rng, b_type, (33, 5))
        zA = int(rand_codes(rng, a_type, ()))
        zB = int(rand_codes(rng, b_type, ()))
        axis = O.int8_gemm_y_axis(A, a_type, np.full(7, zA), B, b_type, np.full(5, zB))
        tensor = O.int8_gemm_y(A, a_type, zA, B, b_type, zB)
        assert np.array_equal(axis["Y"], tensor["Y"])


def test_axis_zp_page_proof_shape(golden):
    """8 row zero points and 6 column zero points (the fully per-axis proof),
    on the 8 x 16 x 6 proof shape; checked against an fp64 BLAS product of the
    shifted operands and against brute force."""
    g = golden("onnx_pack_qdq_constants.txt")
    M, K, N = g["proof_shape"]
    assert (M, N) == (g["per_axis_rows"], g["per_axis_cols"])
    rng = np.random.default_rng(23)
    A = rng.integers(-128, 128, (M, K))
    B = rng.integers(-128, 128, (K, N))
    zA = g["zp_x"] + rng.integers(-3, 4, M)
    zB = g["zp_w"] + rng.integers(-3, 4, N)
    r = O.int8_gemm_y_axis(A, "s8", zA, B, "s8", zB)
    direct = (A - zA[:, None]).astype(np.float64) @ (B - zB[None, :]).astype(np.float64)
    assert np.array_equal(r["Y"], direct.astype(np.int64))
    assert r["Y"].tolist() == brute_y_axis(A.tolist(), zA.tolist(), B.tolist(), zB.tolist())


def test_axis_zp_transposed_zero_points_are_caught():
    """A plausible mistake, the row zero points applied along columns and the
    column ones along rows, gives a different Y; the brute-force pin tells
    the two apart (square shape, so both versions are well formed)."""
    rng = np.random.default_rng(24)
    A = rng.integers(-128, 128, (6, 9))
    B = rng.integers(-128, 128, (9, 6))
    zA = rng.integers(-128, 128, 6)
    zB = rng.integers(-128, 128, 6)
    good = O.int8_gemm_y_axis(A, "s8", zA, B, "s8", zB)["Y"].tolist()
    assert good == brute_y_axis(A.tolist(), zA.tolist(), B.tolist(), zB.tolist())
    assert good != brute_y_axis(A.tolist(), zB.tolist(), B.tolist(), zA.tolist())

"""Pins for the 4-bit half of the oracle (CPU only)."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 10.0 ** rng.integers(-8, 8, 10000),
                        np.array([1.00390625, 1.01171875, -1.00390625, 3.0e38, 0.0, -0.0],
                                 dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_rne(x), ref)


def test_tile_geometry(golden):
    g = golden("q4nx_tile_geometry.txt")
    assert (O.TILE_ROWS, O.TILE_COLS, O.TILE_BYTES, O.BLOCK) == (
        g["tile_rows"], g["tile_cols"], g["tile_bytes"], g["block"])
    # codes take half a byte each, plus one bf16 scale and one bf16 min per block
    assert g["tile_rows"] * g["tile_cols"] // 2 + g["tile_rows"] * g["tile_cols"] // g["block"] * 4 \
        == g["tile_bytes"]


def scalar_tile_writer(q, s, m):
    """Independent, element-by-element writer of the documented tile format."""
    N, K = q.shape
    TR, TC = N // 32, K // 256
    buf = bytearray(TR * TC * 5120)
    sb = O.bf16_bits(s)
    mb = O.bf16_bits(m)
    for n in range(N):
        tr, r = divmod(n, 32)
        for k in range(K):
            tc, kk = divmod(k, 256)
            b, rest = divmod(kk, 32)
            t, j = divmod(rest, 8)
            i, hi = divmod(j, 2)
            bit = 4 * i + 16 * hi
            base = (tr * TC + tc) * 5120
            word_off = base + r * 128 + 16 * b + 4 * t
            byte = word_off + bit // 8
            buf[byte] |= int(q[n, k]) << (bit % 8)
        for blk in range(K // 32):
            tc, b = divmod(blk, 8)
            base = (tr * TC + tc) * 5120 + 4096 + 4 * (8 * r + b)
            buf[base:base + 2] = int(sb[n, blk]).to_bytes(2, "little")
            buf[base + 2:base + 4] = int(mb[n, blk]).to_bytes(2, "little")
    return np.frombuffer(bytes(buf), dtype=np.uint8)


def random_blocks(rng, N, K):
    q = rng.integers(0, 16, (N, K))
    s = O.bf16_rne(rng.uniform(1e-4, 1e-2, (N, K // 32)))
    m = O.bf16_rne(rng.uniform(-0.1, 0.0, (N, K // 32)))
    return q, s, m


def test_tile_format_against_scalar_writer():
    rng = np.random.default_rng(1)
    q, s, m = random_blocks(rng, 64, 512)
    t = O.q4_tiles_from_blocks(q, s, m)
    assert np.array_equal(t, scalar_tile_writer(q, s, m))
    q2, s2, m2 = O.q4_blocks_from_tiles(t, 64, 512)
    assert np.array_equal(q2, q) and np.array_equal(s2, s) and np.array_equal(m2, m)


def test_pack_decode_round_trip_bound():
    rng = np.random.default_rng(2)
    N, K = 64, 512
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    W[3, :32] = 0.25                              # a constant block: scale 0
    tiles = O.pack_q4(W)
    assert tiles.size == (N // 32) * (K // 256) * 5120
    dec = O.q4_decode(tiles, N, K)
    Wb = W.astype(np.float64).reshape(N, K // 32, 32)
    mx, mn = Wb.max(axis=2), Wb.min(axis=2)
    q, s, m = O.q4_blocks_from_tiles(tiles, N, K)
    bound = 0.5 * s + 2.0 ** -8 * (np.abs(mn) + (mx - mn)) + 1e-7 * np.abs(Wb).max(axis=2)
    err = np.abs(dec.reshape(N, K // 32, 32) - Wb).max(axis=2)
    assert np.all(err <= bound)
    assert s[3, 0] == 0 and np.all(q[3, :32] == 0) and dec[3, 0] == O.bf16_rne(0.25)
    # quantiser pinned against torch's own bf16 rounding and float32 division
    Wt = torch.from_numpy(W).reshape(N, K // 32, 32)
    st = ((Wt.amax(2) - Wt.amin(2)) / 15).to(torch.bfloat16).double().numpy()
    mt = Wt.amin(2).to(torch.bfloat16)
    qt = torch.clamp(torch.round((Wt - mt.float()[:, :, None]) / torch.from_numpy(st).float().clamp_min(1e-30)[:, :, None]), 0, 15)
    qt[torch.from_numpy(st) == 0] = 0
    assert np.array_equal(s, st) and np.array_equal(m, mt.double().numpy())
    assert np.array_equal(q.reshape(N, K // 32, 32), qt.numpy().astype(np.int64))


def test_integer_special_case_exact():
    # scale 1, min 0: the product is an integer GEMM and must equal the int64 dot
    rng = np.random.default_rng(3)
    N, K, M = 32, 512, 3
    q = rng.integers(0, 16, (N, K))
    tiles = O.q4_tiles_from_blocks(q, np.ones((N, K // 32)), np.zeros((N, K // 32)))
    X = rng.integers(-8, 9, (M, K))
    y, _ = O.q4_gemm(tiles, N, K, X.astype(np.float64))
    assert np.array_equal(y, (X @ q.T).astype(np.float64))


def test_constant_codes_closed_form():
    rng = np.random.default_rng(4)
    N, K = 32, 256
    qb = rng.integers(0, 16, (N, K // 32))
    q = np.repeat(qb, 32, axis=1)
    s = O.bf16_rne(rng.uniform(1e-3, 1e-2, (N, K // 32)))
    m = O.bf16_rne(rng.uniform(-0.05, 0.05, (N, K // 32)))
    tiles = O.q4_tiles_from_blocks(q, s, m)
    x = O.bf16_rne(rng.standard_normal(K))
    y, _ = O.q4_gemm(tiles, N, K, x[None, :])
    xs = x.reshape(K // 32, 32).sum(axis=1)
    closed = ((qb * s + m) * xs[None, :]).sum(axis=1)
    assert np.allclose(y[0], closed, rtol=1e-12, atol=1e-15)


def test_one_hot_selects_weight():
    rng = np.random.default_rng(5)
    N, K = 64, 512
    q, s, m = random_blocks(rng, N, K)
    tiles = O.q4_tiles_from_blocks(q, s, m)
    for k in (0, 1, 7, 8, 31, 32, 255, 256, 300, 511):
        x = np.zeros((1, K))
        x[0, k] = 1.0
        y, _ = O.q4_gemm(tiles, N, K, x)
        for n in (0, 5, 31, 32, 63):
            assert y[0, n] == q[n, k] * s[n, k // 32] + m[n, k // 32]


@pytest.mark.parametrize("M", [1, 2, 3])
def test_brute_force_tiny(M):
    rng = np.random.default_rng(6 + M)
    N, K = 32, 256
    q, s, m = random_blocks(rng, N, K)
    tiles = O.q4_tiles_from_blocks(q, s, m)
    X = O.bf16_rne(rng.standard_normal((M, K)))
    y, norm = O.q4_gemm(tiles, N, K, X)
    for mm in range(M):
        for n in range(N):
            acc = 0.0
            nrm = 0.0
            for k in range(K):
                w = float(q[n, k]) * float(s[n, k // 32]) + float(m[n, k // 32])
                acc += float(X[mm, k]) * w
                nrm += abs(float(X[mm, k])) * abs(w)
            assert abs(acc - y[mm, n]) <= 1e-12 * max(1.0, nrm)
            assert abs(nrm - norm[mm, n]) <= 1e-12 * max(1.0, nrm)


def test_decode_rows_matches_full():
    rng = np.random.default_rng(9)
    N, K = 96, 512
    q, s, m = random_blocks(rng, N, K)
    tiles = O.q4_tiles_from_blocks(q, s, m)
    full = O.q4_decode(tiles, N, K)
    rows = [0, 33, 95, 64]
    assert np.array_equal(O.q4_decode_rows(tiles, N, K, rows), full[rows])


def test_moe_strided_ids_and_per_slot(golden):
    g = golden("zaya_strided_ids.txt")
    ld = g["ids_per_token"]
    assert ld * 4 == g["row_stride_bytes"]
    rng = np.random.default_rng(10)
    E, N, K, T, n_used = 6, 32, 256, 5, 3
    W = (rng.standard_normal((E, N, K)) * 0.02).astype(np.float32)
    tiles = np.concatenate([O.pack_q4(W[e]) for e in range(E)])
    ids_buf = np.stack([rng.permutation(E).tolist() + [0] * (ld - E) for _ in range(T)]).astype(np.int32)
    Xs = O.bf16_rne(rng.standard_normal((T, K)))
    Y, _ = O.q4_gemm_id(tiles, E, N, K, Xs, True, ids_buf, ld, n_used, T)
    for t in range(T):
        for i in range(n_used):
            e = int(ids_buf[t, i])
            dense = O.q4_decode(O.pack_q4(W[e]), N, K)
            assert np.allclose(Y[t, i], dense @ Xs[t], rtol=0, atol=1e-12)
    # reading the ids contiguously picks other experts (the bug on the page)
    wrong = ids_buf.reshape(-1)[:T * n_used].reshape(T, n_used)
    assert not np.array_equal(wrong, O.moe_ids_view(ids_buf, ld, n_used, T))
    # per-slot src1: slot i of token t reads its own activation row
    Xp = O.bf16_rne(rng.standard_normal((T, n_used, K)))
    Yp, _ = O.q4_gemm_id(tiles, E, N, K, Xp, False, ids_buf, ld, n_used, T)
    t, i = 2, 1
    dense = O.q4_decode(O.pack_q4(W[int(ids_buf[t, i])]), N, K)
    assert np.allclose(Yp[t, i], dense @ Xp[t, i], atol=1e-12)
    assert not np.allclose(Yp[t, i], dense @ Xp[t, 0], atol=1e-6)


def test_moe_rejects_bad_ids():
    tiles = O.pack_q4(np.zeros((32, 256), np.float32))
    ids = np.array([[0, 1]], dtype=np.int32)
    with pytest.raises(AssertionError):
        O.q4_gemm_id(tiles, 1, 32, 256, np.zeros((1, 256)), True, ids, 2, 2, 1)


def test_normalized_error():
    assert O.normalized_error([1.0, 0.0], [1.0, 0.0], [2.0, 0.0]) == 0.0
    assert O.normalized_error([1.1, 0.0], [1.0, 0.0], [2.0, 0.0]) == pytest.approx(0.05)
    assert O.normalized_error([1.0, 1e-9], [1.0, 0.0], [2.0, 0.0]) == float("inf")


# ---------------------------------------------------------------------------
# W8A16 (int8 weights, a scale for every 1,024 weights of a row)
# ---------------------------------------------------------------------------

def test_w8_blocks_are_packb_columns():
    # each (row, 1024-block) follows packB's column rule: compare block by block
    g = np.random.default_rng(11)
    W = (g.standard_normal((5, 2500)) * np.array([[0.02], [1.0], [0.0], [3e-4], [50.0]])).astype(np.float32)
    q, s = O.pack_w8(W)
    assert s.shape == (5, 3)
    for b in range(3):
        blk = W[:, b * 1024:(b + 1) * 1024]
        qc, sc = O.quantize_columns_f32(blk.T)
        assert np.array_equal(q[:, b * 1024:(b + 1) * 1024], qc.T) and np.array_equal(s[:, b], sc)
    assert not q[2].any() and not s[2].any()            # zero row: scale 0, codes 0
    assert np.abs(q).max() == 127


def test_w8_gemm_brute_force_and_block_scales():
    g = np.random.default_rng(12)
    N, K, M = 3, 2100, 2
    q = g.integers(-127, 128, (N, K))
    s = g.uniform(1e-3, 1e-1, (N, 3))
    X = g.standard_normal((M, K))
    Y, norm = O.w8_gemm(q, s, X)
    for m in range(M):
        for n in range(N):
            want = sum(s[n, k // 1024] * q[n, k] * X[m, k] for k in range(K))
            assert abs(Y[m, n] - want) <= 1e-9 * norm[m, n]
            assert abs(norm[m, n] - sum(abs(s[n, k // 1024] * q[n, k] * X[m, k]) for k in range(K))) <= 1e-9 * norm[m, n]
    # a block's scale multiplies only that block's partial sum
    s2 = s.copy()
    s2[1, 2] *= 2
    Y2, _ = O.w8_gemm(q, s2, X)
    part = X[:, 2048:] @ q[1, 2048:].astype(np.float64)
    assert np.allclose(Y2[:, 1] - Y[:, 1], part * s[1, 2])
    assert np.array_equal(Y2[:, [0, 2]], Y[:, [0, 2]])


def test_w8_decode_bound():
    g = np.random.default_rng(13)
    W = (g.standard_normal((4, 3000)) * 0.05).astype(np.float32)
    q, s = O.pack_w8(W)
    dec = q * np.repeat(s, 1024, axis=1)[:, :3000]
    lim = np.repeat(s, 1024, axis=1)[:, :3000] * 0.5 * (1 + 2.0 ** -22)
    assert np.all(np.abs(W.astype(np.float64) - dec) <= lim)

"""CPU oracle for the quantized projection matmul: plain, slow and meant to be checked by eye.

TEST INFRASTRUCTURE ONLY.  Nothing on the library's product path imports this
module.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA library: the two
meet only through the seeded inputs from ``quantized_matmul_qmm_gb300.inputs``.

Arithmetic
----------
* Integer work runs in int64 (numpy).
* Float work runs in fp64.  Where the method fixes fp32 (the int8 epilogue and
  the packers), each fp32 operation is one exact or correctly rounded fp64
  operation followed by rounding to fp32 (``_f32``).  fp64 has 53 >= 2*24+2
  significand bits, so that double rounding gives the correctly rounded fp32
  result of +, -, *, / (Figueroa's theorem).
* bf16 values are made by round-to-nearest-even from fp32 (``bf16_rne``).

Sources (page title, section)
-----------------------------
* int8 inference -- "Product kernel (Int8Gemm)": the zero-point algebra,
  the uint8 shift by 128, the K*255*128 < 2^31 bound and the epilogue order
  (zero-point correction, optional bias, requantisation or float output).
* The ONNX pack: weights to Q4NX, matmuls to our kernels, no VitisAI --
  "The three layers of the pack": packB quantises each weight column with
  scale = amax/127 and keeps the column scales.  Float dequant is
  C = Cm * ascale[row] * wscale[col].
* same page, "Why it folds without a new kernel" and "What works today":
  y_q = clamp(round(C_s32 * s_x * s_w / s_y)) with round-half-to-even, the
  output zero point added after rounding, and the column sums computed once
  per weight.
* NPU engine: full ELFs, no xclbin -- "Q4NX chunks": 32-row x 256-column
  tiles of 5120 bytes, row-major over the tile grid; q4_1 blocks.
* Zaya 8B Q4NX on the AMD NPU -- round 26 ("the twin"): W = q4*scale + zp
  with per-(row, 32-column) bf16 scale and zero.  The dense "twin" decodes
  every tile to full precision and runs a plain matmul.  "The bugs that were
  the work": the ids of MUL_MAT_ID are a strided view, and down-projection
  experts read a per-slot src1 column i + t*n_expert_used.
* NPU engine: full ELFs, no xclbin -- "Q4NX chunks": Q4_K weights are
  converted to q4_1, losing only the bf16 rounding of the two per-sub-block
  products (super-block scale times scale code, and the same for the min);
  Q8 tiles store code (r, k) at byte k*32 + r or at
  (r/16)*4096 + (k/32)*512 + (k%32)*16 + r%16.

Readings where the pages are silent
-----------------------------------
These are the repository's own choices, and the design notes list them.
* packB rounds R(W/s) half-to-even and clamps to [-127, 127].  A column with
  amax == 0 gets scale 0 and codes 0.
* F32 output is R(R(R(Y)*s_x[m])*s_w[n]).  The int8/uint8 output uses
  Mq = R(R(s_x[m]*s_w[n])/s_y), then q = clamp(rint_even(R(R(Y)*Mq)) + zp_y).
* q4 quantiser, per block of 32 along K:
  s = bf16(R(R(max-min)/15)), m = bf16(min),
  q = clamp(rint_even(R(R(x-m)/s)), 0, 15), and q = 0 when s == 0.
* The intra-tile byte map is defined below in ``Q4 TILE FORMAT``.  The pages
  do not print the byte layout of a tile.
* Q4_K bytes follow GGML's published super-block layout (the pages name the
  type only).  Q8 tiles add one bf16 scale per (row, 32 columns) after the
  8192 code bytes, and quantise with s = bf16(amax/127) and packB's rounding.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# small exact helpers
# ----------------------------------------------------------------------------

U8, S8 = "u8", "s8"
K_BOUND = 2 ** 31  # int8 inference, "Product kernel": sums are safe while K*255*128 < 2^31


def _f32(x):
    """Round fp64 value(s) to the nearest fp32 (ties to even), returned as fp64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16_rne(x):
    """Round fp32-representable value(s) to bf16, ties to even; returns fp64.

    bf16 keeps the top 16 bits of the fp32 encoding.  Rounding adds 0x7FFF
    plus the lowest kept bit, then truncates.  NaN never occurs in these inputs.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    r = ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16_bits(x):
    """uint16 encoding of bf16 value(s) (x must already be bf16-representable)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value is not bf16-representable"
    return (bits >> 16).astype(np.uint16)


def bf16_from_bits(b):
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def check_k_bound(K: int) -> bool:
    """True when K*255*128 < 2^31 (int8 inference, "Product kernel")."""
    return K * 255 * 128 < K_BOUND


# ----------------------------------------------------------------------------
# int8 half: shifted domain, sums, zero-point algebra
# ----------------------------------------------------------------------------

def shift(x, dtype: str):
    """A' = A - 128 for uint8, A for int8 (int8 inference, "Product kernel")."""
    x = np.asarray(x, dtype=np.int64)
    if dtype == U8:
        assert x.min(initial=0) >= 0 and x.max(initial=0) <= 255
        return x - 128
    assert dtype == S8
    assert x.min(initial=0) >= -128 and x.max(initial=0) <= 127
    return x


def shift_zp(z: int, dtype: str) -> int:
    """zA' = zA - 128 for uint8 operands, zA for int8."""
    return int(z) - 128 if dtype == U8 else int(z)


def int8_gemm_y(A, a_type, zA, B, b_type, zB):
    """Exact zero-point-corrected product, int8 inference "Product kernel".

    A: [M][K] codes, B: [K][N] codes (both int arrays in their own domain).
    Returns dict with S, rowSum, colSum and Y, all int64.

        S[m,n]  = sum_k A'[m,k] B'[k,n]
        Y[m,n]  = S - zA' colSum[n] - zB' (rowSum[m] - K zA')

    and asserts Y equals the direct definition sum_k (A-zA)(B-zB).
    """
    Ap = shift(A, a_type)
    Bp = shift(B, b_type)
    M, K = Ap.shape
    K2, N = Bp.shape
    assert K == K2
    zAp = shift_zp(zA, a_type)
    zBp = shift_zp(zB, b_type)
    S = Ap @ Bp                                   # int64 matmul (library primitive)
    rowSum = Ap.sum(axis=1)                       # [M]
    colSum = Bp.sum(axis=0)                       # [N]
    Y = S - zAp * colSum[None, :] - zBp * (rowSum[:, None] - K * zAp)
    # the zero-point identity, written on the raw integers
    Ydirect = (np.asarray(A, np.int64) - int(zA)) @ (np.asarray(B, np.int64) - int(zB))
    assert np.array_equal(Y, Ydirect), "zero-point identity violated"
    return {"S": S, "rowSum": rowSum, "colSum": colSum, "Y": Y, "zAp": zAp, "zBp": zBp}


def int8_gemm_y_axis(A, a_type, zA_rows, B, b_type, zB_cols):
    """Per-axis zero points: one per activation row (zA_rows [M]) and one per
    weight column (zB_cols [N]), each in its operand's own domain.

    "The ONNX pack: weights to Q4NX, matmuls to our kernels, no VitisAI",
    "What works today": the asymmetric corrections come per tensor or per
    axis, laid out like the scales (row zero points beside row scales,
    column zero points beside column scales), exact in integers:

        Y[m,n] = S - zA'[m] colSum[n] - zB'[n] (rowSum[m] - K zA'[m])

    with the shifted zero points zA'[m] = zA[m] - 128 for uint8 A (B alike).
    Asserts Y equals the direct definition sum_k (A[m,k] - zA[m])(B[k,n] - zB[n]).
    """
    Ap = shift(A, a_type)
    Bp = shift(B, b_type)
    M, K = Ap.shape
    K2, N = Bp.shape
    assert K == K2
    zA = np.asarray(zA_rows, dtype=np.int64).reshape(M)
    zB = np.asarray(zB_cols, dtype=np.int64).reshape(N)
    lo_a, hi_a = (0, 255) if a_type == U8 else (-128, 127)
    lo_b, hi_b = (0, 255) if b_type == U8 else (-128, 127)
    assert zA.min(initial=lo_a) >= lo_a and zA.max(initial=hi_a) <= hi_a
    assert zB.min(initial=lo_b) >= lo_b and zB.max(initial=hi_b) <= hi_b
    zAp = zA - (128 if a_type == U8 else 0)
    zBp = zB - (128 if b_type == U8 else 0)
    S = Ap @ Bp
    rowSum = Ap.sum(axis=1)
    colSum = Bp.sum(axis=0)
    Y = S - zAp[:, None] * colSum[None, :] - zBp[None, :] * (rowSum[:, None] - K * zAp[:, None])
    Ydirect = (np.asarray(A, np.int64) - zA[:, None]) @ (np.asarray(B, np.int64) - zB[None, :])
    assert np.array_equal(Y, Ydirect), "zero-point identity violated"
    return {"S": S, "rowSum": rowSum, "colSum": colSum, "Y": Y, "zAp": zAp, "zBp": zBp}


def int8_epilogue(Y, out_type: str, bias=None, s_x=None, s_w=None, s_y=1.0, zp_y=0):
    """Epilogue after the zero-point correction (int8 inference "Product kernel"
    and the ONNX pack page's fused QuantizeLinear).

    Y: int64 [M][N].  bias: int [N] or None.  s_x: None (=1), a scalar, or [M].
    s_w: None (=1) or [N].  out_type: "s32" | "f32" | "s8" | "u8".
    """
    Y = np.asarray(Y, dtype=np.int64)
    M, N = Y.shape
    Yb = Y + (np.asarray(bias, np.int64)[None, :] if bias is not None else 0)
    for name, v in (("Y", Y), ("Yb", Yb)):
        assert np.abs(v).max(initial=0) < 2 ** 31, f"{name} leaves int32"
    if out_type == "s32":
        return Yb.astype(np.int64)
    sx = np.ones(M) if s_x is None else np.broadcast_to(_f32(s_x), (M,)).astype(np.float64)
    sw = np.ones(N) if s_w is None else _f32(np.asarray(s_w, np.float64))
    sx = _f32(sx)[:, None]
    sw = _f32(sw)[None, :]
    yf = _f32(Yb.astype(np.float64))              # int32 -> fp32 (RNE)
    if out_type == "f32":
        return _f32(_f32(yf * sx) * sw)            # C = Cm * ascale[row] * wscale[col]
    assert out_type in ("s8", "u8")
    mq = _f32(_f32(sx * sw) / _f32(s_y))          # one multiplier per element
    r = _f32(yf * mq)
    q = np.rint(r).astype(np.int64) + int(zp_y)    # round half to even, then zp
    lo, hi = (-128, 127) if out_type == "s8" else (0, 255)
    return np.clip(q, lo, hi)


def int8_gemm(A, a_type, zA, B, b_type, zB, out_type="s32", bias=None, s_x=None,
              s_w=None, s_y=1.0, zp_y=0):
    """Full int8 path: zero-point algebra then the epilogue."""
    r = int8_gemm_y(A, a_type, zA, B, b_type, zB)
    return int8_epilogue(r["Y"], out_type, bias, s_x, s_w, s_y, zp_y)


# ----------------------------------------------------------------------------
# packB (int8 weights)
# ----------------------------------------------------------------------------

def padded_k(K: int) -> int:
    """Packed int8 rows hold K rounded up to 64 bytes (zeros past K)."""
    return (K + 63) // 64 * 64


def quantize_columns_f32(W):
    """Per-column symmetric int8 quantisation, scale = amax/127.

    W: fp32 [K][N].  Returns (codes int64 [K][N], scale fp64 [N] (fp32 values)).
    (ONNX pack page, "The three layers of the pack".)
    """
    W = _f32(np.asarray(W, np.float64))
    amax = np.abs(W).max(axis=0)
    scale = _f32(amax / 127.0)
    q = np.zeros(W.shape, dtype=np.int64)
    nz = scale > 0
    if np.any(nz):
        r = _f32(W[:, nz] / scale[None, nz])
        q[:, nz] = np.clip(np.rint(r), -127, 127).astype(np.int64)
    return q, scale


def quantize_activations_f32(X, per_row: bool):
    """Symmetric int8 activations: scale = amax/127 over each row (per_row) or
    over the whole tensor, then packB's rounding, q = clamp(rint_even(R(x/s)),
    -127, 127), and q = 0 where s == 0.

    (int8 inference, "Product kernel (Int8Gemm)": per-tensor symmetric
    activations with scale amax/127; ONNX pack page, "What works today": the
    per-row activation scale s_x[m] of the float epilogue.)
    X: fp32 values [M][K].  Returns (codes int64 [M][K], scales fp64 holding
    fp32 values: [M] per row, [1] per tensor).
    """
    X = _f32(np.asarray(X, np.float64))
    M = X.shape[0]
    amax = np.abs(X).max(axis=1) if per_row else np.array([np.abs(X).max()])
    scale = _f32(amax / 127.0)
    q = np.zeros(X.shape, dtype=np.int64)
    for m in range(M):
        s = scale[m] if per_row else scale[0]
        if s > 0:
            q[m] = np.clip(np.rint(_f32(X[m] / s)), -127, 127).astype(np.int64)
    return q, scale


def pack_b_int8(B, b_type: str):
    """Packed weights for the int8 GEMM.

    B: [K][N], either fp32 ("f32": quantised per column) or integer codes
    ("s8"/"u8": shifted to int8 by the "Product kernel" rule).
    Returns dict: packed int8 [N][Kp] (K-major, zero padding), col_scale fp32 [N]
    (ones for integer inputs, the library leaves it untouched there),
    col_sum int64 [N] = sum_k B'[k,n] and the int8 codes B' [K][N].
    """
    B = np.asarray(B)
    K, N = B.shape
    if b_type == "f32":
        Bp, scale = quantize_columns_f32(B)
    else:
        Bp = shift(B, b_type)
        scale = None
    Kp = padded_k(K)
    packed = np.zeros((N, Kp), dtype=np.int8)
    packed[:, :K] = Bp.T.astype(np.int8)
    return {"packed": packed, "col_scale": scale, "col_sum": Bp.sum(axis=0),
            "codes": Bp, "Kp": Kp}


# ----------------------------------------------------------------------------
# 4-bit half: q4_1 blocks in 32 x 256 tiles
# ----------------------------------------------------------------------------
#
# Q4 TILE FORMAT (5120 bytes per tile; tiles row-major over the grid
# [N/32][K/256]; tile (tr, tc) covers rows 32*tr.., columns 256*tc..)
#
#   bytes [0, 4096): codes.  Row r (0..31) owns bytes [128 r, 128 r + 128) as
#     8 blocks of 16 bytes: block b (columns 32 b .. 32 b + 31) sits at bytes
#     [128 r + 16 b, 128 r + 16 b + 16) as 4 little-endian uint32 words; word
#     t (t = 0..3) holds the codes of columns k = 32 b + 8 t + j, j = 0..7.
#     Inside the word, code j = 2i sits in bits [4i, 4i+4) and code j = 2i+1
#     in bits [16+4i, 16+4i+4), i = 0..3.
#   bytes [4096, 5120): 256 (scale, min) pairs of bf16.  The pair of (row r,
#     block b) is at byte 4096 + 4*(8 r + b): scale in the low 16 bits, min in
#     the high 16 bits.
#
#   Decoded weight: w[32 tr + r][256 tc + k] = q * scale + min.

TILE_ROWS, TILE_COLS, TILE_BYTES = 32, 256, 5120
BLOCK = 32


def q4_quantize_blocks(W):
    """Quantise fp32 W [N][K] to q4_1 blocks of 32 along K.

    Returns (q int64 [N][K], scale fp64 [N][K/32] (bf16 values), mn (same)).
    """
    W = _f32(np.asarray(W, np.float64))
    N, K = W.shape
    assert K % BLOCK == 0
    Wb = W.reshape(N, K // BLOCK, BLOCK)
    mx = Wb.max(axis=2)
    mnv = Wb.min(axis=2)
    s = bf16_rne(_f32(_f32(mx - mnv) / 15.0))
    m = bf16_rne(mnv)
    q = np.zeros(Wb.shape, dtype=np.int64)
    nz = s > 0
    diff = _f32(Wb - m[:, :, None])
    with np.errstate(divide="ignore", invalid="ignore"):
        u = _f32(diff / np.where(nz, s, 1.0)[:, :, None])
    qq = np.clip(np.rint(u), 0, 15).astype(np.int64)
    q[nz] = qq[nz]
    return q.reshape(N, K), s, m


def q4_tiles_from_blocks(q, s, m):
    """Write the tile bytes for codes q [N][K], scale/min [N][K/32] (bf16 values)."""
    q = np.asarray(q, np.int64)
    N, K = q.shape
    assert N % TILE_ROWS == 0 and K % TILE_COLS == 0
    assert q.min(initial=0) >= 0 and q.max(initial=0) <= 15
    TR, TC = N // TILE_ROWS, K // TILE_COLS
    out = np.zeros((TR, TC, TILE_BYTES), dtype=np.uint8)
    # codes: q[n, k] with n = 32 tr + r, k = 256 tc + 32 b + 8 t + j
    qv = q.reshape(TR, TILE_ROWS, TC, 8, 4, 8)        # tr, r, tc, b, t, j
    words = np.zeros((TR, TILE_ROWS, TC, 8, 4), dtype=np.uint64)
    for j in range(8):
        i, hi = divmod(j, 2)
        shift = 4 * i + (16 if hi else 0)
        words |= qv[..., j].astype(np.uint64) << np.uint64(shift)
    # word index within the row: 4 b + t
    words = words.transpose(0, 2, 1, 3, 4)            # tr, tc, r, b, t
    wbytes = words.astype(np.uint32).reshape(TR, TC, TILE_ROWS * 32).view(np.uint8)
    out[:, :, :4096] = wbytes.reshape(TR, TC, 4096)
    sb = bf16_bits(s).reshape(TR, TILE_ROWS, TC, 8)   # tr, r, tc, b
    mb = bf16_bits(m).reshape(TR, TILE_ROWS, TC, 8)
    pair = sb.astype(np.uint32) | (mb.astype(np.uint32) << 16)
    pair = pair.transpose(0, 2, 1, 3)                 # tr, tc, r, b
    out[:, :, 4096:] = pair.reshape(TR, TC, 256).astype(np.uint32).view(np.uint8).reshape(TR, TC, 1024)
    return out.reshape(-1)


def pack_q4(W):
    """fp32 W [N][K] -> tile bytes (uint8, TR*TC*5120)."""
    q, s, m = q4_quantize_blocks(W)
    return q4_tiles_from_blocks(q, s, m)


def q4_blocks_from_tiles(tiles, N, K):
    """Read tile bytes back into (q [N][K], scale [N][K/32], min [N][K/32])."""
    TR, TC = N // TILE_ROWS, K // TILE_COLS
    t = np.asarray(tiles, dtype=np.uint8).reshape(TR, TC, TILE_BYTES)
    words = t[:, :, :4096].copy().view(np.uint32).reshape(TR, TC, TILE_ROWS, 8, 4)  # tr tc r b t
    q = np.zeros((TR, TC, TILE_ROWS, 8, 4, 8), dtype=np.int64)  # tr tc r b t j
    w64 = words.astype(np.uint64)
    for j in range(8):
        i, hi = divmod(j, 2)
        shift = 4 * i + (16 if hi else 0)
        q[..., j] = ((w64 >> np.uint64(shift)) & np.uint64(0xF)).astype(np.int64)
    # k within tile = 32 b + 8 t + j
    q = q.transpose(0, 2, 1, 3, 4, 5).reshape(N, K)   # tr r tc b t j
    pairs = t[:, :, 4096:].copy().view(np.uint32).reshape(TR, TC, TILE_ROWS, 8)  # tr tc r b
    s = bf16_from_bits((pairs & 0xFFFF).astype(np.uint16))
    m = bf16_from_bits((pairs >> 16).astype(np.uint16))
    s = s.transpose(0, 2, 1, 3).reshape(N, K // BLOCK)  # tr r tc b
    m = m.transpose(0, 2, 1, 3).reshape(N, K // BLOCK)
    return q, s, m


def q4_decode(tiles, N, K):
    """Dense fp64 weights w[n][k] = q*scale + min (the "twin" of round 26)."""
    q, s, m = q4_blocks_from_tiles(tiles, N, K)
    return q.astype(np.float64) * np.repeat(s, BLOCK, axis=1) + np.repeat(m, BLOCK, axis=1)


def q4_gemm(tiles, N, K, X):
    """y[m][n] = sum_k x[m][k] w[n][k] in fp64, plus the normaliser sum_k |x||w|.

    X: activations [M][K] given as bf16 values (fp64 array).
    """
    W = q4_decode(tiles, N, K)
    X = np.asarray(X, np.float64)
    return X @ W.T, np.abs(X) @ np.abs(W).T


def q4_gemm_rows(tiles, N, K, X, rows):
    """Selected output columns n in ``rows`` only (cheap sampled checks)."""
    rows = np.asarray(rows)
    W = q4_decode_rows(tiles, N, K, rows)
    X = np.asarray(X, np.float64)
    return X @ W.T, np.abs(X) @ np.abs(W).T


def q4_decode_rows(tiles, N, K, rows):
    """Decode only the weight rows listed (each row lives in one tile row)."""
    rows = np.asarray(rows)
    out = np.empty((len(rows), K))
    TC = K // TILE_COLS
    t = np.asarray(tiles, dtype=np.uint8).reshape(N // TILE_ROWS, TC * TILE_BYTES)
    for i, n in enumerate(rows):
        tr, r = divmod(int(n), TILE_ROWS)
        sub = t[tr].reshape(TC * TILE_BYTES)
        W32 = q4_decode(sub, TILE_ROWS, K)
        out[i] = W32[r]
    return out


def moe_ids_view(ids_buf, ld_ids: int, n_used: int, T: int):
    """The strided top-k view: element (t, i) is ids_buf[t*ld_ids + i]
    (Zaya page, "The bugs that were the work": nb[1] = 17*4 bytes)."""
    flat = np.asarray(ids_buf).reshape(-1)
    return np.array([[int(flat[t * ld_ids + i]) for i in range(n_used)] for t in range(T)],
                    dtype=np.int64)


def q4_gemm_id(tiles_experts, n_expert, N, K, X, shared_src1: bool, ids_buf, ld_ids,
               n_used, T):
    """MUL_MAT_ID over q4 experts (Zaya page, round 24-25 MoE fix).

    tiles_experts: n_expert consecutive tile sets, each N x K.
    X: shared src1 [T][K] (gate/up) or per-slot [T][n_used][K] (down).
    dst[t][i][:] = W_{ids(t,i)} . src1(t, shared ? 0 : i).
    Returns (Y [T][n_used][N], norm [T][n_used][N]).
    """
    ids = moe_ids_view(ids_buf, ld_ids, n_used, T)
    assert ids.min(initial=0) >= 0 and ids.max(initial=0) < n_expert, "expert id out of range"
    per = (N // TILE_ROWS) * (K // TILE_COLS) * TILE_BYTES
    tiles_experts = np.asarray(tiles_experts, dtype=np.uint8).reshape(n_expert, per)
    X = np.asarray(X, np.float64)
    Y = np.zeros((T, n_used, N))
    Z = np.zeros((T, n_used, N))
    dense = {}
    for t in range(T):
        for i in range(n_used):
            e = int(ids[t, i])
            if e not in dense:
                dense[e] = q4_decode(tiles_experts[e], N, K)
            x = X[t] if shared_src1 else X[t, i]
            Y[t, i] = dense[e] @ x
            Z[t, i] = np.abs(dense[e]) @ np.abs(x)
    return Y, Z


def normalized_error(y_test, y_ref, norm):
    """max |y_test - y_ref| / sum_k |x||w|; where norm == 0, y_test must be 0."""
    y_test = np.asarray(y_test, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    norm = np.asarray(norm, np.float64)
    zero = norm == 0
    if np.any(zero) and np.any(y_test[zero] != 0):
        return float("inf")
    d = np.abs(y_test - y_ref)
    return float((d[~zero] / norm[~zero]).max(initial=0.0))


# ----------------------------------------------------------------------------
# W8A16: int8 weights with a scale for every 1,024 weights of a row, bf16 activations
# ----------------------------------------------------------------------------
# "llama.cpp-xdna -- CPU, iGPU and XDNA1 NPU on AMD Ryzen APUs", sections "The
# NPU worker" and "Running" (GGML_XDNA_NPU_W8): each 1,024-weight block of a
# row is int8 with its own scale, activations are bf16, and each scale
# multiplies its block's partial sum.  The per-block quantisation rule is packB's (amax/127, round half to
# even, clamp to +-127, zero block -> scale 0): the pages give the granularity,
# not the rounding.

W8_BLOCK = 1024


def pack_w8(W):
    """W: fp32 values [N][K] (weight rows).  Returns (codes int64 [N][K],
    scales fp64 holding fp32 values [N][ceil(K/1024)])."""
    W = _f32(np.asarray(W, np.float64))
    N, K = W.shape
    nb = (K + W8_BLOCK - 1) // W8_BLOCK
    q = np.zeros((N, K), dtype=np.int64)
    s = np.zeros((N, nb))
    for b in range(nb):
        blk = W[:, b * W8_BLOCK:(b + 1) * W8_BLOCK]
        sc = _f32(np.abs(blk).max(axis=1) / 127.0)
        s[:, b] = sc
        for n in range(N):
            if sc[n] > 0:
                q[n, b * W8_BLOCK:(b + 1) * W8_BLOCK] = np.clip(np.rint(_f32(blk[n] / sc[n])), -127, 127)
    return q, s


def w8_gemm(codes, scales, X):
    """Y[m][n] = sum_b scales[n][b] * sum_{k in block b} codes[n][k] * X[m][k], in fp64.
    Also returns the normaliser sum_k |x| |w| per output (w = code * scale)."""
    codes = np.asarray(codes, np.float64)
    X = np.asarray(X, np.float64)
    N, K = codes.shape
    M = X.shape[0]
    Y = np.zeros((M, N))
    norm = np.zeros((M, N))
    for b in range(scales.shape[1]):
        sl = slice(b * W8_BLOCK, min(K, (b + 1) * W8_BLOCK))
        Y += (X[:, sl] @ codes[:, sl].T) * scales[:, b][None, :]
        norm += (np.abs(X[:, sl]) @ np.abs(codes[:, sl]).T) * scales[:, b][None, :]
    return Y, norm


# ----------------------------------------------------------------------------
# More weight formats ("NPU engine: full ELFs, no xclbin", section "Q4NX
# chunks"): Q4_K repacked into q4_1 tiles, and 8-bit (Q8) tiles in the two
# code layouts that the section describes.
# ----------------------------------------------------------------------------
#
# Q4_K -> q4_1.  The section says the repack keeps the 4-bit codes and is exact
# apart from rounding S*scale and M*min to bf16.  The pages name Q4_K but do
# not print its bytes; the layout read here is GGML's published k-quant
# super-block (it must match the files the weights come from).  Per 256
# consecutive weights of one row, 144 bytes:
#   [0, 2)    d, fp16 (the super-block scale S of the 6-bit scale codes)
#   [2, 4)    dmin, fp16 (the super-block scale M of the 6-bit min codes)
#   [4, 16)   twelve bytes b[0..11] holding eight 6-bit scale codes sc_j and
#             eight 6-bit min codes mn_j, one pair per sub-block j of 32:
#               j < 4:  sc_j = b[j] & 63,   mn_j = b[j+4] & 63
#               j >= 4: sc_j = (b[j+4] & 15) | ((b[j-4] >> 6) << 4)
#                       mn_j = (b[j+4] >> 4) | ((b[j] >> 6) << 4)
#   [16, 144) 128 code bytes: weight 64c + l (c = 0..3, l = 0..31) is the low
#             nibble of byte 32c + l, weight 64c + 32 + l its high nibble.
#   Weight of sub-block j: w = d*sc_j*q - dmin*mn_j.
# The q4_1 block of sub-block j then has scale bf16(d*sc_j), min
# bf16(-(dmin*mn_j)) and the same codes.  Both products are exact in fp32 (an
# 11-bit significand times a 6-bit integer), so each is rounded once.

Q4K_SB, Q4K_BYTES = 256, 144


def q4k_fields(buf, N: int, K: int, row_bytes: int | None = None):
    """Parse Q4_K super-blocks of an N x K weight (rows of K/256 blocks,
    ``row_bytes`` apart; default contiguous).  Returns
    (d [N][K/256], dmin, sc [N][K/256][8], mn [N][K/256][8], q [N][K]),
    d and dmin as fp64, the codes as int64."""
    assert K % Q4K_SB == 0
    nsb = K // Q4K_SB
    if row_bytes is None:
        row_bytes = nsb * Q4K_BYTES
    raw = np.asarray(buf, dtype=np.uint8).reshape(-1)
    blk = np.stack([raw[n * row_bytes:n * row_bytes + nsb * Q4K_BYTES] for n in range(N)])
    blk = blk.reshape(N, nsb, Q4K_BYTES)
    d = blk[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = blk[:, :, 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    b = blk[:, :, 4:16].astype(np.int64)
    sc = np.zeros((N, nsb, 8), dtype=np.int64)
    mn = np.zeros((N, nsb, 8), dtype=np.int64)
    for j in range(8):
        if j < 4:
            sc[..., j] = b[..., j] & 63
            mn[..., j] = b[..., j + 4] & 63
        else:
            sc[..., j] = (b[..., j + 4] & 15) | ((b[..., j - 4] >> 6) << 4)
            mn[..., j] = (b[..., j + 4] >> 4) | ((b[..., j] >> 6) << 4)
    qs = blk[:, :, 16:].astype(np.int64).reshape(N, nsb, 4, 32)   # n, sb, c, l
    q = np.stack([qs & 15, qs >> 4], axis=3)                      # n, sb, c, half, l
    return d, dmin, sc, mn, q.reshape(N, K)


def q4k_decode(buf, N: int, K: int, row_bytes: int | None = None):
    """Dense fp64 weights of a Q4_K tensor: w = d*sc_j*q - dmin*mn_j."""
    d, dmin, sc, mn, q = q4k_fields(buf, N, K, row_bytes)
    scale = (d[:, :, None] * sc).reshape(N, K // BLOCK)
    mins = (dmin[:, :, None] * mn).reshape(N, K // BLOCK)
    return q * np.repeat(scale, BLOCK, axis=1) - np.repeat(mins, BLOCK, axis=1)


def repack_q4k(buf, N: int, K: int, row_bytes: int | None = None):
    """Q4_K -> q4_1 tile bytes: scale bf16(d*sc), min bf16(-(dmin*mn)), same codes."""
    d, dmin, sc, mn, q = q4k_fields(buf, N, K, row_bytes)
    s = bf16_rne(_f32((d[:, :, None] * sc).reshape(N, K // BLOCK)))
    m = bf16_rne(_f32(-(dmin[:, :, None] * mn).reshape(N, K // BLOCK)))
    return q4_tiles_from_blocks(q, s, m)


# Q8 tiles.  The section gives the two code layouts of a 32 x 256 tile:
#   layout 0: code (r, k) at byte k*32 + r;
#   layout 1: code (r, k) at byte (r/16)*4096 + (k/32)*512 + (k%32)*16 + r%16.
# It gives no scale bytes (it defers them to a header the pages do not hold), so these are
# the library's own: each tile is 8704 bytes, the 8192 code bytes followed by
# one bf16 scale per (row r, block g of 32 columns) at byte
# 8192 + 2*(32 g + r); codes are int8 and w = code * scale (the section rules
# out expressing Q8 as q4_1's code + min form).  Tiles are row-major over the [N/32][K/256] grid,
# as for q4.  Quantiser (the pages give none; packB's rule per block with the
# scale kept in bf16):
#   s = bf16(fl(amax / 127)); q = clamp(rint_even(fl(x / s)), -127, 127);
#   q = 0 where s == 0.

Q8_TILE_BYTES, Q8_CODE_BYTES = 8704, 8192


def q8_code_offsets(layout: int):
    """Byte offset of code (r, k) in a tile, as an int64 array [32][256]."""
    r = np.arange(TILE_ROWS, dtype=np.int64)[:, None]
    k = np.arange(TILE_COLS, dtype=np.int64)[None, :]
    if layout == 0:
        return k * 32 + r
    if layout == 1:
        return (r // 16) * 4096 + (k // 32) * 512 + (k % 32) * 16 + r % 16
    raise ValueError("Q8 layout is 0 or 1")


def q8_quantize_blocks(W):
    """fp32 W [N][K] -> (q int64 [N][K], scale fp64 bf16 values [N][K/32])."""
    W = _f32(np.asarray(W, np.float64))
    N, K = W.shape
    assert K % BLOCK == 0
    Wb = W.reshape(N, K // BLOCK, BLOCK)
    s = bf16_rne(_f32(np.abs(Wb).max(axis=2) / 127.0))
    nz = s > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        u = _f32(Wb / np.where(nz, s, 1.0)[:, :, None])
    q = np.where(nz[:, :, None], np.clip(np.rint(u), -127, 127), 0).astype(np.int64)
    return q.reshape(N, K), s


def q8_tiles_from_blocks(q, s, layout: int):
    q = np.asarray(q, np.int64)
    N, K = q.shape
    assert N % TILE_ROWS == 0 and K % TILE_COLS == 0
    assert q.min(initial=0) >= -128 and q.max(initial=0) <= 127
    TR, TC = N // TILE_ROWS, K // TILE_COLS
    off = q8_code_offsets(layout)
    out = np.zeros((TR, TC, Q8_TILE_BYTES), dtype=np.uint8)
    qt = q.reshape(TR, TILE_ROWS, TC, TILE_COLS).transpose(0, 2, 1, 3)   # tr tc r k
    codes = np.zeros((TR, TC, Q8_CODE_BYTES), dtype=np.uint8)
    codes[:, :, off] = (qt & 0xFF).astype(np.uint8)
    out[:, :, :Q8_CODE_BYTES] = codes
    sb = bf16_bits(s).reshape(TR, TILE_ROWS, TC, 8).transpose(0, 2, 3, 1)   # tr tc g r
    out[:, :, Q8_CODE_BYTES:] = sb.reshape(TR, TC, 256).astype(np.uint16).view(np.uint8).reshape(TR, TC, 512)
    return out.reshape(-1)


def pack_q8(W, layout: int):
    """fp32 W [N][K] -> Q8 tile bytes in the given code layout."""
    q, s = q8_quantize_blocks(W)
    return q8_tiles_from_blocks(q, s, layout)


def q8_blocks_from_tiles(tiles, N: int, K: int, layout: int):
    """Tile bytes -> (q int64 [N][K], scale fp64 [N][K/32])."""
    TR, TC = N // TILE_ROWS, K // TILE_COLS
    t = np.asarray(tiles, dtype=np.uint8).reshape(TR, TC, Q8_TILE_BYTES)
    off = q8_code_offsets(layout)
    q = t[:, :, :Q8_CODE_BYTES][:, :, off].view(np.int8).astype(np.int64)   # tr tc r k
    q = q.transpose(0, 2, 1, 3).reshape(N, K)
    sb = t[:, :, Q8_CODE_BYTES:].copy().view(np.uint16).reshape(TR, TC, 8, TILE_ROWS)   # tr tc g r
    s = bf16_from_bits(sb).transpose(0, 3, 1, 2).reshape(N, K // BLOCK)
    return q, s


def q8_decode(tiles, N: int, K: int, layout: int):
    """Dense fp64 weights w = code * scale."""
    q, s = q8_blocks_from_tiles(tiles, N, K, layout)
    return q.astype(np.float64) * np.repeat(s, BLOCK, axis=1)


def q8_gemm(tiles, N: int, K: int, X, layout: int):
    """y[m][n] = sum_k x[m][k] w[n][k] in fp64, plus the normaliser sum_k |x||w|."""
    W = q8_decode(tiles, N, K, layout)
    X = np.asarray(X, np.float64)
    return X @ W.T, np.abs(X) @ np.abs(W).T

"""Pins of the oracle's extra weight formats: Q4_K repacked into q4_1 tiles, and
8-bit (Q8) tiles in their two code layouts ("NPU engine: full ELFs, no
xclbin", section "Q4NX chunks").

Each pin checks the oracle against something other than its own formula: the
hand-decoded super-block and hand-worked layout offsets in tests/golden, an
encoder of the Q4_K scale bytes written here as the inverse map, the page's
rounding bound for the repack, and the integer special case of Q8."""
import os

import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O
from quantized_matmul_qmm_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kv(path):
    out = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split("=", 1)
        out[k.strip()] = v.strip()
    return out


# --------------------------------------------------------------------------
# Q4_K
# --------------------------------------------------------------------------

def _golden_block():
    g = _kv(os.path.join(GOLDEN, "q4k_superblock.txt"))
    blk = np.zeros(144, dtype=np.uint8)
    blk[:16] = [int(h, 16) for h in g["header"].split()]
    for item in g["code_bytes"].split():
        i, v = item.split(":")
        blk[16 + int(i)] = int(v, 16)
    sc = [int(x) for x in g["sc"].split()]
    mn = [int(x) for x in g["mn"].split()]
    w = {int(a): float(b) for a, b in (it.split(":") for it in g["weights"].split())}
    return blk, sc, mn, w


def test_q4k_hand_block_decodes_to_hand_values():
    blk, sc, mn, w = _golden_block()
    d, dmin, sc_o, mn_o, q = O.q4k_fields(blk, 1, 256)
    assert d[0, 0] == 0.5 and dmin[0, 0] == 0.25
    assert sc_o[0, 0].tolist() == sc
    assert mn_o[0, 0].tolist() == mn
    dec = O.q4k_decode(blk, 1, 256)[0]
    for k, v in w.items():
        assert dec[k] == v, (k, dec[k], v)


def test_q4k_hand_block_repacks_exactly():
    # d*sc and dmin*mn are small multiples of powers of two: exact in bf16
    blk, _, _, w = _golden_block()
    rows = np.tile(blk, 32)          # one tile needs 32 rows: the same block in each
    tiles = O.repack_q4k(rows, 32, 256)
    dec = O.q4_decode(tiles, 32, 256)
    ref = O.q4k_decode(rows, 32, 256)
    assert np.array_equal(dec, ref)
    for k, v in w.items():
        assert dec[7, k] == v


def _encode_scale_bytes(sc, mn):
    """Inverse of the 6-bit scale/min packing, written from the map's
    description: the low six bits of b[0..3] / b[4..7] are sc/mn of
    sub-blocks 0..3; sub-blocks 4..7 keep their low four bits in b[8..11]
    (scale low nibble, min high nibble) and their top two bits in the top two
    bits of b[0..3] (scale) and b[4..7] (min)."""
    b = [0] * 12
    for j in range(4):
        b[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        b[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        b[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return b


def test_q4k_scale_codes_round_trip_every_value():
    rng = np.random.default_rng(5)
    blocks = []
    expect = []
    for j in range(8):
        for v in range(64):
            sc = rng.integers(0, 64, 8)
            mn = rng.integers(0, 64, 8)
            sc[j] = v
            mn[7 - j] = 63 - v
            blk = np.zeros(144, dtype=np.uint8)
            blk[0:2] = np.array([1.0], np.float16).view(np.uint8)
            blk[4:16] = _encode_scale_bytes(sc, mn)
            blocks.append(blk)
            expect.append((sc.copy(), mn.copy()))
    buf = np.concatenate(blocks)
    n = len(blocks)
    _, _, sc_o, mn_o, _ = O.q4k_fields(buf, n, 256)
    for i, (sc, mn) in enumerate(expect):
        assert sc_o[i, 0].tolist() == sc.tolist()
        assert mn_o[i, 0].tolist() == mn.tolist()


def test_q4k_code_nibbles_round_trip():
    rng = np.random.default_rng(6)
    q = rng.integers(0, 16, 256)
    blk = np.zeros(144, dtype=np.uint8)
    for c in range(4):
        for l in range(32):
            blk[16 + 32 * c + l] = q[64 * c + l] | (q[64 * c + 32 + l] << 4)
    _, _, _, _, q_o = O.q4k_fields(blk, 1, 256)
    assert np.array_equal(q_o[0], q)


def test_q4k_repack_within_bf16_bound():
    N, K = 64, 1024
    buf = I.q4k_superblocks(11, N, K).numpy()
    d, dmin, sc, mn, q = O.q4k_fields(buf, N, K)
    ref = O.q4k_decode(buf, N, K)
    dec = O.q4_decode(O.repack_q4k(buf, N, K), N, K)
    s_abs = np.repeat(np.abs(d[:, :, None] * sc).reshape(N, K // 32), 32, axis=1)
    m_abs = np.repeat(np.abs(dmin[:, :, None] * mn).reshape(N, K // 32), 32, axis=1)
    # bf16 keeps 8 significant bits: each rounding moves a value by <= 2^-8 of it
    bound = 2.0 ** -8 * (q * s_abs + m_abs)
    err = np.abs(dec - ref)
    assert np.all(err <= bound * (1 + 1e-12))
    assert err.max() > 0   # the random scales do need rounding
    # codes are kept unchanged
    q_rep, _, _ = O.q4_blocks_from_tiles(O.repack_q4k(buf, N, K), N, K)
    assert np.array_equal(q_rep, q)


def test_q4k_row_stride():
    N, K = 32, 512
    buf = I.q4k_superblocks(12, N, K).numpy()
    row = K // 256 * 144
    padded = np.zeros((N, row + 48), dtype=np.uint8)
    padded[:, :row] = buf.reshape(N, row)
    padded[:, row:] = 0xAB
    assert np.array_equal(O.repack_q4k(padded, N, K, row + 48), O.repack_q4k(buf, N, K))


def test_q4k_planted_mistake_is_caught():
    """A decoder that swaps the nibble halves fails the hand block."""
    blk, _, _, w = _golden_block()
    swapped = blk.copy()
    swapped[16:] = ((blk[16:] >> 4) | (blk[16:] << 4)).astype(np.uint8)
    dec = O.q4k_decode(swapped, 1, 256)[0]
    assert any(dec[k] != v for k, v in w.items())


# --------------------------------------------------------------------------
# Q8 tiles
# --------------------------------------------------------------------------

def _golden_offsets():
    out = []
    for line in open(os.path.join(GOLDEN, "q8_tile_layouts.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append(tuple(int(x) for x in line.split()))
    return out


@pytest.mark.parametrize("layout", [0, 1])
def test_q8_layout_is_a_bijection(layout):
    off = O.q8_code_offsets(layout).reshape(-1)
    assert np.array_equal(np.sort(off), np.arange(8192))


def test_q8_one_hot_weights_land_on_the_hand_offsets():
    for layout, r, k, byte in _golden_offsets():
        W = np.zeros((32, 256), dtype=np.float32)
        W[r, k] = 0.75
        t = O.pack_q8(W, layout)
        nz = np.nonzero(t[:8192])[0]
        assert nz.tolist() == [byte], (layout, r, k, nz)
        assert t[byte] == 127
        # its scale sits at 8192 + 2 (32 g + r)
        sbits = t[8192:].view(np.uint16)
        g = k // 32
        assert np.nonzero(sbits)[0].tolist() == [32 * g + r]
        assert O.bf16_from_bits(sbits[32 * g + r]) == O.bf16_rne(np.float32(0.75) / np.float32(127))


def test_q8_layouts_decode_the_same_weights():
    W = I.q4_weights(21, 64, 512).numpy()
    a = O.q8_decode(O.pack_q8(W, 0), 64, 512, 0)
    b = O.q8_decode(O.pack_q8(W, 1), 64, 512, 1)
    assert np.array_equal(a, b)
    assert not np.array_equal(O.pack_q8(W, 0), O.pack_q8(W, 1))


def test_q8_quantiser_bound():
    W = I.q4_weights(22, 64, 1024).numpy().astype(np.float64)
    W[3, 32:64] = 0.0             # an all-zero block: scale 0, codes 0
    q, s = O.q8_quantize_blocks(W)
    assert np.all(q[3, 32:64] == 0) and s[3, 1] == 0
    assert np.abs(q).max() <= 127
    dec = O.q8_decode(O.pack_q8(W, 1), 64, 1024, 1)
    se = np.repeat(s, 32, axis=1)
    amax = np.repeat(np.abs(W.reshape(64, 32, 32)).max(axis=2), 32, axis=1)
    # within half a step, or (rounded-down bf16 scale) clamped at 127 s
    bound = np.maximum(0.5 * se, amax - 127 * se) * (1 + 2.0 ** -20) + 1e-12
    assert np.all(np.abs(W - dec) <= bound)


def test_q8_integer_weights_give_the_integer_gemm():
    # blocks whose amax is 127 get scale exactly 1: codes equal the weights
    rng = np.random.default_rng(7)
    N, K, M = 64, 512, 3
    W = rng.integers(-127, 128, (N, K)).astype(np.float64)
    W[:, ::32] = 127.0
    X = rng.integers(-40, 41, (M, K)).astype(np.float64)
    for layout in (0, 1):
        t = O.pack_q8(W, layout)
        q, s = O.q8_blocks_from_tiles(t, N, K, layout)
        assert np.all(s == 1.0) and np.array_equal(q, W.astype(np.int64))
        y, _ = O.q8_gemm(t, N, K, X, layout)
        assert np.array_equal(y, (X.astype(np.int64) @ W.astype(np.int64).T).astype(np.float64))


def test_q8_gemm_brute_force_tiny():
    W = I.q4_weights(23, 32, 256).numpy()
    X = I.q4_activations(24, 2, 256).float().numpy().astype(np.float64)
    t = O.pack_q8(W, 0)
    q, s = O.q8_quantize_blocks(W)
    y, norm = O.q8_gemm(t, 32, 256, X, 0)
    for m in range(2):
        for n in range(0, 32, 7):
            acc = 0.0
            for k in range(256):
                acc += X[m, k] * (q[n, k] * s[n, k // 32])
            assert abs(y[m, n] - acc) <= 1e-12 * norm[m, n]


def test_q8_quantiser_hand_worked_block():
    """A block with amax 127 has scale bf16(127/127) = 1, so the codes are the
    weights rounded half to even; amax 1.0 gives bf16(1/127) = 2^-7 * (1 + 2^-7)
    (bits 0x3C01), worked out by hand."""
    W = np.zeros((32, 256), dtype=np.float32)
    W[0, :8] = [127.0, 2.5, 3.5, -2.5, 126.5, -126.5, 0.5, -0.5]
    W[1, 32:35] = [1.0, -1.0, 0.5]
    q, s = O.q8_quantize_blocks(W)
    assert s[0, 0] == 1.0
    assert q[0, :8].tolist() == [127, 2, 4, -2, 126, -126, 0, 0]
    assert O.bf16_bits(s[1, 1]) == 0x3C01 and s[1, 1] == 2.0 ** -7 * (1 + 2.0 ** -7)
    # 1 / s = 127.0077.. -> 127; 0.5 / s = 63.5039.. -> 64
    assert q[1, 32:35].tolist() == [127, -127, 64]
    assert s[2, 0] == 0 and not q[2].any()


def test_q8_quantiser_against_torch():
    """Scales from torch's bf16 rounding of fp32 amax/127, codes from torch's
    half-to-even rounding of the fp32 quotient, clamped to +-127."""
    W = I.q4_weights(25, 64, 512)
    Wb = W.reshape(64, 16, 32)
    st = (Wb.abs().amax(2) / 127).to(torch.bfloat16).float()
    qt = torch.clamp(torch.round(Wb / st[:, :, None]), -127, 127)
    q, s = O.q8_quantize_blocks(W.numpy())
    assert np.array_equal(s, st.double().numpy())
    assert np.array_equal(q.reshape(64, 16, 32), qt.numpy().astype(np.int64))

"""GPU parity of the int8 half against the CPU oracle: packs byte-exact, GEMM
outputs bit-exact, on small odd shapes, on every workload at full size
(sampled rows where the oracle is slow), with canaries around the output."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O
from quantized_matmul_qmm_gb300 import inputs as I

pytestmark = pytest.mark.gpu

NP_IN = {"u8": np.uint8, "s8": np.int8}
T_IN = {"u8": torch.uint8, "s8": torch.int8}


def rand_codes(g, t, shape):
    if t == "u8":
        return torch.randint(0, 256, shape, generator=g, dtype=torch.int64).to(torch.uint8)
    return torch.randint(-128, 128, shape, generator=g, dtype=torch.int64).to(torch.int8)


def gpu_gemm(qmm, dev, A, a_type, zA, B, b_type, zB, out_type, bias=None, s_x=None,
             s_x_stride=0, s_w=None, s_y=1.0, zp_y=0, pad_cols=5, lda_pad=0):
    """Run pack + GEMM on the GPU with a canary-filled, padded output.
    Returns (out [M][N] numpy, packB outputs)."""
    M, K = A.shape
    N = B.shape[1]
    Bd = B.to(dev)
    packed, col_scale, col_sum = qmm.pack_b_int8(Bd, b_type)
    lda = (K + 15) // 16 * 16 + lda_pad
    Ad = torch.zeros((M, lda), dtype=A.dtype, device=dev)
    Ad[:, :K] = A.to(dev)
    Av = Ad[:, :K]                       # row stride lda, K columns
    ld = N + pad_cols
    canary = {"s32": 0x5A5A5A5A, "f32": float("nan"), "s8": 77, "u8": 201}[out_type]
    full = torch.full((M + 1, ld), canary if out_type != "f32" else 0.0,
                      dtype=qmm.TORCH_OUT[out_type], device=dev)
    if out_type == "f32":
        full.view(torch.int32).fill_(0x7FC0DEAD)
    out = full[:M, :N]
    if s_w is None and b_type == "f32":
        s_w = col_scale
    sx = None if s_x is None else torch.as_tensor(s_x, dtype=torch.float32).reshape(-1).to(dev)
    qmm.int8_gemm(Av, a_type, zA, packed, col_sum, N, b_type, zB, out_type,
                  bias=None if bias is None else bias.to(dev), s_x=sx, s_x_stride=s_x_stride,
                  s_w=None if s_w is None else s_w.to(dev), s_y=s_y, zp_y=zp_y, out=out)
    torch.cuda.synchronize()
    f = full.cpu()
    # canaries: padding columns and the extra row are untouched
    raw = f.view(torch.int32) if out_type == "f32" else f
    want = 0x7FC0DEAD if out_type == "f32" else canary
    assert torch.all(raw[:, N:] == want) and torch.all(raw[M, :] == want), "canary overwritten"
    return f[:M, :N].numpy(), (packed.cpu().numpy(), None if col_scale is None else col_scale.cpu().numpy(),
                                col_sum.cpu().numpy())


def oracle_out(A, a_type, zA, B, b_type, zB, out_type, bias=None, s_x=None, s_w=None, s_y=1.0,
               zp_y=0):
    An = A.numpy().astype(np.int64)
    Bn = B.numpy()
    if b_type == "f32":
        p = O.pack_b_int8(Bn, "f32")
        codes, s_w_o = p["codes"], p["col_scale"]
        r = O.int8_gemm_y(An, a_type, zA, codes, "s8", 0)
        sw = s_w_o if s_w is None else s_w
    else:
        r = O.int8_gemm_y(An, a_type, zA, Bn.astype(np.int64), b_type, zB)
        sw = s_w
    sw = None if sw is None else np.asarray(sw)
    return O.int8_epilogue(r["Y"], out_type, None if bias is None else bias.numpy(),
                           None if s_x is None else np.asarray(s_x, np.float64), sw, s_y, zp_y)


def assert_same(got, ref, out_type):
    if out_type == "f32":
        assert np.array_equal(got.astype(np.float32).view(np.int32),
                              ref.astype(np.float32).view(np.int32)), \
            f"max diff {np.abs(got - ref).max()}"
    else:
        bad = np.argwhere(got.astype(np.int64) != ref)
        assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:3].tolist()}"


@pytest.mark.parametrize("b_type", ["f32", "s8", "u8"])
@pytest.mark.parametrize("K,N", [(1, 1), (15, 7), (64, 32), (100, 33), (1024, 96), (1000, 130)])
def test_pack_b_int8_bytes(qmm, cuda, b_type, K, N):
    g = torch.Generator().manual_seed(K * 7 + N)
    if b_type == "f32":
        B = torch.randn((K, N), generator=g) * 0.02
        if N > 3:
            B[:, 3] = 0.0
    else:
        B = rand_codes(g, b_type, (K, N))
    packed, col_scale, col_sum = qmm.pack_b_int8(B.to(cuda), b_type)
    torch.cuda.synchronize()
    ref = O.pack_b_int8(B.numpy(), b_type)
    assert np.array_equal(packed.cpu().numpy(), ref["packed"])
    assert np.array_equal(col_sum.cpu().numpy().astype(np.int64), ref["col_sum"])
    if b_type == "f32":
        assert np.array_equal(col_scale.cpu().numpy().view(np.int32),
                              ref["col_scale"].astype(np.float32).view(np.int32))


SHAPES = [(1, 1, 1), (3, 15, 7), (16, 64, 32), (17, 65, 33), (33, 100, 40), (5, 1024, 96),
          (64, 257, 64), (100, 1000, 130)]


@pytest.mark.parametrize("a_type,b_type", [("u8", "s8"), ("s8", "s8"), ("u8", "u8"), ("s8", "u8"),
                                           ("s8", "f32"), ("u8", "f32")])
@pytest.mark.parametrize("M,K,N", SHAPES)
def test_gemm_s32_exact(qmm, cuda, a_type, b_type, M, K, N):
    g = torch.Generator().manual_seed(M * 1000 + K + N)
    A = rand_codes(g, a_type, (M, K))
    B = torch.randn((K, N), generator=g) * 0.02 if b_type == "f32" else rand_codes(g, b_type, (K, N))
    lo = {"u8": 0, "s8": -128}
    zA = int(torch.randint(lo[a_type], lo[a_type] + 256, (1,), generator=g))
    zB = 0 if b_type == "f32" else int(torch.randint(lo[b_type], lo[b_type] + 256, (1,), generator=g))
    got, _ = gpu_gemm(qmm, cuda, A, a_type, zA, B, b_type, zB, "s32")
    assert_same(got, oracle_out(A, a_type, zA, B, b_type, zB, "s32"), "s32")


@pytest.mark.parametrize("out_type", ["s32", "f32", "s8", "u8"])
@pytest.mark.parametrize("per_row", [False, True])
def test_gemm_epilogues_exact(qmm, cuda, out_type, per_row):
    g = torch.Generator().manual_seed(11)
    M, K, N = 37, 300, 70
    A = rand_codes(g, "u8", (M, K))
    B = rand_codes(g, "s8", (K, N))
    zA, zB = 133, -5
    bias = torch.randint(-20000, 20000, (N,), generator=g, dtype=torch.int32)
    s_w = (torch.rand(N, generator=g) * 9e-3 + 1e-3).float()
    s_x = (torch.rand(M, generator=g) * 0.02 + 0.01).float() if per_row else torch.tensor([1 / 64.0])
    s_y = 0.37
    zp = -7 if out_type == "s8" else 120
    got, _ = gpu_gemm(qmm, cuda, A, "u8", zA, B, "s8", zB, out_type, bias=bias, s_x=s_x,
                      s_x_stride=1 if per_row else 0, s_w=s_w, s_y=s_y, zp_y=zp)
    ref = oracle_out(A, "u8", zA, B, "s8", zB, out_type, bias=bias,
                     s_x=s_x.numpy() if per_row else float(s_x[0]), s_w=s_w.numpy(), s_y=s_y, zp_y=zp)
    assert_same(got, ref, out_type)


def test_page_zero_points(qmm, cuda, golden):
    # "The ONNX pack", "What works today": zp_x=-40, zp_w=-25, zp_y=-7 on 8x16x6
    c = golden("onnx_pack_qdq_constants.txt")
    for (M, K, N) in (c["proof_shape"], c["large_shape"]):
        g = torch.Generator().manual_seed(M + K + N)
        A = rand_codes(g, "s8", (M, K))
        B = rand_codes(g, "s8", (K, N))
        s_w = (torch.rand(N, generator=g) * 9e-3 + 1e-3).float()
        got, _ = gpu_gemm(qmm, cuda, A, "s8", c["zp_x"], B, "s8", c["zp_w"], "s8", s_x=[0.02],
                          s_w=s_w, s_y=0.05, zp_y=c["zp_y"])
        ref = oracle_out(A, "s8", c["zp_x"], B, "s8", c["zp_w"], "s8", s_x=0.02, s_w=s_w.numpy(),
                         s_y=0.05, zp_y=c["zp_y"])
        assert_same(got, ref, "s8")


def test_extreme_codes_exact(qmm, cuda):
    # every product -128 * -128 with K = 4608: |S| = 4608 * 16384, far beyond 2^24
    M, K, N = 32, 4608, 64
    A = torch.zeros((M, K), dtype=torch.uint8)             # A' = -128
    B = torch.full((K, N), -128, dtype=torch.int8)
    B[:, 1::2] = 127
    got, _ = gpu_gemm(qmm, cuda, A, "u8", 0, B, "s8", 0, "s32")
    assert_same(got, oracle_out(A, "u8", 0, B, "s8", 0, "s32"), "s32")


def test_workload_int8_m16(qmm, cuda):
    c = I.int8_gemm_small()
    for out_type, s_w in (("s32", None), ("f32", c.s_w)):
        got, _ = gpu_gemm(qmm, cuda, c.A, c.a_type, c.zA, c.B, c.b_type, c.zB, out_type, s_w=s_w)
        assert_same(got, oracle_out(c.A, c.a_type, c.zA, c.B, c.b_type, c.zB, out_type,
                                    s_w=None if s_w is None else s_w.numpy()), out_type)


@pytest.mark.parametrize("idx", range(7))
def test_workload_qwen_projection_m32(qmm, cuda, idx):
    c = I.int8_qwen_projection(idx)
    got, (packed, col_scale, col_sum) = gpu_gemm(qmm, cuda, c.A, c.a_type, c.zA, c.B, c.b_type,
                                                 c.zB, "f32", s_x=[c.s_x])
    ref = oracle_out(c.A, c.a_type, c.zA, c.B, c.b_type, c.zB, "f32", s_x=c.s_x)
    assert_same(got, ref, "f32")


def test_workload_large_sampled(qmm, cuda):
    """M=4096 K=N=4608 uint8 x int8, int8 output, in the launch configuration
    the benchmark times: one row from every 128-row half of each 256-row pair
    tile (so every one of the 288 output tiles and both CTAs' halves of it are
    compared, including the tiles each CTA pair reaches on its later passes),
    plus the first, last and tile-boundary rows, each in full; and the column
    sums exactly."""
    c = I.int8_gemm_large()
    dev = cuda
    Bd = c.B.to(dev)
    packed, _, col_sum = qmm.pack_b_int8(Bd, c.b_type)
    out = qmm.int8_gemm(c.A.to(dev), c.a_type, c.zA, packed, col_sum, c.N, c.b_type, c.zB,
                        "s8", bias=c.bias.to(dev), s_x=torch.tensor([c.s_x], device=dev),
                        s_w=c.s_w.to(dev), s_y=c.s_y, zp_y=c.zp_y)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    rng = np.random.default_rng(8)
    halves = np.arange(0, 4096, 128) + rng.integers(0, 128, 32)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, 2047, 2048, 4095], halves]))
    ref = oracle_out(c.A[rows], c.a_type, c.zA, c.B, c.b_type, c.zB, "s8", bias=c.bias,
                     s_x=c.s_x, s_w=c.s_w.numpy(), s_y=c.s_y, zp_y=c.zp_y)
    assert_same(got[rows], ref, "s8")
    # the workload exercises rounding and both clamps
    assert (got == 127).mean() > 0.001 and (got == -128).mean() > 0.001
    assert np.array_equal(col_sum.cpu().numpy().astype(np.int64), c.B.numpy().astype(np.int64).sum(0))
    # the same call with the weights widened once beforehand: the whole output identical
    b16 = qmm.widen_b_int8(packed, c.K, c.N)
    out2 = qmm.int8_gemm(c.A.to(dev), c.a_type, c.zA, packed, col_sum, c.N, c.b_type, c.zB,
                         "s8", bias=c.bias.to(dev), s_x=torch.tensor([c.s_x], device=dev),
                         s_w=c.s_w.to(dev), s_y=c.s_y, zp_y=c.zp_y, b16=b16)
    assert torch.equal(out2, out)


# ---------------------------------------------------------------------------
# tensor-core route (M >= 65): same function, bit-exact
# ---------------------------------------------------------------------------
UMMA_SHAPES = [(65, 300, 200), (96, 1088, 64), (128, 4608, 300), (200, 1000, 257), (256, 64, 256), (300, 1000, 300), (257, 4608, 130),
               (512, 2048, 520), (520, 130, 64), (1300, 2050, 1000)]


@pytest.mark.parametrize("a_type,b_type", [("u8", "s8"), ("s8", "u8"), ("u8", "f32")])
@pytest.mark.parametrize("M,K,N", UMMA_SHAPES)
def test_umma_route_s32_exact(qmm, cuda, a_type, b_type, M, K, N):
    assert qmm.int8_gemm_workspace_size(M, K, N) > 0
    g = torch.Generator().manual_seed(M + 7 * K + N)
    A = rand_codes(g, a_type, (M, K))
    B = torch.randn((K, N), generator=g) * 0.02 if b_type == "f32" else rand_codes(g, b_type, (K, N))
    zA = 200 if a_type == "u8" else -90
    zB = 0 if b_type == "f32" else 3
    got, _ = gpu_gemm(qmm, cuda, A, a_type, zA, B, b_type, zB, "s32")
    assert_same(got, oracle_out(A, a_type, zA, B, b_type, zB, "s32"), "s32")


def test_umma_route_more_tiles_than_pairs_exact(qmm, cuda):
    """110 output tiles of 256 x 256 (10 x 11), more than the CTA pairs that fit
    on the GPU, so pairs walk several tiles, alternate their two accumulators
    across tiles and prefetch the next tile's column constants; K = 1088
    crosses a 1024-k accumulator chunk.  Every element against the oracle."""
    M, K, N = 2560, 1088, 2816
    g = torch.Generator().manual_seed(2560)
    A = rand_codes(g, "u8", (M, K))
    B = rand_codes(g, "s8", (K, N))
    bias = torch.randint(-20000, 20000, (N,), generator=g, dtype=torch.int32)
    s_w = (torch.rand(N, generator=g) * 9e-3 + 1e-3).float()
    got, _ = gpu_gemm(qmm, cuda, A, "u8", 130, B, "s8", 5, "s8", bias=bias, s_x=[1.0 / 64], s_w=s_w,
                      s_y=0.1, zp_y=3)
    ref = oracle_out(A, "u8", 130, B, "s8", 5, "s8", bias=bias, s_x=1.0 / 64, s_w=s_w.numpy(), s_y=0.1, zp_y=3)
    assert_same(got, ref, "s8")
    assert (got == 127).any() and (got == -128).any()


@pytest.mark.parametrize("out_type", ["f32", "s8", "u8"])
def test_umma_route_epilogues_exact(qmm, cuda, out_type):
    g = torch.Generator().manual_seed(21)
    M, K, N = 384, 777, 260
    A = rand_codes(g, "u8", (M, K))
    B = rand_codes(g, "s8", (K, N))
    bias = torch.randint(-50000, 50000, (N,), generator=g, dtype=torch.int32)
    s_w = (torch.rand(N, generator=g) * 9e-3 + 1e-3).float()
    s_x = (torch.rand(M, generator=g) * 0.02 + 0.01).float()
    got, _ = gpu_gemm(qmm, cuda, A, "u8", 140, B, "s8", -6, out_type, bias=bias, s_x=s_x, s_x_stride=1,
                      s_w=s_w, s_y=0.61, zp_y=5 if out_type != "f32" else 0)
    ref = oracle_out(A, "u8", 140, B, "s8", -6, out_type, bias=bias, s_x=s_x.numpy(), s_w=s_w.numpy(),
                     s_y=0.61, zp_y=5 if out_type != "f32" else 0)
    assert_same(got, ref, out_type)


@pytest.mark.parametrize("pattern", ["all_extreme", "mixed_magnitudes"])
def test_umma_fp32_accumulation_is_exact(qmm, cuda, pattern):
    """The tensor-core route carries the integer sum in fp32 chunks of 1024 K.
    Adversarial operands: partial sums near 2^24 inside a chunk, mixed with
    products of 1, so a dropped low bit anywhere shows up as a mismatch."""
    M, K, N = 256, 4608, 256
    if pattern == "all_extreme":
        A = torch.zeros((M, K), dtype=torch.uint8)                  # A' = -128
        B = torch.full((K, N), -128, dtype=torch.int8)
        B[:, 1::3] = 127
    else:
        g = torch.Generator().manual_seed(5)
        kk = torch.arange(K)
        big = (kk % 16) < 8
        A = torch.where(big, torch.zeros(K, dtype=torch.int64), 129 + (kk % 3)).repeat(M, 1)
        A = (A + torch.randint(0, 2, (M, K), generator=g) * (~big).long()).to(torch.uint8)
        B = torch.where(big[:, None], torch.full((K, N), -128), torch.randint(1, 3, (K, N), generator=g))
        B = B.to(torch.int8)
    got, _ = gpu_gemm(qmm, cuda, A, "u8", 128, B, "s8", 0, "s32")
    assert_same(got, oracle_out(A, "u8", 128, B, "s8", 0, "s32"), "s32")


@pytest.mark.parametrize("K,N", [(100, 37), (4608, 300), (1, 5)])
def test_widen_b_int8_bytes(qmm, cuda, K, N):
    """The one-time f16 copy of the packed weights holds every packed code
    exactly, the padding columns as zeros."""
    g = torch.Generator().manual_seed(K + N)
    B = rand_codes(g, "s8", (K, N))
    packed, _, _ = qmm.pack_b_int8(B.to(cuda), "s8")
    b16 = qmm.widen_b_int8(packed, K, N)
    torch.cuda.synchronize()
    assert b16.shape == packed.shape
    assert torch.equal(b16.cpu(), packed.cpu().to(torch.float16))


@pytest.mark.parametrize("M,K,N,out_type", [(65, 300, 200, "s32"), (257, 4607, 130, "s8"), (512, 2048, 520, "f32"),
                                            (2560, 1088, 2816, "u8"), (16, 1024, 64, "s32")])
def test_gemm_with_widened_weights_exact(qmm, cuda, M, K, N, out_type):
    """qmm_int8_gemm_b16 (weights widened once beforehand) against the oracle,
    bit-exact: tensor-core shapes with ragged K and N, more tiles than CTA
    pairs, every output type, and one small-M call (which ignores the copy)."""
    g = torch.Generator().manual_seed(3 * M + K + N)
    A = rand_codes(g, "u8", (M, K))
    B = rand_codes(g, "s8", (K, N))
    bias = torch.randint(-20000, 20000, (N,), generator=g, dtype=torch.int32)
    s_w = (torch.rand(N, generator=g) * 9e-3 + 1e-3).float()
    s_y = 0.1 if out_type in ("s8", "u8") else 1.0
    packed, _, col_sum = qmm.pack_b_int8(B.to(cuda), "s8")
    b16 = qmm.widen_b_int8(packed, K, N)
    sx = torch.tensor([1.0 / 64], device=cuda)
    Ad = torch.zeros((M, (K + 15) // 16 * 16), dtype=torch.uint8, device=cuda)   # row stride a multiple of 16
    Ad[:, :K] = A.to(cuda)
    out = qmm.int8_gemm(Ad[:, :K], "u8", 131, packed, col_sum, N, "s8", -4, out_type, bias=bias.to(cuda), s_x=sx,
                        s_w=s_w.to(cuda), s_y=s_y, zp_y=3 if out_type == "u8" else 0, b16=b16)
    torch.cuda.synchronize()
    ref = oracle_out(A, "u8", 131, B, "s8", -4, out_type, bias=bias, s_x=1.0 / 64, s_w=s_w.numpy(), s_y=s_y,
                     zp_y=3 if out_type == "u8" else 0)
    assert_same(out.cpu().numpy(), ref, out_type)


def test_umma_route_tail_and_edge_rows_exact(qmm, cuda):
    """The tensor-core route widens the weight tiles in shared memory and the
    activations in a pass before the GEMM: K not a multiple of 64 (the bytes
    past K count as 0), M and N past the last full tile, extreme codes, row
    sums over a ragged K."""
    for (M, K, N, zA, zB) in [(257, 65, 300, 255, -8), (300, 4607, 130, 0, 8), (513, 1, 257, 7, 3)]:
        g = torch.Generator().manual_seed(M + K + N)
        A = rand_codes(g, "u8", (M, K))
        A[0] = 0
        A[1] = 255
        B = rand_codes(g, "s8", (K, N))
        B[:, 0] = -128
        got, _ = gpu_gemm(qmm, cuda, A, "u8", zA, B, "s8", zB, "s32")
        assert_same(got, oracle_out(A, "u8", zA, B, "s8", zB, "s32"), "s32")


# ---------------------------------------------------------------------------
# small-M routes (M <= 64): f16 MMA on exact integer codes; the streaming
# form (one CTA per SM, weight rows through a shared-memory ring) when the
# rows fit its shared memory, else clusters of 8 CTAs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,K", [(16, 1024), (32, 2048), (48, 4608), (64, 4608), (16, 20000)])
def test_small_route_extreme_codes_exact(qmm, cuda, M, K):
    """Every product at its largest magnitude (A' = B' = -128, with one row at
    A' = +127 and one column at B' = +127): the fp32 chunks of 1024 k reach
    2^24 exactly and are drained into int32; K = 20000 spans 20 chunks."""
    N = 72
    A = torch.zeros((M, K), dtype=torch.uint8)
    A[1] = 255
    B = torch.full((K, N), -128, dtype=torch.int8)
    B[:, 1] = 127
    got, _ = gpu_gemm(qmm, cuda, A, "u8", 128, B, "s8", 0, "s32")
    assert_same(got, oracle_out(A, "u8", 128, B, "s8", 0, "s32"), "s32")


@pytest.mark.parametrize("M,K,N", [(64, 2200, 2500), (64, 2300, 2500), (1, 10500, 2500), (1, 10600, 2500),
                                   (17, 3300, 2500), (33, 17, 2500), (48, 1000, 4099)])
def test_small_route_form_boundaries_exact(qmm, cuda, M, K, N):
    """Enough columns for the streaming form (at least one 16-column item per
    SM), on both sides of its shared-memory limit (the largest padded K for 64
    rows and for one row, and just past each: those take the cluster form), a
    K of one 64-step (seven of the eight warps idle), a ragged last item;
    extreme codes in a row and a column, zero points on both sides."""
    g = torch.Generator().manual_seed(3 * M + K + N)
    A = rand_codes(g, "u8", (M, K))
    A[0] = 255
    B = rand_codes(g, "s8", (K, N))
    B[:, 0] = -128
    got, _ = gpu_gemm(qmm, cuda, A, "u8", 201, B, "s8", -7, "s32")
    assert_same(got, oracle_out(A, "u8", 201, B, "s8", -7, "s32"), "s32")


@pytest.mark.parametrize("K", [3000, 1000])
@pytest.mark.parametrize("a_type,b_type,out_type", [("u8", "s8", "s8"), ("s8", "u8", "f32"), ("u8", "f32", "u8")])
def test_small_route_stream_epilogues_exact(qmm, cuda, a_type, b_type, out_type, K):
    """The streaming form with every operand type, both zero points (row sums),
    bias, per-row s_x and each output type: M = 32, N = 2600; K = 3000 keeps
    A as int8 codes (three chunks of the ring, the last one ragged), K = 1000
    widens A to f16 once (a ragged last 64-k block)."""
    M, N = 32, 2600
    g = torch.Generator().manual_seed(91)
    A = rand_codes(g, a_type, (M, K))
    B = torch.randn((K, N), generator=g) * 0.02 if b_type == "f32" else rand_codes(g, b_type, (K, N))
    zA = 37 if a_type == "u8" else -21
    zB = 0 if b_type == "f32" else (200 if b_type == "u8" else 5)
    bias = torch.randint(-5000, 5000, (N,), generator=g, dtype=torch.int32)
    s_x = (torch.rand(M, generator=g) * 0.01 + 0.001).numpy()
    s_w = (torch.rand(N, generator=g) * 9e-3 + 1e-3).float()
    s_y = 40.0 if out_type in ("s8", "u8") else 1.0
    got, _ = gpu_gemm(qmm, cuda, A, a_type, zA, B, b_type, zB, out_type, bias=bias, s_x=s_x, s_x_stride=1,
                      s_w=s_w, s_y=s_y, zp_y=3 if out_type == "u8" else -2)
    ref = oracle_out(A, a_type, zA, B, b_type, zB, out_type, bias=bias, s_x=s_x, s_w=s_w.numpy(), s_y=s_y,
                     zp_y=3 if out_type == "u8" else -2)
    assert_same(got, ref, out_type)


@pytest.mark.parametrize("a_type,b_type,out_type", [("u8", "s8", "s8"), ("s8", "u8", "f32"), ("u8", "f32", "u8")])
@pytest.mark.parametrize("M,K,N", [(64, 4608, 200), (48, 3000, 65), (2, 130, 1), (31, 20000, 100), (40, 1000, 130)])
def test_small_route_epilogues_exact(qmm, cuda, a_type, b_type, out_type, M, K, N):
    """Zero points on both sides (row sums needed), bias, per-row s_x, every
    output type; K not a multiple of 64 and N not a multiple of 64."""
    g = torch.Generator().manual_seed(M + K + N)
    A = rand_codes(g, a_type, (M, K))
    B = torch.randn((K, N), generator=g) * 0.02 if b_type == "f32" else rand_codes(g, b_type, (K, N))
    zA = 37 if a_type == "u8" else -21
    zB = 0 if b_type == "f32" else (200 if b_type == "u8" else 5)
    bias = torch.randint(-5000, 5000, (N,), generator=g, dtype=torch.int32)
    s_x = (torch.rand(M, generator=g) * 0.01 + 0.001).numpy()
    s_w = (torch.rand(N, generator=g) * 9e-3 + 1e-3).float()
    s_y = 40.0 if out_type in ("s8", "u8") else 1.0
    got, _ = gpu_gemm(qmm, cuda, A, a_type, zA, B, b_type, zB, out_type, bias=bias, s_x=s_x, s_x_stride=1,
                      s_w=s_w, s_y=s_y, zp_y=3 if out_type == "u8" else -2)
    ref = oracle_out(A, a_type, zA, B, b_type, zB, out_type, bias=bias, s_x=s_x, s_w=s_w.numpy(), s_y=s_y,
                     zp_y=3 if out_type == "u8" else -2)
    assert_same(got, ref, out_type)

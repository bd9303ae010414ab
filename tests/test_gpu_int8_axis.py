"""GPU parity of the int8 GEMM with per-axis zero points (one per activation
row, one per weight column; "The ONNX pack...", "What works today"): bit-exact
against the oracle for every output type, on both GEMM routes (legacy MMA for
M < 256, tensor cores above), on the page's 8 x 16 x 6 per-axis proof shape
and at M=4096 K=N=4608 (sampled rows), with canaries around the output."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O
from quantized_matmul_qmm_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def codes(g, t, shape):
    if t == "u8":
        return torch.randint(0, 256, shape, generator=g, dtype=torch.int64)
    return torch.randint(-128, 128, shape, generator=g, dtype=torch.int64)


def run_axis(qmm, dev, A, a_type, zA, B, b_type, zB, out_type, bias=None, s_x=None, s_x_stride=0, s_w=None,
             s_y=1.0, zp_y=0, status=None):
    """A [M][K], B [K][N] int64 codes (CPU); zA [M] / zB [N] int64 or None."""
    M, K = A.shape
    N = B.shape[1]
    tA = torch.uint8 if a_type == "u8" else torch.int8
    tB = torch.uint8 if b_type == "u8" else torch.int8
    packed, _, col_sum = qmm.pack_b_int8(B.to(tB).to(dev), b_type)
    lda = (K + 15) // 16 * 16
    Ad = torch.zeros((M, lda), dtype=tA, device=dev)
    Ad[:, :K] = A.to(tA).to(dev)
    canary = {"s32": 0x5A5A5A5A, "f32": 0, "s8": 77, "u8": 201}[out_type]
    full = torch.full((M + 1, N + 3), canary, dtype=qmm.TORCH_OUT[out_type], device=dev)
    if out_type == "f32":
        full.view(torch.int32).fill_(0x7FC0DEAD)
    dz = lambda z: None if z is None else z.to(torch.int32).to(dev)
    qmm.int8_gemm_axis_zp(Ad[:, :K], a_type, dz(zA), packed, col_sum, N, b_type, dz(zB), out_type,
                          bias=None if bias is None else bias.to(torch.int32).to(dev),
                          s_x=None if s_x is None else torch.as_tensor(s_x, dtype=torch.float32).reshape(-1).to(dev),
                          s_x_stride=s_x_stride, s_w=None if s_w is None else s_w.to(dev), s_y=s_y, zp_y=zp_y,
                          out=full[:M, :N], dev_status=status)
    torch.cuda.synchronize()
    f = full.cpu()
    raw = f.view(torch.int32) if out_type == "f32" else f
    want = 0x7FC0DEAD if out_type == "f32" else canary
    assert torch.all(raw[:, N:] == want) and torch.all(raw[M, :] == want), "canary overwritten"
    return f[:M, :N].numpy()


def oracle_axis(A, a_type, zA, B, b_type, zB, out_type, bias=None, s_x=None, s_w=None, s_y=1.0, zp_y=0):
    M, N = A.shape[0], B.shape[1]
    za = np.zeros(M, np.int64) if zA is None else zA.numpy()
    zb = np.zeros(N, np.int64) if zB is None else zB.numpy()
    r = O.int8_gemm_y_axis(A.numpy(), a_type, za, B.numpy(), b_type, zb)
    return O.int8_epilogue(r["Y"], out_type, None if bias is None else bias.numpy(),
                           None if s_x is None else np.asarray(s_x, np.float64),
                           None if s_w is None else s_w.numpy(), s_y, zp_y)


def same(got, ref, out_type):
    if out_type == "f32":
        assert np.array_equal(got.astype(np.float32).view(np.int32), ref.astype(np.float32).view(np.int32))
    else:
        bad = np.argwhere(got.astype(np.int64) != ref)
        assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:3].tolist()}"


def epilogue_args(g, M, N, out_type, Y_scale):
    bias = codes(g, "s8", (N,)) * 37
    s_x = (torch.rand(M, generator=g, dtype=torch.float64) * 0.02 + 0.01).float()
    s_w = (torch.rand(N, generator=g, dtype=torch.float64) * 0.009 + 0.001).float()
    s_y = float(Y_scale * 0.02 * 0.005 / 40.0)
    return dict(bias=bias, s_x=s_x.numpy(), s_x_stride=1, s_w=s_w, s_y=s_y, zp_y=-7 if out_type == "s8" else 128)


@pytest.mark.parametrize("a_type,b_type", [("u8", "s8"), ("s8", "s8"), ("u8", "u8"), ("s8", "u8")])
@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (5, 33, 7), (37, 1000, 130), (300, 1000, 260), (512, 2048, 520)])
@pytest.mark.parametrize("out_type", ["s32", "f32", "s8", "u8"])
def test_axis_zp_exact(qmm, cuda, a_type, b_type, M, K, N, out_type):
    g = torch.Generator().manual_seed(M * 7 + K * 13 + N + len(out_type))
    A, B = codes(g, a_type, (M, K)), codes(g, b_type, (K, N))
    zA, zB = codes(g, a_type, (M,)), codes(g, b_type, (N,))
    kw = {} if out_type == "s32" else epilogue_args(g, M, N, out_type, float(np.sqrt(K)) * 128 * 64)
    if out_type == "s32":
        kw = dict(bias=codes(g, "s8", (N,)) * 1000)
    kw_o = {k: v for k, v in kw.items() if k != "s_x_stride"}
    got = run_axis(qmm, cuda, A, a_type, zA, B, b_type, zB, out_type, **kw)
    same(got, oracle_axis(A, a_type, zA, B, b_type, zB, out_type, **kw_o), out_type)


def test_axis_zp_page_proof_shape(qmm, cuda, golden):
    """8 row zero points and 6 column zero points on the 8 x 16 x 6 proof shape,
    per-axis scales and zp_y, int8 out."""
    gd = golden("onnx_pack_qdq_constants.txt")
    M, K, N = gd["proof_shape"]
    g = torch.Generator().manual_seed(11)
    A, B = codes(g, "s8", (M, K)), codes(g, "s8", (K, N))
    zA = gd["zp_x"] + torch.randint(-3, 4, (M,), generator=g)
    zB = gd["zp_w"] + torch.randint(-3, 4, (N,), generator=g)
    s_x = (torch.rand(M, generator=g, dtype=torch.float64) * 0.02 + 0.01).float().numpy()
    s_w = (torch.rand(N, generator=g, dtype=torch.float64) * 0.009 + 0.001).float()
    kw = dict(s_x=s_x, s_w=s_w, s_y=0.002, zp_y=gd["zp_y"])
    got = run_axis(qmm, cuda, A, "s8", zA, B, "s8", zB, "s8", s_x_stride=1, **kw)
    same(got, oracle_axis(A, "s8", zA, B, "s8", zB, "s8", **kw), "s8")


def test_axis_zp_null_and_constant_match_per_tensor(qmm, cuda):
    """NULL arrays mean zero points of 0, and constant arrays reproduce
    qmm_int8_gemm with that per-tensor zero point, bit for bit."""
    g = torch.Generator().manual_seed(12)
    M, K, N = 300, 700, 96
    A, B = codes(g, "u8", (M, K)), codes(g, "s8", (K, N))
    got0 = run_axis(qmm, cuda, A, "u8", None, B, "s8", None, "s32")
    same(got0, oracle_axis(A, "u8", None, B, "s8", None, "s32"), "s32")
    packed, _, col_sum = qmm.pack_b_int8(B.to(torch.int8).to(cuda), "s8")
    Ad = torch.zeros((M, 704), dtype=torch.uint8, device=cuda)
    Ad[:, :K] = A.to(torch.uint8).to(cuda)
    ref = qmm.int8_gemm(Ad[:, :K], "u8", 131, packed, col_sum, N, "s8", -5, "s32")
    got = qmm.int8_gemm_axis_zp(Ad[:, :K], "u8", torch.full((M,), 131, dtype=torch.int32, device=cuda), packed,
                                col_sum, N, "s8", torch.full((N,), -5, dtype=torch.int32, device=cuda), "s32")
    torch.cuda.synchronize()
    assert torch.equal(ref, got)


def test_axis_zp_fp32_weights(qmm, cuda):
    """Symmetric fp32 weights (packB quantises them): row zero points only."""
    g = torch.Generator().manual_seed(13)
    M, K, N = 40, 300, 50
    A = codes(g, "u8", (M, K))
    W = torch.randn((K, N), generator=g) * 0.02
    zA = codes(g, "u8", (M,))
    packed, col_scale, col_sum = qmm.pack_b_int8(W.to(cuda), "f32")
    Ad = torch.zeros((M, 304), dtype=torch.uint8, device=cuda)
    Ad[:, :K] = A.to(torch.uint8).to(cuda)
    got = qmm.int8_gemm_axis_zp(Ad[:, :K], "u8", zA.to(torch.int32).to(cuda), packed, col_sum, N, "f32", None,
                                "f32", s_w=col_scale)
    torch.cuda.synchronize()
    p = O.pack_b_int8(W.numpy(), "f32")
    r = O.int8_gemm_y_axis(A.numpy(), "u8", zA.numpy(), p["codes"], "s8", np.zeros(N, np.int64))
    ref = O.int8_epilogue(r["Y"], "f32", None, None, p["col_scale"])
    same(got.cpu().numpy(), ref, "f32")


def test_axis_zp_out_of_domain_sets_status(qmm, cuda):
    g = torch.Generator().manual_seed(14)
    M, K, N = 8, 64, 16
    A, B = codes(g, "u8", (M, K)), codes(g, "s8", (K, N))
    zA = codes(g, "u8", (M,))
    zA[3] = 300                                  # outside 0..255
    st = torch.zeros(1, dtype=torch.int32, device=cuda)
    run_axis(qmm, cuda, A, "u8", zA, B, "s8", None, "s32", status=st)
    assert int(st.item()) == qmm.QMM_ERR_INVALID_ARG
    st.zero_()
    zB = codes(g, "s8", (N,))
    zB[5] = -129                                 # outside -128..127
    run_axis(qmm, cuda, A, "u8", None, B, "s8", zB, "s32", status=st)
    assert int(st.item()) == qmm.QMM_ERR_INVALID_ARG


def test_axis_zp_large_sampled(qmm, cuda):
    """M=4096 K=N=4608 uint8 x int8 with random per-axis zero points, per-row
    s_x, bias, int8 out: 12 sampled rows against the oracle."""
    c = I.int8_gemm_large()
    g = torch.Generator().manual_seed(15)
    zA = codes(g, "u8", (c.M,))
    zB = torch.randint(-8, 9, (c.N,), generator=g)
    s_x = (torch.rand(c.M, generator=g, dtype=torch.float64) * 0.01 + 1.0 / 64).float()
    packed, _, col_sum = qmm.pack_b_int8(c.B.to(cuda), c.b_type)
    Ad = c.A.to(cuda)
    out = qmm.int8_gemm_axis_zp(Ad, c.a_type, zA.to(torch.int32).to(cuda), packed, col_sum, c.N, c.b_type,
                                zB.to(torch.int32).to(cuda), "s8", bias=c.bias.to(cuda), s_x=s_x.to(cuda),
                                s_x_stride=1, s_w=c.s_w.to(cuda), s_y=c.s_y, zp_y=c.zp_y)
    torch.cuda.synchronize()
    rows = np.concatenate([[0, c.M - 1], np.random.default_rng(16).choice(c.M, 10, replace=False)])
    An = c.A.numpy().astype(np.int64)[rows]
    r = O.int8_gemm_y_axis(An, c.a_type, zA.numpy()[rows], c.B.numpy().astype(np.int64), c.b_type, zB.numpy())
    ref = O.int8_epilogue(r["Y"], "s8", c.bias.numpy(), s_x.numpy()[rows].astype(np.float64), c.s_w.numpy(),
                          c.s_y, c.zp_y)
    same(out.cpu().numpy()[rows], ref, "s8")

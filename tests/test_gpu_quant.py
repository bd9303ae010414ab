"""GPU parity of the activation quantiser (qmm_quantize_act_int8): codes and
scales bit-exact against the oracle, per row and per tensor, from fp32 and
bf16, and end to end into the int8 GEMM on the Qwen3-0.6B projection shapes
with fp32 N(0,1) activations quantised per tensor (s_x = amax/127)."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O
from quantized_matmul_qmm_gb300 import inputs as I

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1), (3, 15), (5, 1024), (17, 4607), (64, 4608), (300, 1000), (2, 70000)]


def gpu_quant(qmm, dev, X, per_row, pad=16):
    M, K = X.shape
    lda = (K + 15) // 16 * 16 + pad
    buf = torch.full((M, lda), 77, dtype=torch.int8, device=dev)
    A, s = qmm.quantize_act_int8(X.to(dev), per_row=per_row, A=buf[:, :K])
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert (b[:, K:] == 77).all(), "bytes past K were written"
    return b[:, :K].astype(np.int64), s.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("per_row", [True, False])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,K", SHAPES)
def test_quantize_bit_exact(qmm, cuda, M, K, dtype, per_row):
    g = torch.Generator().manual_seed(M * 7 + K)
    X = (torch.randn((M, K), generator=g) * torch.exp(torch.randn((M, 1), generator=g) * 2)).to(dtype)
    q, s = gpu_quant(qmm, cuda, X, per_row)
    qr, sr = O.quantize_activations_f32(X.float().numpy(), per_row)
    assert np.array_equal(s, sr)
    assert np.array_equal(q, qr)


@pytest.mark.parametrize("per_row", [True, False])
def test_quantize_zero_rows_and_ties(qmm, cuda, per_row):
    X = torch.zeros((4, 40), dtype=torch.float32)
    X[1, :8] = torch.tensor([127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -126.5, 126.5])
    X[3, 5] = -3.0e-3
    q, s = gpu_quant(qmm, cuda, X, per_row)
    qr, sr = O.quantize_activations_f32(X.numpy(), per_row)
    assert np.array_equal(s, sr) and np.array_equal(q, qr)
    if per_row:
        assert s[0] == 0 and not q[0].any()
        assert q[1, :8].tolist() == [127, 2, 4, -2, 0, 2, -126, 126]


@pytest.mark.parametrize("idx", range(7))
def test_projection_chain_per_tensor(qmm, cuda, idx):
    """fp32 N(0,1) activations -> per-tensor int8 on the device -> int8 GEMM
    with the device's s_x and fp32 output, against the oracle chain."""
    name, K, N = I.QWEN3_06B_PROJ[idx]
    M = 32
    g = torch.Generator().manual_seed(1000 + idx)
    X = torch.randn((M, K), generator=g, dtype=torch.float64).to(torch.float32)
    W = (torch.randn((K, N), generator=g, dtype=torch.float64) * 0.02).to(torch.float32)
    Xd = X.to(cuda)
    A, s_x = qmm.quantize_act_int8(Xd, per_row=False)
    packed, s_w, col_sum = qmm.pack_b_int8(W.to(cuda), "f32")
    out = qmm.int8_gemm(A, "s8", 0, packed, col_sum, N, "f32", 0, "f32", s_x=s_x, s_w=s_w)
    torch.cuda.synchronize()
    qa, sa = O.quantize_activations_f32(X.numpy(), per_row=False)
    qw, sw = O.quantize_columns_f32(W.numpy())
    ref = O.int8_gemm(qa, "s8", 0, qw, "s8", 0, "f32", s_x=np.full(M, sa[0]), s_w=sw)
    assert np.array_equal(s_x.cpu().numpy().astype(np.float64), sa)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)


def test_large_chain_per_row_requant(qmm, cuda):
    """Per-row scales into the tensor-core route (M >= 65) with int8 output."""
    M, K, N = 384, 1000, 520
    g = torch.Generator().manual_seed(77)
    X = (torch.randn((M, K), generator=g) * torch.exp(torch.randn((M, 1), generator=g))).to(torch.bfloat16)
    W = (torch.randn((K, N), generator=g) * 0.02).float()
    A, s_x = qmm.quantize_act_int8(X.to(cuda), per_row=True)
    packed, s_w, col_sum = qmm.pack_b_int8(W.to(cuda), "f32")
    ws = torch.empty(max(qmm.int8_gemm_workspace_size(M, K, N), 256), dtype=torch.uint8, device=cuda)
    out = qmm.int8_gemm(A, "s8", 0, packed, col_sum, N, "f32", 0, "s8", s_x=s_x, s_x_stride=1, s_w=s_w,
                        s_y=0.05, zp_y=3, workspace=ws)
    torch.cuda.synchronize()
    qa, sa = O.quantize_activations_f32(X.float().numpy(), per_row=True)
    qw, sw = O.quantize_columns_f32(W.numpy())
    ref = O.int8_gemm(qa, "s8", 0, qw, "s8", 0, "s8", s_x=sa, s_w=sw, s_y=0.05, zp_y=3)
    assert np.array_equal(out.cpu().numpy().astype(np.int64), ref)

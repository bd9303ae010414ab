"""GPU parity of the W8A16 path (int8 weights with one fp32 scale per row and
1,024 weights, bf16 activations): the device pack bit-exact against the
oracle, and the GEMV (M <= 16) and tensor-core GEMM (M > 16) within
max |y - y_ref| <= 2e-4 * sum_k |x| |w| of the oracle's fp64 product, on codes
and scales the oracle packed."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O
from quantized_matmul_qmm_gb300 import inputs as I

pytestmark = pytest.mark.gpu
TOL = 2e-4


def upload_w8(qmm, dev, codes, scales):
    """Oracle codes [N][K] and scales [N][nb] in the library's layout (codes
    [N][Kp] with zero padding, fp32 scales)."""
    N, K = codes.shape
    cb, _ = qmm.pack_w8_size(N, K)
    Kp = cb // N
    c = np.zeros((N, Kp), dtype=np.int8)
    c[:, :K] = codes
    return torch.from_numpy(c).to(dev), torch.from_numpy(scales.astype(np.float32)).to(dev)


def gpu_w8(qmm, dev, codes_d, scales_d, N, K, X, pad=3):
    """X goes to the device with a row stride rounded up to 8 elements (the
    API's 16-byte row rule) unless it already has an admissible stride."""
    M = X.shape[0]
    if X.is_cuda:
        Xd = X
    elif X.stride(0) % 8 != 0:
        Xd = torch.zeros((M, (K + 7) // 8 * 8), dtype=X.dtype, device=dev)[:, :K]
        Xd.copy_(X)
    else:
        Xd = X.to(dev)
    full = torch.full((M + 1, N + pad), float("nan"), dtype=torch.float32, device=dev)
    Y = full[:M, :N]
    qmm.w8_gemm(codes_d, scales_d, N, K, Xd, Y=Y)
    torch.cuda.synchronize()
    f = full.cpu()
    assert torch.isnan(f[:, N:]).all() and torch.isnan(f[M]).all(), "canary overwritten"
    return f[:M, :N].numpy().astype(np.float64)


def check(Y, ref, norm):
    err = np.abs(Y - ref)
    bad = err > TOL * norm
    assert not bad.any(), f"{bad.sum()} outputs off; worst ratio {(err / np.maximum(norm, 1e-300)).max():.3g}"


@pytest.mark.parametrize("N,K", [(1, 1), (3, 63), (5, 1000), (7, 1024), (9, 1025), (33, 3000), (64, 4097)])
def test_pack_w8_bit_exact(qmm, cuda, N, K):
    g = torch.Generator().manual_seed(N * 31 + K)
    W = torch.randn((N, K), generator=g) * torch.exp(torch.randn((N, 1), generator=g))
    if N >= 5:
        W[1] = 0.0                              # every block of a row zero: s = 0, codes 0
        W[2, : min(K, 1024)] = 0.0              # one zero block
        W[3, :8] = torch.tensor([127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -126.5, 126.5])[: min(8, K)]
    codes, scales = qmm.pack_w8(W.to(cuda))
    torch.cuda.synchronize()
    qr, sr = O.pack_w8(W.numpy())
    c = codes.cpu().numpy().astype(np.int64)
    assert c.shape[1] == (K + 63) // 64 * 64
    assert np.array_equal(c[:, :K], qr)
    assert not c[:, K:].any(), "padding codes must be zero"
    assert np.array_equal(scales.cpu().numpy().astype(np.float64), sr)


@pytest.mark.parametrize("N,K", [(64, 64), (300, 1000), (520, 1025), (257, 3000), (1024, 1024)])
@pytest.mark.parametrize("M", [1, 2, 5, 16, 17, 64, 255, 256, 300, 577])
def test_w8_gemm_small_shapes(qmm, cuda, N, K, M):
    g = torch.Generator().manual_seed(N + 7 * K + 131 * M)
    W = torch.randn((N, K), generator=g) * 0.02
    X = torch.randn((M, K), generator=g).to(torch.bfloat16)
    codes, scales = O.pack_w8(W.numpy())
    cd, sd = upload_w8(qmm, cuda, codes, scales)
    Y = gpu_w8(qmm, cuda, cd, sd, N, K, X)
    ref, norm = O.w8_gemm(codes, scales, X.float().double().numpy())
    check(Y, ref, norm)


@pytest.mark.parametrize("M", [3, 40])
def test_w8_gemm_zero_block_and_strided_x(qmm, cuda, M):
    """A weight block of zeros (scale 0) contributes nothing; X with a row
    stride above K; K straddling a block edge by 8."""
    N, K = 96, 2056
    g = torch.Generator().manual_seed(5 + M)
    W = torch.randn((N, K), generator=g) * 0.05
    W[:, 1024:2048] = 0.0
    Xfull = torch.randn((M, K + 24), generator=g).to(torch.bfloat16)
    X = Xfull[:, :K]
    codes, scales = O.pack_w8(W.numpy())
    assert (scales[:, 1] == 0).all()
    cd, sd = upload_w8(qmm, cuda, codes, scales)
    Xd = Xfull.to(cuda)[:, :K]
    assert Xd.stride(0) == K + 24
    Y = gpu_w8(qmm, cuda, cd, sd, N, K, Xd)
    ref, norm = O.w8_gemm(codes, scales, X.float().double().numpy())
    check(Y, ref, norm)


@pytest.mark.parametrize("idx", range(7))
@pytest.mark.parametrize("M", [1, 512])
def test_w8_qwen_projections(qmm, cuda, idx, M):
    """The Qwen3-0.6B projection shapes, decode and a 512-token prefill."""
    name, K, N = I.QWEN3_06B_PROJ[idx]
    c = I.q4_case(name, K, N, M)
    codes, scales = O.pack_w8(c.W.numpy())
    cd, sd = upload_w8(qmm, cuda, codes, scales)
    Y = gpu_w8(qmm, cuda, cd, sd, N, K, c.X)
    ref, norm = O.w8_gemm(codes, scales, c.X.float().double().numpy())
    check(Y, ref, norm)


def test_w8_lm_head_decode_full_size(qmm, cuda):
    """The Qwen3-0.6B lm_head (N = 151936, K = 1024) at M = 1, every output."""
    name, K, N = I.QWEN3_06B_LM_HEAD
    c = I.q4_case(name, K, N, 1)
    codes, scales = O.pack_w8(c.W.numpy())
    cd, sd = upload_w8(qmm, cuda, codes, scales)
    Y = gpu_w8(qmm, cuda, cd, sd, N, K, c.X)
    ref, norm = O.w8_gemm(codes, scales, c.X.float().double().numpy())
    check(Y, ref, norm)


@pytest.mark.parametrize("K,items_per_sm,extra", [(128, 2, 0), (1000, 3, 17), (1100, 2, 5), (1536, 3, 0),
                                                 (2048, 4, 31)])
def test_w8_gemv_streaming_ring(qmm, cuda, K, items_per_sm, extra):
    """M = 1 over many rows: the streaming ring kernel.  K = 128 (one k-block,
    the second half-warp idle, 12 slots), 1000 and 1536 (one scale block),
    1100 (nine k-blocks split 5 + 4, the second half crossing into the second
    scale block) and 2048 (two scale blocks, 3 slots); N past a multiple of 32
    leaves the last item partly outside the matrix; every slot is refilled."""
    sms = torch.cuda.get_device_properties(cuda).multi_processor_count
    N = 32 * sms * items_per_sm + extra
    g = torch.Generator().manual_seed(K + extra)
    W = torch.randn((N, K), generator=g) * 0.02
    W[7] = 0.0
    X = torch.randn((1, K), generator=g).to(torch.bfloat16)
    codes, scales = O.pack_w8(W.numpy())
    cd, sd = upload_w8(qmm, cuda, codes, scales)
    Y = gpu_w8(qmm, cuda, cd, sd, N, K, X)
    ref, norm = O.w8_gemm(codes, scales, X.float().double().numpy())
    check(Y, ref, norm)
    assert (Y[0, 7] == 0.0)


def test_w8_large_gemm_sampled_rows(qmm, cuda):
    """M = 4096, K = N = 4608 on the tensor-core route, checked on 48 sampled
    rows (rows are independent, so the oracle runs on those rows alone)."""
    M, K, N = 4096, 4608, 4608
    g = torch.Generator().manual_seed(4608)
    W = torch.randn((N, K), generator=g) * 0.02
    X = torch.randn((M, K), generator=g).to(torch.bfloat16)
    codes, scales = O.pack_w8(W.numpy())
    cd, sd = upload_w8(qmm, cuda, codes, scales)
    Y = gpu_w8(qmm, cuda, cd, sd, N, K, X)
    rows = np.sort(np.random.default_rng(1).choice(M, 48, replace=False))
    rows[0], rows[-1] = 0, M - 1
    ref, norm = O.w8_gemm(codes, scales, X[torch.from_numpy(rows)].float().double().numpy())
    check(Y[rows], ref, norm)

"""GPU parity of the extra weight formats ("NPU engine: full ELFs, no xclbin",
section "Q4NX chunks"):

* Q4_K -> q4_1 repack: device bytes equal the oracle's repack, and the 4-bit
  kernels run the repacked tiles;
* Q8 tiles in both code layouts: the device pack is byte-exact against the
  oracle; the decode GEMV (M <= 16) is within 2e-5 * sum_k |x||w| of the
  oracle's fp64 product and the tensor-core route (M > 16, weights rounded once
  to bf16) within 2e-3 * sum_k |x||w|, on tiles the oracle packed."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O
from quantized_matmul_qmm_gb300 import inputs as I

pytestmark = pytest.mark.gpu
TOL_GEMV = 2e-5
TOL_TC = 2e-3


def check(Y, ref, norm, tol):
    err = np.abs(Y - ref)
    bad = err > tol * norm
    assert not bad.any(), f"{bad.sum()} outputs off; worst ratio {(err / np.maximum(norm, 1e-300)).max():.3g}"


def run_q8(qmm, dev, tiles_d, layout, N, K, X, pad=5):
    M = X.shape[0]
    full = torch.full((M + 1, N + pad), float("nan"), dtype=torch.float32, device=dev)
    Y = full[:M, :N]
    qmm.q8_gemm(tiles_d, layout, N, K, X.to(dev), Y=Y)
    torch.cuda.synchronize()
    f = full.cpu()
    assert torch.isnan(f[:, N:]).all() and torch.isnan(f[M]).all(), "canary overwritten"
    return f[:M, :N].numpy().astype(np.float64)


# --------------------------------------------------------------------------
# Q4_K repack
# --------------------------------------------------------------------------

def special_q4k(N, K, seed):
    """Random super-blocks plus rows with negative, zero and subnormal fp16 d/dmin."""
    buf = I.q4k_superblocks(seed, N, K).clone()
    v = buf.view(N, K // 256, 144)
    vals = torch.tensor([-1.5e-3, 0.0, 6.0e-8, 3.0e-5], dtype=torch.float16).view(torch.uint8).reshape(4, 2)
    for i in range(min(4, N)):
        v[i, 0, 0:2] = vals[i]
        v[i, -1, 2:4] = vals[(i + 1) % 4]
    return buf


@pytest.mark.parametrize("N,K,extra", [(32, 256, 0), (64, 1024, 0), (96, 512, 48), (160, 2048, 16)])
def test_repack_q4k_bit_exact(qmm, cuda, N, K, extra):
    buf = special_q4k(N, K, N + K)
    row = K // 256 * 144
    src = torch.full((N, row + extra), 0xAB, dtype=torch.uint8)
    src[:, :row] = buf
    tiles = qmm.repack_q4k(src.to(cuda), N, K)
    torch.cuda.synchronize()
    ref = O.repack_q4k(src.numpy(), N, K, row + extra)
    got = tiles.cpu().numpy()
    assert np.array_equal(got, ref), f"{(got != ref).sum()} bytes differ"


@pytest.mark.parametrize("M", [1, 3, 16, 17, 300])
def test_q4_gemm_runs_repacked_q4k(qmm, cuda, M):
    N, K = 256, 1024
    buf = I.q4k_superblocks(31, N, K)
    tiles = qmm.repack_q4k(buf.to(cuda), N, K)
    X = I.q4_activations(32 + M, M, K)
    Y = qmm.q4_gemm(tiles, N, K, X.to(cuda))
    torch.cuda.synchronize()
    ref, norm = O.q4_gemm(O.repack_q4k(buf.numpy(), N, K), N, K, X.float().numpy().astype(np.float64))
    check(Y.cpu().numpy().astype(np.float64), ref, norm, TOL_GEMV if M <= 16 else TOL_TC)


def test_repack_q4k_lm_head_sampled(qmm, cuda):
    """Full lm_head size (K=1024, N=151936): sampled tile rows byte-exact, and
    the M=1 GEMV on the repacked tiles against the oracle on those rows."""
    N, K = 151936, 1024
    buf = I.q4k_superblocks(33, N, K)
    tiles = qmm.repack_q4k(buf.to(cuda), N, K)
    X = I.q4_activations(34, 1, K)
    Y = qmm.q4_gemm(tiles, N, K, X.to(cuda))
    torch.cuda.synchronize()
    t = tiles.cpu().numpy().reshape(N // 32, -1)
    rng = np.random.default_rng(35)
    trs = np.concatenate([[0, N // 32 - 1], rng.choice(N // 32, 14, replace=False)])
    for tr in trs:
        sub = buf[32 * tr:32 * tr + 32].numpy()
        assert np.array_equal(t[tr], O.repack_q4k(sub, 32, K))
        ref, norm = O.q4_gemm(t[tr], 32, K, X.float().numpy().astype(np.float64))
        check(Y[:, 32 * tr:32 * tr + 32].cpu().numpy().astype(np.float64), ref, norm, TOL_GEMV)


# --------------------------------------------------------------------------
# Q8 tiles
# --------------------------------------------------------------------------

@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("N,K", [(32, 256), (64, 512), (96, 1024), (32, 2304)])
def test_pack_q8_bit_exact(qmm, cuda, layout, N, K):
    g = torch.Generator().manual_seed(N * 7 + K + layout)
    W = torch.randn((N, K), generator=g) * torch.exp(torch.randn((N, 1), generator=g))
    W[1, 32:64] = 0.0                                  # a zero block: scale 0, codes 0
    W[2, :32] = torch.arange(-16, 16, dtype=torch.float32) * 0.5 + 0.25
    W[3, :8] = torch.tensor([127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -126.5, 126.5])   # s = 1: half-even ties
    W[3, 8:32] = 0.0
    Wp = torch.zeros((N, K + 3))
    Wp[:, :K] = W
    tiles = qmm.pack_q8(Wp.to(cuda)[:, :K], layout)
    torch.cuda.synchronize()
    ref = O.pack_q8(W.numpy(), layout)
    got = tiles.cpu().numpy()
    assert np.array_equal(got, ref), f"{(got != ref).sum()} bytes differ"


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("N,K", [(32, 256), (64, 768), (1024, 1024), (2048, 3072), (3072, 1024)])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16, 17, 64, 256, 300])
def test_q8_gemm(qmm, cuda, layout, N, K, M):
    W = I.q4_weights(41 + N + K, N, K).numpy()
    X = I.q4_activations(42 + M + K, M, K)
    t = O.pack_q8(W, layout)
    Y = run_q8(qmm, cuda, torch.from_numpy(t).to(cuda), layout, N, K, X)
    ref, norm = O.q8_gemm(t, N, K, X.float().numpy().astype(np.float64), layout)
    check(Y, ref, norm, TOL_GEMV if M <= 16 else TOL_TC)


def test_q8_gemm_strided_x_and_y(qmm, cuda):
    N, K, M = 64, 512, 6
    W = I.q4_weights(50, N, K).numpy()
    Xf = I.q4_activations(51, M, K + 24)
    X = Xf.to(cuda)[:, 8:K + 8]                  # row stride K + 24, offset 16 bytes
    t = O.pack_q8(W, 1)
    Yfull = torch.zeros((M, N + 40), dtype=torch.float32, device=cuda)
    qmm.q8_gemm(torch.from_numpy(t).to(cuda), 1, N, K, X, Y=Yfull[:, 20:20 + N])
    torch.cuda.synchronize()
    ref, norm = O.q8_gemm(t, N, K, Xf[:, 8:K + 8].float().numpy().astype(np.float64), 1)
    check(Yfull[:, 20:20 + N].cpu().numpy().astype(np.float64), ref, norm, TOL_GEMV)
    assert not Yfull[:, :20].any() and not Yfull[:, 20 + N:].any()


def test_q8_integer_weights_exact(qmm, cuda):
    """Blocks with amax 127 have scale 1, so integer activations give exact integer sums."""
    rng = np.random.default_rng(52)
    N, K = 64, 1024
    W = rng.integers(-127, 128, (N, K)).astype(np.float32)
    W[:, ::32] = 127.0
    X = torch.from_numpy(rng.integers(-8, 9, (4, K)).astype(np.float32)).to(torch.bfloat16)
    for layout in (0, 1):
        t = qmm.pack_q8(torch.from_numpy(W).to(cuda), layout)
        Y = run_q8(qmm, cuda, t, layout, N, K, X)
        ref = X.float().numpy().astype(np.int64) @ W.astype(np.int64).T
        assert np.array_equal(Y, ref.astype(np.float64))


@pytest.mark.parametrize("layout", [0, 1])
def test_q8_lm_head_sampled_and_deterministic(qmm, cuda, layout):
    """Full lm_head size (K=1024, N=151936) packed on the device: sampled tile
    rows byte-exact and their outputs within the GEMV bound; two runs equal."""
    N, K = 151936, 1024
    W = I.q4_weights(60, N, K)
    tiles = qmm.pack_q8(W.to(cuda), layout)
    X = I.q4_activations(61, 1, K).to(cuda)
    Y1 = qmm.q8_gemm(tiles, layout, N, K, X)
    Y2 = qmm.q8_gemm(tiles, layout, N, K, X)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
    t = tiles.cpu().numpy().reshape(N // 32, -1)
    rng = np.random.default_rng(62)
    xs = X.float().cpu().numpy().astype(np.float64)
    for tr in np.concatenate([[0, N // 32 - 1], rng.choice(N // 32, 14, replace=False)]):
        sub = W[32 * tr:32 * tr + 32].numpy()
        assert np.array_equal(t[tr], O.pack_q8(sub, layout))
        ref, norm = O.q8_gemm(t[tr], 32, K, xs, layout)
        check(Y1[:, 32 * tr:32 * tr + 32].cpu().numpy().astype(np.float64), ref, norm, TOL_GEMV)

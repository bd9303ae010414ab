"""GPU parity of the 4-bit dense path: tile packing byte-exact against the
oracle, GEMV/GEMM within max |y - y_ref| <= 2e-3 * sum|x||w| (the oracle is the
fp64 decode-then-dense "twin")."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O
from quantized_matmul_qmm_gb300 import inputs as I

pytestmark = pytest.mark.gpu
TOL = 2e-3


def gpu_q4(qmm, dev, W, X, pad=3):
    N, K = W.shape
    M = X.shape[0]
    tiles = qmm.pack_q4(W.to(dev))
    full = torch.full((M + 1, N + pad), float("nan"), dtype=torch.float32, device=dev)
    Y = full[:M, :N]
    qmm.q4_gemm(tiles, N, K, X.to(dev), Y=Y)
    torch.cuda.synchronize()
    f = full.cpu()
    assert torch.isnan(f[:, N:]).all() and torch.isnan(f[M]).all(), "canary overwritten"
    return tiles.cpu().numpy(), f[:M, :N].numpy()


def xnp(X):
    return X.float().double().numpy()


@pytest.mark.parametrize("N,K", [(32, 256), (64, 512), (96, 768), (1024, 1024), (1024, 3072)])
@pytest.mark.parametrize("M", [1, 2, 7, 8, 9, 16, 17, 33, 100, 300, 577])
def test_q4_gemm_small_shapes(qmm, cuda, N, K, M):
    g = torch.Generator().manual_seed(N + K + M)
    W = torch.randn((N, K), generator=g) * 0.02
    X = torch.randn((M, K), generator=g).to(torch.bfloat16)
    tiles, Y = gpu_q4(qmm, cuda, W, X)
    ref_tiles = O.pack_q4(W.numpy())
    assert np.array_equal(tiles, ref_tiles)
    y, norm = O.q4_gemm(ref_tiles, N, K, xnp(X))
    err = O.normalized_error(Y, y, norm)
    assert err <= TOL, err
    if M <= 16:  # decode kernel: weights never rounded, only fp32 accumulation error
        assert err <= 2e-5, f"error {err} far above the fp32 accumulation level"


def test_q4_special_weights(qmm, cuda):
    # constant blocks (scale 0), a zero row, one-hot activations
    N, K = 64, 512
    g = torch.Generator().manual_seed(3)
    W = torch.randn((N, K), generator=g) * 0.02
    W[5, 32:64] = 0.125
    W[7] = 0.0
    X = torch.zeros((3, K)).to(torch.bfloat16)
    X[0, 0] = 1
    X[1, 300] = 1
    X[2] = torch.randn(K, generator=g).to(torch.bfloat16)
    tiles, Y = gpu_q4(qmm, cuda, W, X)
    ref_tiles = O.pack_q4(W.numpy())
    assert np.array_equal(tiles, ref_tiles)
    y, norm = O.q4_gemm(ref_tiles, N, K, xnp(X))
    assert O.normalized_error(Y, y, norm) <= TOL
    dense = O.q4_decode(ref_tiles, N, K)
    assert np.allclose(Y[0], dense[:, 0], rtol=1e-6, atol=1e-7)
    assert np.allclose(Y[1], dense[:, 300], rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("M", [1, 512])
@pytest.mark.parametrize("idx", range(7))
def test_workload_qwen_projection(qmm, cuda, idx, M):
    name, K, N = I.QWEN3_06B_PROJ[idx]
    c = I.q4_case(name, K, N, M)
    tiles, Y = gpu_q4(qmm, cuda, c.W, c.X)
    ref_tiles = O.pack_q4(c.W.numpy())
    assert np.array_equal(tiles, ref_tiles)
    y, norm = O.q4_gemm(ref_tiles, N, K, xnp(c.X))
    err = O.normalized_error(Y, y, norm)
    assert err <= TOL, err


@pytest.mark.parametrize("M", [1, 16, 512])
def test_workload_lm_head_sampled(qmm, cuda, M):
    name, K, N = I.QWEN3_06B_LM_HEAD
    c = I.q4_case(name, K, N, M)
    tiles, Y = gpu_q4(qmm, cuda, c.W, c.X, pad=0)
    rng = np.random.default_rng(M)
    trs = np.unique(np.concatenate([[0, 1, N // 32 - 1], rng.choice(N // 32, 40, replace=False)]))
    per = (K // 256) * 5120
    rows = np.concatenate([np.arange(32 * tr, 32 * tr + 32) for tr in trs])
    Wn = c.W.numpy()
    for tr in trs:   # packing of the sampled tile rows, byte for byte
        assert np.array_equal(tiles[tr * per:(tr + 1) * per], O.pack_q4(Wn[32 * tr:32 * tr + 32]))
    y, norm = O.q4_gemm_rows(tiles, N, K, xnp(c.X), rows)
    err = O.normalized_error(Y[:, rows], y, norm)
    assert err <= TOL, err


@pytest.mark.parametrize("M", [1, 5, 16])
def test_q4_gemv_streaming_path_full(qmm, cuda, M):
    # N large enough that every SM streams several tile rows
    N, K = 10240, 512
    g = torch.Generator().manual_seed(77 + M)
    W = torch.randn((N, K), generator=g) * 0.02
    X = torch.randn((M, K), generator=g).to(torch.bfloat16)
    tiles, Y = gpu_q4(qmm, cuda, W, X)
    ref_tiles = O.pack_q4(W.numpy())
    assert np.array_equal(tiles, ref_tiles)
    y, norm = O.q4_gemm(ref_tiles, N, K, xnp(X))
    err = O.normalized_error(Y, y, norm)
    assert err <= 2e-5, err


@pytest.mark.parametrize("K,rows_per_sm", [(1024, 12), (2048, 7), (2560, 5)])
def test_q4_gemv_ring_slot_reuse(qmm, cuda, K, rows_per_sm):
    """M=1 streaming GEMV with more tile rows per CTA than ring slots, so every
    slot is refilled: K=1024 (8 slots, 4 consumer pairs), K=2048 (4 slots),
    K=2560 (3 slots, 3 pairs).  Sampled tile rows include every row of the
    first CTA's sequence and the last rows of the launch."""
    sms = torch.cuda.get_device_properties(cuda).multi_processor_count
    N = 32 * sms * rows_per_sm
    g = torch.Generator().manual_seed(K + rows_per_sm)
    W = torch.randn((N, K), generator=g) * 0.02
    X = torch.randn((1, K), generator=g).to(torch.bfloat16)
    tiles, Y = gpu_q4(qmm, cuda, W, X, pad=0)
    rng = np.random.default_rng(K)
    ntr = N // 32
    trs = np.unique(np.concatenate([np.arange(0, ntr, sms), np.arange(ntr - 8, ntr),
                                    rng.choice(ntr, 24, replace=False)]))
    per = (K // 256) * 5120
    rows = np.concatenate([np.arange(32 * tr, 32 * tr + 32) for tr in trs])
    Wn = W.numpy()
    for tr in trs:   # packing of the sampled tile rows, byte for byte
        assert np.array_equal(tiles[tr * per:(tr + 1) * per], O.pack_q4(Wn[32 * tr:32 * tr + 32]))
    y, norm = O.q4_gemm_rows(tiles, N, K, xnp(X), rows)
    err = O.normalized_error(Y[:, rows], y, norm)
    assert err <= 2e-5, err


@pytest.mark.parametrize("M,K,rows_per_sm", [(2, 1024, 9), (5, 1280, 3), (8, 2048, 5), (9, 1792, 6),
                                           (16, 1024, 11), (16, 2048, 4)])
def test_q4_gemv_small_batch_ring(qmm, cuda, M, K, rows_per_sm):
    """2 <= M <= 16 over many tile rows: the streaming ring kernel, with every
    slot refilled.  The shapes cover one TMA box per tile row (K=1024, 1280),
    two (K=2048 at four tiles a box) and one box per tile (K=1792, seven tiles),
    one and two 8-token MMA column groups, and 3 to 8 ring slots."""
    sms = torch.cuda.get_device_properties(cuda).multi_processor_count
    N = 32 * sms * rows_per_sm
    g = torch.Generator().manual_seed(M * 1000 + K + rows_per_sm)
    W = torch.randn((N, K), generator=g) * 0.02
    X = torch.randn((M, K), generator=g).to(torch.bfloat16)
    tiles, Y = gpu_q4(qmm, cuda, W, X, pad=0)
    assert np.isfinite(Y).all()
    rng = np.random.default_rng(M + K)
    ntr = N // 32
    trs = np.unique(np.concatenate([np.arange(0, ntr, sms), np.arange(ntr - 8, ntr),
                                    rng.choice(ntr, 24, replace=False)]))
    per = (K // 256) * 5120
    rows = np.concatenate([np.arange(32 * tr, 32 * tr + 32) for tr in trs])
    Wn = W.numpy()
    for tr in trs:   # packing of the sampled tile rows, byte for byte
        assert np.array_equal(tiles[tr * per:(tr + 1) * per], O.pack_q4(Wn[32 * tr:32 * tr + 32]))
    y, norm = O.q4_gemm_rows(tiles, N, K, xnp(X), rows)
    err = O.normalized_error(Y[:, rows], y, norm)
    assert err <= 2e-5, err


@pytest.mark.parametrize("M,N,K", [(577, 8192, 256), (300, 12288, 256)])
def test_q4_prefill_192_token_chunks(qmm, cuda, M, N, K):
    """Prefill GEMMs large enough in N to take 192-token jobs (the MMA's N),
    with a ragged last chunk: 577 = 3 x 192 + 1, 300 = 192 + 108."""
    g = torch.Generator().manual_seed(M + N)
    W = torch.randn((N, K), generator=g) * 0.02
    X = torch.randn((M, K), generator=g).to(torch.bfloat16)
    tiles, Y = gpu_q4(qmm, cuda, W, X)
    ref_tiles = O.pack_q4(W.numpy())
    assert np.array_equal(tiles, ref_tiles)
    y, norm = O.q4_gemm(ref_tiles, N, K, xnp(X))
    err = O.normalized_error(Y, y, norm)
    assert err <= TOL, err


def test_bounded_wait_times_out_and_context_survives(qmm, cuda):
    """The device error path of the pipelined kernels: a bounded wait on a
    barrier nothing arrives on gives up after its limit, QMM_ERR_TIMEOUT
    reaches dev_status, the block's other wait leaves on the abort flag, the
    kernel frees its tensor memory and returns; the tensor-core kernels
    (which allocate tensor memory) then still run correctly."""
    limit = 5_000_000   # 5 ms
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    out = torch.full((4,), -1, dtype=torch.int64, device=cuda)
    qmm.selftest_wait_timeout(limit, status, out)
    torch.cuda.synchronize()
    r = out.cpu().tolist()
    assert int(status.item()) == qmm.QMM_ERR_TIMEOUT
    assert r[0] == 0 and r[1] == 0, r
    assert limit <= r[2] < limit + 50_000_000, r
    assert -1_000_000 < r[3] < 20_000_000, r   # the second wait leaves within a suspend interval
    # the context is usable: a tensor-core prefill GEMM and a second self-test
    N, K, M = 256, 512, 64
    g = torch.Generator().manual_seed(99)
    W = torch.randn((N, K), generator=g) * 0.02
    X = torch.randn((M, K), generator=g).to(torch.bfloat16)
    status.zero_()
    tiles, Y = gpu_q4(qmm, cuda, W, X)
    y, norm = O.q4_gemm(O.pack_q4(W.numpy()), N, K, xnp(X))
    assert O.normalized_error(Y, y, norm) <= TOL
    qmm.selftest_wait_timeout(limit, status, out)
    torch.cuda.synchronize()
    assert int(status.item()) == qmm.QMM_ERR_TIMEOUT

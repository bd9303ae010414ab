"""GPU parity of the tensor-core routes that round a weight: the 4-bit prefill
GEMM (M >= 17), MUL_MAT_ID, and the Q8 GEMM above the decode sizes.

They form every weight once in f16 and convert every activation row to f16
after a power-of-two scale, so for weight blocks in f16's normal range the
worst case over all inputs is |y - y_exact| <= (2^-11 + K 2^-23) sum_k |x||w|.
These cases are built so that a coarser weight rounding fails the 2e-3 gate:

* every 32-weight block takes two values, 1.0 and 1.0039 (codes 0 and 15),
  and the activations are positive only where the weight is 1.0039, so every
  weight's rounding error in a row has the same sign (the tests first check
  on the CPU that one bf16 rounding per weight would miss the gate);
* Q8 blocks whose codes were picked so that code * scale lies just below a
  bf16 rounding midpoint;
* activation rows spanning bf16's exponent range (2^100, 2^-100, mixed
  magnitudes, zeros), which the row scale must carry exactly;
* weight blocks beyond f16's range, which must be reported as QMM_ERR_RANGE
  on the tensor-core routes while the decode GEMV stays exact.

Every result is compared element by element with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O

pytestmark = pytest.mark.gpu
TOL = 2e-3


def bound(K):
    """The tensor-core route's worst case for weights in f16's normal range."""
    return 2.0 ** -11 + K * 2.0 ** -23


def bf16_weight_error(tiles, N, K, X, decode=O.q4_decode):
    """Normalised error of a product whose weights are each rounded once to
    bf16 (the rounding this route no longer takes), against the oracle."""
    W = decode(tiles, N, K)
    y = X @ W.T
    yb = X @ O.bf16_rne(W).T
    return O.normalized_error(yb, y, np.abs(X) @ np.abs(W).T)


def two_valued(seed, N, K, lo=1.0, hi=1.0039):
    """Weights [N][K] whose every block holds lo and hi on one column pattern
    shared by all rows (each row scaled by its own power of two), and the
    pattern."""
    rng = np.random.default_rng(seed)
    pat = rng.random(K) < 0.5
    pat[0::32], pat[1::32] = False, True
    W = np.where(pat, hi, lo)[None, :] * (2.0 ** rng.integers(-8, 9, N))[:, None]
    return W.astype(np.float32), pat


def pattern_acts(seed, M, pat):
    """Activations positive on the pattern's columns, zero elsewhere; row 0 is
    exactly the pattern."""
    rng = np.random.default_rng(seed)
    a = rng.uniform(0.5, 2.0, (M, pat.size)) * pat[None, :]
    a[0] = pat
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)


def xnp(X):
    return X.float().double().numpy()


def run_q4(qmm, dev, tiles_np, N, K, X, status=None):
    M = X.shape[0]
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    qmm.q4_gemm(torch.from_numpy(tiles_np).to(dev), N, K, X.to(dev), Y=Y, dev_status=status)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


@pytest.mark.parametrize("M", [17, 512])
def test_q4_gemm_same_sign_rounding(qmm, cuda, M):
    N, K = 256, 1024
    W, pat = two_valued(M, N, K)
    X = pattern_acts(M + 1, M, pat)
    tiles = O.pack_q4(W)
    assert bf16_weight_error(tiles, N, K, xnp(X)) > 3.5e-3   # the case has teeth
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    Y = run_q4(qmm, cuda, tiles, N, K, X, status)
    assert int(status.item()) == 0
    y, norm = O.q4_gemm(tiles, N, K, xnp(X))
    err = O.normalized_error(Y, y, norm)
    assert err <= bound(K) and err <= TOL, err


def test_q4_gemm_same_sign_rounding_long_k(qmm, cuda):
    # K = 4096 spans 16 tile columns and the accumulation term of the bound
    N, K, M = 128, 4096, 40
    W, pat = two_valued(5, N, K)
    X = pattern_acts(6, M, pat)
    tiles = O.pack_q4(W)
    Y = run_q4(qmm, cuda, tiles, N, K, X)
    y, norm = O.q4_gemm(tiles, N, K, xnp(X))
    assert O.normalized_error(Y, y, norm) <= bound(K)


@pytest.mark.parametrize("shared", [True, False])
@pytest.mark.parametrize("packed", [True, False])
def test_moe_same_sign_rounding(qmm, cuda, shared, packed):
    E, N, K, T, n_used, ld = 8, 128, 512, 37, 3, 5
    rng = np.random.default_rng(11 + shared + 2 * packed)
    W, pat = two_valued(12, E * N, K)
    tiles = O.pack_q4(W)   # expert e is rows e*N .. e*N+N-1: consecutive tile sets
    ids = torch.from_numpy(rng.integers(0, E, (T, ld)).astype(np.int32))
    X = pattern_acts(13, T if shared else T * n_used, pat)
    if not shared:
        X = X.reshape(T, n_used, K)
    ws_full = qmm.q4_gemm_id_workspace_size(E, n_used, T, K)
    ws_bytes = ws_full if packed else ws_full - T * n_used * K * 2   # tables only: the gather mode
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    Y = qmm.q4_gemm_id(torch.from_numpy(tiles).to(cuda), E, N, K, X.to(cuda), ids.to(cuda), ld, n_used, T,
                       workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y, norm = O.q4_gemm_id(tiles, E, N, K, xnp(X), shared, ids.numpy(), ld, n_used, T)
    err = O.normalized_error(Y.cpu().numpy(), y, norm)
    assert err <= bound(K), err


def q8_adversarial(seed, N, K):
    """Q8 codes and bf16 scales whose products code * scale lie just below a
    bf16 rounding midpoint (so one bf16 rounding per weight errs downwards by
    close to half a unit), with the activation pattern of those columns."""
    rng = np.random.default_rng(seed)
    s = float(O.bf16_rne(np.float64(1.66 / 127)))   # 16 codes in 1..127 land just below a midpoint
    q = np.arange(-127, 128)
    w = q * s
    rel = (w - O.bf16_rne(w)) / np.where(w == 0, 1, np.abs(w))
    good = q[(rel > 3.0e-3) & (q > 0)]
    assert good.size >= 4
    codes = rng.choice(good, (N, K))
    codes[:, 0::32] = 127   # each block's largest code
    scales = np.full((N, K // 32), s) * (2.0 ** rng.integers(-6, 7, N))[:, None]
    pat = np.ones(K, dtype=bool)
    pat[0::32] = False
    return codes, O.bf16_rne(scales), pat


@pytest.mark.parametrize("layout", [0, 1])
def test_q8_gemm_same_sign_rounding(qmm, cuda, layout):
    N, K, M = 256, 1024, 300
    codes, scales, pat = q8_adversarial(20 + layout, N, K)
    tiles = O.q8_tiles_from_blocks(codes, scales, layout)
    X = pattern_acts(22, M, pat)
    dec = lambda t, n, k: O.q8_decode(t, n, k, layout)   # noqa: E731
    assert bf16_weight_error(tiles, N, K, xnp(X), dec) > 2.5e-3
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device=cuda)
    qmm.q8_gemm(torch.from_numpy(tiles).to(cuda), layout, N, K, X.to(cuda), Y=Y, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y, norm = O.q8_gemm(tiles, N, K, xnp(X), layout)
    err = O.normalized_error(Y.cpu().numpy(), y, norm)
    assert err <= 2.0 ** -11 + 1024 * 2.0 ** -23 + (K / 1024) * 2.0 ** -24, err


def wide_range_acts(seed, M, K):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn((M, K), generator=g, dtype=torch.float64)
    X[0] *= 2.0 ** 100
    X[1] *= 2.0 ** -100
    X[2] = 0.0
    X[3] *= 2.0 ** torch.randint(-20, 21, (K,), generator=g).double()
    X[4, 7] = 3.0e4   # one large element among N(0, 1) values
    X[5] *= 1.0e-38   # bf16 subnormals
    return X.float().to(torch.bfloat16)


def test_q4_gemm_activation_range(qmm, cuda):
    N, K, M = 256, 1024, 40
    g = torch.Generator().manual_seed(30)
    W = (torch.randn((N, K), generator=g) * 0.02).numpy()
    tiles = O.pack_q4(W)
    X = wide_range_acts(31, M, K)
    assert torch.isfinite(X.float()).all()
    Y = run_q4(qmm, cuda, tiles, N, K, X)
    y, norm = O.q4_gemm(tiles, N, K, xnp(X))
    assert not np.any(Y[2]), "a zero activation row gives zeros"
    err = O.normalized_error(Y, y, norm)
    assert err <= bound(K), err


def test_moe_activation_range(qmm, cuda):
    E, N, K, T, n_used, ld = 4, 64, 512, 9, 2, 2
    rng = np.random.default_rng(32)
    W = (rng.standard_normal((E * N, K)) * 0.02).astype(np.float32)
    tiles = O.pack_q4(W)
    ids = torch.from_numpy(rng.integers(0, E, (T, ld)).astype(np.int32))
    X = wide_range_acts(33, T, K)
    Y = qmm.q4_gemm_id(torch.from_numpy(tiles).to(cuda), E, N, K, X.to(cuda), ids.to(cuda), ld, n_used, T)
    torch.cuda.synchronize()
    y, norm = O.q4_gemm_id(tiles, E, N, K, xnp(X), True, ids.numpy(), ld, n_used, T)
    assert O.normalized_error(Y.cpu().numpy(), y, norm) <= bound(K)


def test_weight_range_reported(qmm, cuda):
    """A q4 block with min 7e4 (beyond f16's 65504): the tensor-core routes
    report QMM_ERR_RANGE; the decode GEMV forms the weights in fp32 and is
    exact to its own bound."""
    N, K = 64, 512
    g = torch.Generator().manual_seed(40)
    W = (torch.randn((N, K), generator=g) * 0.02).numpy()
    W[9, 64:96] = 7.0e4 + np.arange(32)
    tiles = O.pack_q4(W)
    X = torch.randn((17, K), generator=g).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    run_q4(qmm, cuda, tiles, N, K, X, status)
    assert int(status.item()) == qmm.QMM_ERR_RANGE
    status.zero_()
    Y1 = run_q4(qmm, cuda, tiles, N, K, X[:1], status)
    assert int(status.item()) == 0
    y, norm = O.q4_gemm(tiles, N, K, xnp(X[:1]))
    assert O.normalized_error(Y1, y, norm) <= 2e-5
    # MUL_MAT_ID on the same weights as one expert
    status.zero_()
    ids = torch.zeros((17, 1), dtype=torch.int32, device=cuda)
    qmm.q4_gemm_id(torch.from_numpy(tiles).to(cuda), 1, N, K, X.to(cuda), ids, 1, 1, 17, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == qmm.QMM_ERR_RANGE
    # Q8: a block whose scale times 128 passes 65504
    Wq = (torch.randn((N, K), generator=g) * 0.02).numpy()
    Wq[3, 32:64] = 1.0e6
    tq = qmm.pack_q8(torch.from_numpy(Wq).to(cuda), 0)
    status.zero_()
    qmm.q8_gemm(tq, 0, N, K, X.to(cuda), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == qmm.QMM_ERR_RANGE

"""GPU parity of MUL_MAT_ID: strided ids, shared and per-slot src1, bad ids."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O
from quantized_matmul_qmm_gb300 import inputs as I

pytestmark = pytest.mark.gpu
TOL = 2e-3


def table_bytes(E, n_used, T):
    """Routing tables alone: offsets [E+1] and pair ids [T*n_used], int32, and
    the activation-row scales [T*n_used], fp32, each padded to 256 bytes (the
    documented workspace layout)."""
    pad = lambda b: (b + 255) // 256 * 256
    return pad((E + 1) * 4) + 2 * pad(T * n_used * 4)


def run_moe(qmm, dev, W, X, ids_buf, ld_ids, n_used, T, status=None, ws_bytes=None):
    E, N, K = W.shape
    tiles = torch.cat([qmm.pack_q4(W[e].to(dev)) for e in range(E)])
    full = torch.full((T, n_used, N + 4), float("nan"), dtype=torch.float32, device=dev)
    Y = full[:, :, :N]
    ws = None if ws_bytes is None else torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    qmm.q4_gemm_id(tiles, E, N, K, X.to(dev), ids_buf.to(dev), ld_ids, n_used, T, Y=Y,
                   workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    f = full.cpu()
    assert torch.isnan(f[:, :, N:]).all(), "canary overwritten"
    # the oracle gets its own packing; the GPU's must be the same bytes
    ref = np.concatenate([O.pack_q4(W[e].numpy()) for e in range(E)])
    assert np.array_equal(tiles.cpu().numpy(), ref)
    return ref, f[:, :, :N].numpy()


@pytest.mark.parametrize("shared", [True, False])
def test_moe_small_full(qmm, cuda, shared):
    g = torch.Generator().manual_seed(5)
    E, N, K, T, n_used, ld = 8, 64, 512, 37, 3, 5
    W = torch.randn((E, N, K), generator=g) * 0.02
    ids_buf = torch.randint(0, E, (T, ld), generator=g, dtype=torch.int32)
    X = torch.randn((T, K) if shared else (T, n_used, K), generator=g).to(torch.bfloat16)
    tiles, Y = run_moe(qmm, cuda, W, X, ids_buf, ld, n_used, T)
    y, norm = O.q4_gemm_id(tiles, E, N, K, X.float().double().numpy(), shared,
                           ids_buf.numpy(), ld, n_used, T)
    assert O.normalized_error(Y, y, norm) <= TOL


def test_moe_contiguous_read_would_differ(qmm, cuda):
    # the ids view has row stride 17 while n_used = 8: reading 8 contiguous ids
    # per token would hand token t the experts of other tokens
    c = I.moe_case("gate", T=16, n_expert=32)
    Wsmall = c.W[:, :64, :512].contiguous()
    X = c.X[:, :512].contiguous()
    ids = c.ids_buf.contiguous()
    assert ids.shape == (16, 17)
    tiles, Y = run_moe(qmm, cuda, Wsmall, X, ids, 17, 8, 16)
    y, norm = O.q4_gemm_id(tiles, 32, 64, 512, X.float().double().numpy(), True, ids.numpy(), 17, 8, 16)
    assert O.normalized_error(Y, y, norm) <= TOL
    wrong = ids.numpy().reshape(-1)[:16 * 8].reshape(16, 8)
    y_wrong, _ = O.q4_gemm_id(tiles, 32, 64, 512, X.float().double().numpy(), True,
                              wrong.reshape(-1), 8, 8, 16)
    assert O.normalized_error(Y, y_wrong, norm) > 0.01


@pytest.mark.parametrize("T", [6, 150])
def test_moe_bad_id_sets_status(qmm, cuda, T):
    # T=6: the grouped kernel routes in-CTA; T=150: router + packed activations
    g = torch.Generator().manual_seed(6)
    E, N, K, n_used, ld = 4, 32, 256, 2, 3
    W = torch.randn((E, N, K), generator=g) * 0.02
    ids = torch.randint(0, E, (T, ld), generator=g, dtype=torch.int32)
    ids[2, 1] = E          # out of range
    ids[4, 0] = -1
    X = torch.randn((T, K), generator=g).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    tiles, Y = run_moe(qmm, cuda, W, X, ids, ld, n_used, T, status=status)
    assert int(status.item()) == qmm.QMM_ERR_BAD_EXPERT_ID
    assert np.isnan(Y[2, 1]).all() and np.isnan(Y[4, 0]).all()
    good = ids.clone()
    good[2, 1] = 0
    good[4, 0] = 0
    y, norm = O.q4_gemm_id(tiles, E, N, K, X.float().double().numpy(), True, good.numpy(), ld, n_used, T)
    mask = np.ones((T, n_used), bool)
    mask[2, 1] = mask[4, 0] = False
    assert O.normalized_error(Y[mask], y[mask], norm[mask]) <= TOL


@pytest.mark.parametrize("kind", ["gate", "down"])
def test_workload_moe_sampled(qmm, cuda, kind):
    """128 experts, top-8 of 17 stored ids, 512 tokens: all pairs computed on
    the GPU, 24 sampled pairs checked against the oracle."""
    c = I.moe_case(kind)
    tiles, Y = run_moe(qmm, cuda, c.W, c.X, c.ids_buf, c.ld_ids, c.n_used, c.T)
    rng = np.random.default_rng(10)
    ids = O.moe_ids_view(c.ids_buf.numpy(), c.ld_ids, c.n_used, c.T)
    per = (c.N // 32) * (c.K // 256) * 5120
    Xn = c.X.float().double().numpy()
    dense = {}
    for _ in range(24):
        t, i = int(rng.integers(c.T)), int(rng.integers(c.n_used))
        e = int(ids[t, i])
        if e not in dense:
            dense[e] = O.q4_decode(tiles[e * per:(e + 1) * per], c.N, c.K)
        x = Xn[t] if c.shared_src1 else Xn[t, i]
        y = dense[e] @ x
        norm = np.abs(dense[e]) @ np.abs(x)
        assert O.normalized_error(Y[t, i], y, norm) <= TOL
    assert np.isfinite(Y).all()


def test_moe_passes_partial_rows_empty_expert(qmm, cuda):
    """One expert with more pairs than a pass holds (64), N not a multiple of
    the 128-row CTA block, K shorter than the staging pipeline, and an expert
    that no pair selects."""
    g = torch.Generator().manual_seed(11)
    E, N, K, T, n_used, ld = 3, 96, 256, 150, 2, 3
    W = torch.randn((E, N, K), generator=g) * 0.02
    ids = torch.zeros((T, ld), dtype=torch.int32)
    ids[::7, 1] = 1                      # expert 1: a few pairs; expert 2: none
    ids[:, 2] = 2                        # outside the n_used view
    X = torch.randn((T, K), generator=g).to(torch.bfloat16)
    tiles, Y = run_moe(qmm, cuda, W, X, ids, ld, n_used, T)
    y, norm = O.q4_gemm_id(tiles, E, N, K, X.float().double().numpy(), True, ids.numpy(), ld, n_used, T)
    assert O.normalized_error(Y, y, norm) <= TOL


def test_moe_router_table_mode(qmm, cuda):
    """More (token, slot) pairs than the in-kernel scan covers: the one-CTA
    router fills the workspace and the grouped kernel reads it."""
    g = torch.Generator().manual_seed(12)
    E, N, K, T, n_used, ld = 8, 32, 256, 1040, 8, 9
    W = torch.randn((E, N, K), generator=g) * 0.02
    ids = torch.randint(0, E, (T, ld), generator=g, dtype=torch.int32)
    X = torch.randn((T, n_used, K), generator=g).to(torch.bfloat16)
    tiles, Y = run_moe(qmm, cuda, W, X, ids, ld, n_used, T)
    y, norm = O.q4_gemm_id(tiles, E, N, K, X.float().double().numpy(), False, ids.numpy(), ld, n_used, T)
    assert O.normalized_error(Y, y, norm) <= TOL


@pytest.mark.parametrize("kind", ["gate", "down"])
def test_workload_moe_full(qmm, cuda, kind):
    """128 experts, top-8 of 17 stored ids, 512 tokens: every pair against the
    oracle."""
    c = I.moe_case(kind)
    tiles, Y = run_moe(qmm, cuda, c.W, c.X, c.ids_buf, c.ld_ids, c.n_used, c.T)
    y, norm = O.q4_gemm_id(tiles, c.n_expert, c.N, c.K, c.X.float().double().numpy(), c.shared_src1,
                           c.ids_buf.numpy(), c.ld_ids, c.n_used, c.T)
    assert O.normalized_error(Y, y, norm) <= TOL


@pytest.mark.parametrize("kind", ["gate", "down"])
def test_workload_moe_tables_only_workspace(qmm, cuda, kind):
    """A workspace holding only the routing tables and row scales runs the
    in-kernel gather of the activation rows; every pair against the oracle."""
    c = I.moe_case(kind)
    full = qmm.q4_gemm_id_workspace_size(c.n_expert, c.n_used, c.T, c.K)
    tb = table_bytes(c.n_expert, c.n_used, c.T)
    assert full == tb + c.T * c.n_used * c.K * 2
    tiles, Y = run_moe(qmm, cuda, c.W, c.X, c.ids_buf, c.ld_ids, c.n_used, c.T, ws_bytes=tb)
    y, norm = O.q4_gemm_id(tiles, c.n_expert, c.N, c.K, c.X.float().double().numpy(), c.shared_src1,
                           c.ids_buf.numpy(), c.ld_ids, c.n_used, c.T)
    assert O.normalized_error(Y, y, norm) <= TOL


# ---------------------------------------------------------------------------
# the gate/up pair in one call (qmm_q4_gemm_id_pair)
# ---------------------------------------------------------------------------
def run_pair(qmm, dev, Wg, Wu, X, ids_buf, ld_ids, n_used, T, ws_bytes=None, status=None):
    E, N, K = Wg.shape
    tg = torch.cat([qmm.pack_q4(Wg[e].to(dev)) for e in range(E)])
    tu = torch.cat([qmm.pack_q4(Wu[e].to(dev)) for e in range(E)])
    fg = torch.full((T, n_used, N + 4), float("nan"), dtype=torch.float32, device=dev)
    fu = torch.full((T, n_used, N + 4), float("nan"), dtype=torch.float32, device=dev)
    ws = None if ws_bytes is None else torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    qmm.q4_gemm_id_pair(tg, tu, E, N, K, X.to(dev), ids_buf.to(dev), ld_ids, n_used, T, Y_gate=fg[:, :, :N],
                        Y_up=fu[:, :, :N], workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    out = []
    for f, W, t in ((fg, Wg, tg), (fu, Wu, tu)):
        h = f.cpu()
        assert torch.isnan(h[:, :, N:]).all(), "canary overwritten"
        ref = np.concatenate([O.pack_q4(W[e].numpy()) for e in range(E)])
        assert np.array_equal(t.cpu().numpy(), ref)
        y, norm = O.q4_gemm_id(ref, E, N, K, X.float().double().numpy(), True, ids_buf.numpy(), ld_ids, n_used, T)
        out.append((h[:, :, :N].numpy(), y, norm))
    return out


def test_moe_pair_small(qmm, cuda):
    g = torch.Generator().manual_seed(21)
    E, N, K, T, n_used, ld = 8, 96, 512, 45, 3, 5
    Wg = torch.randn((E, N, K), generator=g) * 0.02
    Wu = torch.randn((E, N, K), generator=g) * 0.02
    ids_buf = torch.randint(0, E, (T, ld), generator=g, dtype=torch.int32)
    X = torch.randn((T, K), generator=g).to(torch.bfloat16)
    for Y, y, norm in run_pair(qmm, cuda, Wg, Wu, X, ids_buf, ld, n_used, T):
        assert O.normalized_error(Y, y, norm) <= TOL


@pytest.mark.parametrize("tables_only", [False, True])
def test_workload_moe_pair_full(qmm, cuda, tables_only):
    """The C5 gate and up matrices (128 experts, top-8 of 17, 512 tokens) in
    one call, with the packed activations and with the gather mode; every
    pair of both outputs against the oracle, and bit-identical to two
    separate qmm_q4_gemm_id calls."""
    cg, cu = I.moe_case("gate"), I.moe_case("up")
    ws = table_bytes(cg.n_expert, cg.n_used, cg.T) if tables_only else None
    res = run_pair(qmm, cuda, cg.W, cu.W, cg.X, cg.ids_buf, cg.ld_ids, cg.n_used, cg.T, ws_bytes=ws)
    for Y, y, norm in res:
        assert O.normalized_error(Y, y, norm) <= TOL
    # same bits as the separate calls (same kernels, same per-output order)
    _, Yg = run_moe(qmm, cuda, cg.W, cg.X, cg.ids_buf, cg.ld_ids, cg.n_used, cg.T, ws_bytes=ws)
    _, Yu = run_moe(qmm, cuda, cu.W, cg.X, cg.ids_buf, cg.ld_ids, cg.n_used, cg.T, ws_bytes=ws)
    assert np.array_equal(res[0][0], Yg) and np.array_equal(res[1][0], Yu)

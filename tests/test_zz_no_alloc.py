"""MUL_MAT_ID for callers that cannot allocate device memory.

Plugins whose host framework owns all device memory, and latency-critical
paths that must not call cudaMalloc, use qmm_q4_gemm_id_noalloc.  It keeps its
routing tables and activation-row scales in a fixed array inside the library
instead of a workspace from the caller.  Small calls also pack their
activation rows into that array; larger ones gather the rows inside the
grouped kernel.  This file checks, through the C ABI, that calls in a row give
what the workspace entry point qmm_q4_gemm_id gives (both modes), and that
requests beyond the array's limits are refused.  pytest collects this file
last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _case(seed, E, N, K, T, n_used, ld, shared, dev):
    g = torch.Generator().manual_seed(seed)
    W = torch.randn((E, N, K), generator=g) * 0.02
    ids = torch.randint(0, E, (T, ld), generator=g, dtype=torch.int32)
    X = torch.randn((T, K) if shared else (T, n_used, K), generator=g).to(torch.bfloat16)
    return W, ids, X


def test_noalloc_matches_workspace_entry_point_twice(qmm, cuda):
    # calls in a row with different routing: each must not see the previous one's tables.
    # The first two fit their packed activation rows in the array; the third
    # (512 pairs x K=2048 x 2 bytes = 2 MiB of rows) runs the gather mode.
    for seed, (E, N, K, T, n_used, ld, shared) in ((1, (16, 64, 512, 61, 4, 9, True)),
                                                   (2, (5, 96, 256, 23, 3, 3, False)),
                                                   (3, (128, 256, 2048, 64, 8, 17, True))):
        W, ids, X = _case(seed, E, N, K, T, n_used, ld, shared, cuda)
        tiles = torch.cat([qmm.pack_q4(W[e].to(cuda)) for e in range(E)])
        Xd, idsd = X.to(cuda), ids.to(cuda)
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        Y_ref = qmm.q4_gemm_id(tiles, E, N, K, Xd, idsd, ld, n_used, T)
        Y_na = torch.full((T, n_used, N), float("nan"), dtype=torch.float32, device=cuda)
        qmm.q4_gemm_id_noalloc(tiles, E, N, K, Xd, idsd, ld, n_used, T, Y_na, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref_tiles = np.concatenate([O.pack_q4(W[e].numpy()) for e in range(E)])
        assert np.array_equal(tiles.cpu().numpy(), ref_tiles)
        y, norm = O.q4_gemm_id(ref_tiles, E, N, K, X.float().double().numpy(), shared,
                               ids.numpy(), ld, n_used, T)
        err = O.normalized_error(Y_na.cpu().numpy(), Y_ref.cpu().numpy(), norm)
        assert err <= TOL, err
        assert O.normalized_error(Y_na.cpu().numpy(), y, norm) <= TOL


def test_noalloc_rejects_requests_beyond_its_scratch(qmm, cuda):
    P = torch.zeros(16, dtype=torch.uint8, device=cuda)
    # T * n_used = 65537 > 65536 pairs, and 1025 > 1024 experts
    for n_expert, T, n_used in ((4, 65537, 1), (1025, 1, 1)):
        st = qmm.lib.qmm_q4_gemm_id_noalloc(
            qmm._ptr(P), n_expert, 32, 256, qmm._ptr(P), 256, 0, qmm._ptr(P), n_used, n_used, T,
            qmm._ptr(P), 32 * n_used, 32, None, qmm._stream())
        assert st == qmm.QMM_ERR_WORKSPACE

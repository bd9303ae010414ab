"""GPU parity of the grouped decode GEMV (qmm_q4_gemv_group): several q4
weight sets at M = 1 in one launch, each output against the fp64 oracle at
the decode kernels' level (2e-5 * sum|x||w|: weights are never rounded), with
canaries around every output, and repeat calls bit-identical."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O

pytestmark = pytest.mark.gpu
TOL = 2e-5

# the Qwen3-0.6B projection shapes (K, N): q, k, v, o, gate, up, down
QWEN3_PROJ = [(1024, 2048), (1024, 1024), (1024, 1024), (2048, 1024), (1024, 3072), (1024, 3072), (3072, 1024)]


def make_group(qmm, dev, shapes, seed, shared_x=False):
    g = torch.Generator().manual_seed(seed)
    probs, host, bufs = [], [], []
    x_shared = None
    for (K, N) in shapes:
        W = torch.randn((N, K), generator=g) * 0.02
        if shared_x:
            if x_shared is None or x_shared.numel() != K:
                x_shared = torch.randn(K, generator=g).to(torch.bfloat16).to(dev)
            x = x_shared
        else:
            x = torch.randn(K, generator=g).to(torch.bfloat16).to(dev)
        tiles = qmm.pack_q4(W.to(dev))
        buf = torch.full((N + 8,), float("nan"), dtype=torch.float32, device=dev)
        probs.append((tiles, N, K, x, buf[4:4 + N]))
        bufs.append(buf)
        host.append((O.pack_q4(W.numpy()), N, K, x.cpu().float().double().numpy()[None, :]))
    return probs, host, bufs


def check(probs, host, bufs):
    torch.cuda.synchronize()
    for (tiles, N, K, x, y), (ht, _, _, hx), buf in zip(probs, host, bufs):
        b = buf.cpu()
        assert torch.isnan(b[:4]).all() and torch.isnan(b[4 + N:]).all(), "canary overwritten"
        assert np.array_equal(tiles.cpu().numpy(), ht)
        ref, norm = O.q4_gemm(ht, N, K, hx)
        err = O.normalized_error(y.cpu().numpy()[None, :], ref, norm)
        assert err <= TOL, (N, K, err)


def test_group_qwen3_projection_set(qmm, cuda):
    probs, host, bufs = make_group(qmm, cuda, QWEN3_PROJ, 11)
    qmm.q4_gemv_group(probs)
    check(probs, host, bufs)
    first = [y.clone() for (_, _, _, _, y) in probs]
    qmm.q4_gemv_group(probs)
    torch.cuda.synchronize()
    for a, (_, _, _, _, b) in zip(first, probs):
        assert torch.equal(a, b), "repeat call differs"


def test_group_shared_x_and_single_row_problems(qmm, cuda):
    # q/k/v-style problems reading one x, and problems of one tile row or one tile
    shapes = [(1024, 2048), (1024, 1024), (1024, 1024), (256, 32), (512, 32), (2816, 64)]
    probs, host, bufs = make_group(qmm, cuda, shapes, 12, shared_x=False)
    qmm.q4_gemv_group(probs)
    check(probs, host, bufs)
    probs, host, bufs = make_group(qmm, cuda, [(1024, 2048), (1024, 1024), (1024, 1024)], 13, shared_x=True)
    qmm.q4_gemv_group(probs)
    check(probs, host, bufs)


def test_group_single_problem(qmm, cuda):
    for (K, N) in [(256, 32), (1024, 96), (4096, 4096)]:
        probs, host, bufs = make_group(qmm, cuda, [(K, N)], K + N)
        qmm.q4_gemv_group(probs)
        check(probs, host, bufs)


def test_group_more_problems_than_one_launch(qmm, cuda):
    # 40 problems: the call splits them over two launches (32 per launch)
    shapes = [(256 * (1 + i % 5), 32 * (1 + i % 3)) for i in range(40)]
    probs, host, bufs = make_group(qmm, cuda, shapes, 14)
    qmm.q4_gemv_group(probs)
    check(probs, host, bufs)


def test_group_more_rows_than_one_launch_and_large_k(qmm, cuda):
    # 7,168 tile rows (over the 6,144 of one launch), then a K above the
    # grouped kernel's limit, which runs as its own launch
    shapes = [(256, 32768)] * 7 + [(16640, 64), (512, 64)]
    probs, host, bufs = make_group(qmm, cuda, shapes, 15)
    qmm.q4_gemv_group(probs)
    check(probs, host, bufs)


def test_group_special_values(qmm, cuda):
    # constant blocks (scale 0), a zero weight row, one-hot and zero activations
    dev = cuda
    g = torch.Generator().manual_seed(16)
    W1 = torch.randn((64, 512), generator=g) * 0.02
    W1[5, 32:64] = 0.125
    W1[7] = 0.0
    W2 = torch.randn((32, 256), generator=g) * 0.02
    x1 = torch.zeros(512).to(torch.bfloat16)
    x1[300] = 1
    x2 = torch.zeros(256).to(torch.bfloat16)
    probs, host, bufs = [], [], []
    for W, x in [(W1, x1), (W2, x2)]:
        N, K = W.shape
        buf = torch.full((N + 8,), float("nan"), dtype=torch.float32, device=dev)
        probs.append((qmm.pack_q4(W.to(dev)), N, K, x.to(dev), buf[4:4 + N]))
        bufs.append(buf)
        host.append((O.pack_q4(W.numpy()), N, K, x.float().double().numpy()[None, :]))
    qmm.q4_gemv_group(probs)
    check(probs, host, bufs)
    assert torch.count_nonzero(probs[1][4]).item() == 0

"""GPU parity of the grouped small-M int8 GEMM (qmm_int8_gemm_group): each
problem bit-exact against the oracle, with canaries around every output."""
import numpy as np
import pytest
import torch

import oracle.qmm_oracle as O
from quantized_matmul_qmm_gb300 import inputs as I

from test_gpu_int8 import assert_same, oracle_out, rand_codes

pytestmark = pytest.mark.gpu

CANARY = {"s32": 0x5A5A5A5A, "f32": 0x7FC0DEAD, "s8": 77, "u8": 201}


def padded_out(qmm, dev, M, N, out_type):
    full = torch.empty((M + 1, N + 3), dtype=qmm.TORCH_OUT[out_type], device=dev)
    (full.view(torch.int32) if out_type == "f32" else full).fill_(CANARY[out_type])
    return full, full[:M, :N]


def check_canary(full, M, N, out_type):
    raw = full.cpu()
    raw = raw.view(torch.int32) if out_type == "f32" else raw
    assert torch.all(raw[:, N:] == CANARY[out_type]) and torch.all(raw[M, :] == CANARY[out_type])


def run_group(qmm, dev, cases):
    """cases: list of dicts (CPU tensors + scalars); returns [(got, ref)]."""
    probs, fulls = [], []
    for c in cases:
        M, K = c["A"].shape
        N = c["B"].shape[1]
        packed, col_scale, col_sum = qmm.pack_b_int8(c["B"].to(dev), c["b_type"])
        lda = (K + 15) // 16 * 16
        Ad = torch.zeros((M, lda), dtype=c["A"].dtype, device=dev)
        Ad[:, :K] = c["A"].to(dev)
        full, out = padded_out(qmm, dev, M, N, c["out_type"])
        s_w = c.get("s_w")
        if s_w is None and c["b_type"] == "f32":
            s_w = col_scale
        elif s_w is not None:
            s_w = s_w.to(dev)
        s_x = c.get("s_x")
        probs.append(dict(A=Ad[:, :K], a_type=c["a_type"], zA=c["zA"], packed=packed, col_sum=col_sum, N=N,
                          b_orig_type=c["b_type"], zB=c["zB"], out_type=c["out_type"],
                          bias=None if c.get("bias") is None else c["bias"].to(dev),
                          s_x=None if s_x is None else torch.as_tensor(s_x, dtype=torch.float32).reshape(-1).to(dev),
                          s_x_stride=c.get("s_x_stride", 0), s_w=s_w, s_y=c.get("s_y", 1.0),
                          zp_y=c.get("zp_y", 0), out=out))
        fulls.append((full, M, N, c["out_type"]))
    qmm.int8_gemm_group(probs)
    torch.cuda.synchronize()
    res = []
    for c, p, (full, M, N, ot) in zip(cases, probs, fulls):
        check_canary(full, M, N, ot)
        sw = c.get("s_w")
        ref = oracle_out(c["A"], c["a_type"], c["zA"], c["B"], c["b_type"], c["zB"], ot, bias=c.get("bias"),
                         s_x=c.get("s_x"), s_w=None if sw is None else sw.numpy(), s_y=c.get("s_y", 1.0),
                         zp_y=c.get("zp_y", 0))
        res.append((p["out"].cpu().numpy(), ref, ot))
    return res


def test_group_qwen3_projection_set_m32(qmm, cuda):
    """The seven Qwen3-0.6B projections at M = 32 (per-tensor int8
    activations, packB weights, fp32 out) as one grouped call."""
    cases = []
    for idx in range(7):
        c = I.int8_qwen_projection(idx)
        cases.append(dict(A=c.A, a_type=c.a_type, zA=c.zA, B=c.B, b_type=c.b_type, zB=c.zB, out_type="f32",
                          s_x=c.s_x))
    for got, ref, ot in run_group(qmm, cuda, cases):
        assert_same(got, ref, ot)


def test_group_mixed_problems(qmm, cuda):
    """Different M (1..64), K (ragged), N, operand types, zero points and
    every output type in one launch, then 20 problems (two launches)."""
    g = torch.Generator().manual_seed(77)
    specs = [(1, 64, 8, "u8", "s8", "s32"), (16, 1024, 1024, "u8", "s8", "f32"), (33, 1000, 130, "s8", "u8", "s8"),
             (64, 4608, 200, "u8", "u8", "u8"), (7, 257, 65, "s8", "f32", "f32"), (48, 3000, 96, "u8", "s8", "s32")]
    specs = specs + [(1 + i, 64 * (1 + i % 4) + 3, 32 + 8 * i, "u8", "s8", "s32") for i in range(14)]
    cases = []
    for (M, K, N, at, bt, ot) in specs:
        A = rand_codes(g, at, (M, K))
        B = torch.randn((K, N), generator=g) * 0.02 if bt == "f32" else rand_codes(g, bt, (K, N))
        zA = int(torch.randint(0, 256, (1,), generator=g)) if at == "u8" else int(torch.randint(-128, 128, (1,), generator=g))
        zB = 0 if bt == "f32" else (int(torch.randint(0, 256, (1,), generator=g)) if bt == "u8" else 3)
        c = dict(A=A, a_type=at, zA=zA, B=B, b_type=bt, zB=zB, out_type=ot,
                 bias=torch.randint(-3000, 3000, (N,), generator=g, dtype=torch.int32))
        if ot != "s32":
            c["s_x"] = (torch.rand(M, generator=g) * 0.01 + 0.001).numpy()
            c["s_x_stride"] = 1
            if bt != "f32":
                c["s_w"] = (torch.rand(N, generator=g) * 9e-3 + 1e-3).float()
        if ot in ("s8", "u8"):
            c["s_y"], c["zp_y"] = 40.0, 3
        cases.append(c)
    for got, ref, ot in run_group(qmm, cuda, cases[:6]):
        assert_same(got, ref, ot)
    for got, ref, ot in run_group(qmm, cuda, cases):
        assert_same(got, ref, ot)


def test_group_stream_and_cluster_forms(qmm, cuda):
    """A group that splits into a streaming batch (the first two problems:
    158 items of 16 columns) and a cluster batch (the next three do not fit
    the streaming form together with them, and have too few items alone):
    operand types, zero points with row sums, every output type."""
    g = torch.Generator().manual_seed(5)
    specs = [(5, 700, 1500, "u8", "s8", "s32"), (32, 3072, 1024, "s8", "u8", "f32"), (64, 1500, 900, "u8", "u8", "u8"),
             (1, 64, 40, "s8", "f32", "f32"), (20, 2000, 777, "u8", "s8", "s8")]
    cases = []
    for (M, K, N, at, bt, ot) in specs:
        A = rand_codes(g, at, (M, K))
        B = torch.randn((K, N), generator=g) * 0.02 if bt == "f32" else rand_codes(g, bt, (K, N))
        zA = int(torch.randint(0, 256, (1,), generator=g)) if at == "u8" else int(torch.randint(-128, 128, (1,), generator=g))
        zB = 0 if bt == "f32" else (int(torch.randint(0, 256, (1,), generator=g)) if bt == "u8" else -4)
        c = dict(A=A, a_type=at, zA=zA, B=B, b_type=bt, zB=zB, out_type=ot,
                 bias=torch.randint(-3000, 3000, (N,), generator=g, dtype=torch.int32))
        if ot != "s32":
            c["s_x"] = (torch.rand(M, generator=g) * 0.01 + 0.001).numpy()
            c["s_x_stride"] = 1
            if bt != "f32":
                c["s_w"] = (torch.rand(N, generator=g) * 9e-3 + 1e-3).float()
        if ot in ("s8", "u8"):
            c["s_y"], c["zp_y"] = 40.0, 3
        cases.append(c)
    for got, ref, ot in run_group(qmm, cuda, cases):
        assert_same(got, ref, ot)

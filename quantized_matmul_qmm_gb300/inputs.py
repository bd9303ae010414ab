"""Seeded synthetic inputs for the five workloads.

This module only draws random numbers and arranges them into buffers.  It
holds none of the library's arithmetic: no packing, no quantisation of
weights, no zero-point algebra.  The tests, the benchmark and the CPU oracle
all read the same host tensors it returns, so both sides see identical bytes.

Every generator uses ``torch.Generator`` (CPU) seeded with the workload's
seed and returns CPU tensors.

Workloads:
* int8 GEMM, M=16 K=1024 N=1024 (seed 0): uint8 A, zA = 128 + U{-8..8},
  int8 B in [-127, 127], zB = 0, per-column scales in [1e-3, 1e-2].
* Qwen3-0.6B projection set at M=32 (seeds 1..7): fp32 weights N(0, 0.02) for
  packB, and int8 activation codes round(32*N(0,1)) clipped to +-127 with a
  per-tensor scale of 1/32.
* Large uint8 x int8 GEMM, M=4096 K=N=4608 (seed 8): zA in [0,255], zB in
  [-8,8], int32 bias, int8 output.
* 4-bit GEMM/GEMV (seed 9): fp32 weights N(0, 0.02) [N][K], bf16 activations
  N(0,1) [M][K].
* 4-bit MoE MUL_MAT_ID (seed 10): 128 experts, top-8 of 17 stored ids per token.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

QWEN3_06B_PROJ = [  # (K, N) of q, k, v, o, gate, up, down in Qwen3-0.6B
    ("q_proj", 1024, 2048),
    ("k_proj", 1024, 1024),
    ("v_proj", 1024, 1024),
    ("o_proj", 2048, 1024),
    ("gate_proj", 1024, 3072),
    ("up_proj", 1024, 3072),
    ("down_proj", 3072, 1024),
]
QWEN3_06B_LM_HEAD = ("lm_head", 1024, 151936)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _randint(g, lo, hi_incl, shape, dtype):
    return torch.randint(lo, hi_incl + 1, shape, generator=g, dtype=torch.int64).to(dtype)


def _uniform(g, lo, hi, shape):
    return (torch.rand(shape, generator=g, dtype=torch.float64) * (hi - lo) + lo).to(torch.float32)


@dataclass
class Int8Case:
    """Inputs of one int8 GEMM call (all CPU tensors)."""
    name: str
    M: int
    K: int
    N: int
    A: torch.Tensor                 # [M][K] uint8 or int8
    a_type: str                     # "u8" | "s8"
    zA: int
    B: torch.Tensor                 # [K][N] fp32, int8 or uint8 (unpacked weights)
    b_type: str                     # "f32" | "s8" | "u8"
    zB: int
    out_type: str                   # "s32" | "f32" | "s8" | "u8"
    bias: torch.Tensor | None = None   # [N] int32
    s_x: torch.Tensor | float | None = None  # scalar or [M] fp32
    s_w: torch.Tensor | None = None    # [N] fp32 (integer weights only; fp32 weights get packB scales)
    s_y: float = 1.0
    zp_y: int = 0
    extra_out: list = field(default_factory=list)


def int8_gemm_small(seed: int = 0, M: int = 16, K: int = 1024, N: int = 1024) -> Int8Case:
    g = _gen(seed)
    A = _randint(g, 0, 255, (M, K), torch.uint8)
    zA = 128 + int(_randint(g, -8, 8, (1,), torch.int64))
    B = _randint(g, -127, 127, (K, N), torch.int8)
    s_w = _uniform(g, 1e-3, 1e-2, (N,))
    return Int8Case("int8_m16_k1024_n1024", M, K, N, A, "u8", zA, B, "s8", 0, "s32",
                    s_w=s_w, extra_out=["f32"])


def int8_qwen_projection(idx: int, M: int = 32) -> Int8Case:
    name, K, N = QWEN3_06B_PROJ[idx]
    g = _gen(1 + idx)
    W = (torch.randn((K, N), generator=g, dtype=torch.float64) * 0.02).to(torch.float32)
    a = torch.randn((M, K), generator=g, dtype=torch.float64) * 32.0
    A = torch.clamp(torch.round(a), -127, 127).to(torch.int8)
    return Int8Case(f"qwen3_0.6b_{name}_m{M}", M, K, N, A, "s8", 0, W, "f32", 0, "f32",
                    s_x=1.0 / 32.0)


def int8_gemm_large(seed: int = 8, M: int = 4096, K: int = 4608, N: int = 4608) -> Int8Case:
    g = _gen(seed)
    A = _randint(g, 0, 255, (M, K), torch.uint8)
    zA = int(_randint(g, 0, 255, (1,), torch.int64))
    B = _randint(g, -128, 127, (K, N), torch.int8)
    zB = int(_randint(g, -8, 8, (1,), torch.int64))
    s_x = 1.0 / 64.0
    s_w = _uniform(g, 1e-3, 1e-2, (N,))
    bias_real = torch.randn((N,), generator=g, dtype=torch.float64)
    bias = torch.round(bias_real / (s_x * s_w.double())).to(torch.int32)
    # output scale: the root-mean-square of sum_k (A-zA)(B-zB) under the input
    # distributions, mapped to 48 output steps at the mean weight scale
    ea, ea2 = 127.5 - zA, (255 * 257 / 12.0) + (127.5 - zA) ** 2
    eb, eb2 = -0.5 - zB, (255 * 257 / 12.0) + (-0.5 - zB) ** 2
    rms = math.sqrt(K * ea2 * eb2 + K * (K - 1) * (ea * eb) ** 2)
    s_y = float(torch.tensor(s_x * float(s_w.double().mean()) * rms / 48.0, dtype=torch.float32))
    return Int8Case(f"int8_u8s8_m{M}_k{K}_n{N}", M, K, N, A, "u8", zA, B, "s8", zB, "s8",
                    bias=bias, s_x=s_x, s_w=s_w, s_y=s_y, zp_y=0)


@dataclass
class Q4Case:
    name: str
    M: int
    K: int
    N: int
    W: torch.Tensor   # [N][K] fp32
    X: torch.Tensor   # [M][K] bf16


def q4_weights(seed: int, N: int, K: int) -> torch.Tensor:
    g = _gen(seed)
    return (torch.randn((N, K), generator=g, dtype=torch.float32) * 0.02)


def q4_activations(seed: int, M: int, K: int) -> torch.Tensor:
    g = _gen(seed)
    return torch.randn((M, K), generator=g, dtype=torch.float32).to(torch.bfloat16)


def q4_case(name: str, K: int, N: int, M: int, seed: int = 9) -> Q4Case:
    # weights and activations draw from separate streams so a shape's weights
    # are the same at M=1 and M=512
    return Q4Case(f"q4_{name}_m{M}", M, K, N, q4_weights(seed * 1000 + N % 997 + K, N, K),
                  q4_activations(seed * 7919 + M, M, K))


@dataclass
class MoECase:
    name: str
    n_expert: int
    n_used: int
    T: int
    K: int
    N: int
    shared_src1: bool
    W: torch.Tensor      # [n_expert][N][K] fp32
    X: torch.Tensor      # [T][K] or [T][n_used][K] bf16
    ids_buf: torch.Tensor  # [T][ld_ids] int32
    ld_ids: int


def moe_case(kind: str, seed: int = 10, n_expert: int = 128, n_used: int = 8, T: int = 512,
             hidden: int = 2048, inter: int = 768, ld_ids: int = 17) -> MoECase:
    """kind: "gate" / "up" (K=hidden, N=inter, shared src1) or "down"
    (K=inter, N=hidden, per-slot src1)."""
    g = _gen(seed)
    logits = torch.randn((T, n_expert), generator=g, dtype=torch.float32)
    order = torch.argsort(logits, dim=1, descending=True, stable=True)
    ids_buf = order[:, :ld_ids].to(torch.int32).contiguous()
    kseed = {"gate": 1, "up": 2, "down": 3}[kind]
    gw = _gen(seed * 100 + kseed)
    if kind == "down":
        K, N, shared = inter, hidden, False
        X = torch.randn((T, n_used, K), generator=gw, dtype=torch.float32).to(torch.bfloat16)
    else:
        K, N, shared = hidden, inter, True
        X = torch.randn((T, K), generator=gw, dtype=torch.float32).to(torch.bfloat16)
    W = torch.randn((n_expert, N, K), generator=gw, dtype=torch.float32) * 0.02
    return MoECase(f"moe_{kind}_e{n_expert}_top{n_used}_t{T}", n_expert, n_used, T, K, N, shared,
                   W, X, ids_buf, ld_ids)


def q4k_superblocks(seed: int, N: int, K: int, d_range=(1e-4, 2e-3), dmin_range=(1e-4, 2e-3)) -> torch.Tensor:
    """Random Q4_K super-blocks for an N x K weight: uint8 [N][K/256 * 144].

    Each 144-byte block holds two fp16 values drawn uniformly from the given
    ranges at bytes 0..3, then 140 uniformly random bytes (the twelve bytes of
    6-bit scale and min codes and the 128 bytes of 4-bit codes), so every
    scale, min and code value occurs.  Weights of N(0, 0.02) quantised to Q4_K
    have super-block scales in about this range."""
    assert K % 256 == 0
    g = _gen(seed)
    nsb = K // 256
    blk = _randint(g, 0, 255, (N, nsb, 144), torch.uint8)
    d = _uniform(g, d_range[0], d_range[1], (N, nsb)).to(torch.float16)
    dmin = _uniform(g, dmin_range[0], dmin_range[1], (N, nsb)).to(torch.float16)
    blk[:, :, 0:2] = d.view(torch.uint8).reshape(N, nsb, 2)
    blk[:, :, 2:4] = dmin.view(torch.uint8).reshape(N, nsb, 2)
    return blk.reshape(N, nsb * 144).contiguous()

#!/usr/bin/env python
"""Benchmark of the quantized projection matmul hot path on GB300.

One step is one pass over every row of the hot path, on seeded synthetic
inputs that are already resident in HBM:
  * int8 GEMM      uint8 x int8, M=4096 K=N=4608, zero points, bias, int8 out
  * q4 GEMV        lm_head (K=1024, N=151936) and the 7 Qwen3-0.6B projections, M=1
  * q4 prefill     the 7 projections and lm_head at M=512
  * q4 MUL_MAT_ID  128 experts, top-8 of 17 strided ids, 512 tokens: gate, up, down
Weight packing (packB, pack_q4) is done once, before timing, as the pages do it
("once per (tensor, K, N)").  L2 is flushed before every call of the step, outside
its timed bracket: a 256 MiB write, then a 256 MiB read, so that the lines left
in L2 are clean and hold none of the call's inputs.  (A write-only flush leaves
~L2-sized dirty data whose write-back lands inside the timed call; without a
flush between calls, a call pays for the write-back of its predecessor's
outputs and workspace, e.g. the int8 GEMM's 80 MB of f16 operands evicted by
the next weight stream.)  A step's time is the sum of its calls' times.

The printed `value` is int8 GEMM TOPS on the M=4096 K=N=4608 GEMM (the first
half of the metric).  The q4 GEMV weight bandwidth (its second half) is
reported in `gemv`: M=1 launches back to back over rotating copies of the
weights (>= 4x L2, so every launch streams from HBM), for lm_head and for the
7-projection set captured in a CUDA graph; the lm_head call timed alone after
a flush is kept beside it (`gemv.single_call`).  Every kernel's device time comes from CUDA events on the
launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl qmm|reference]

With N > 1 (torchrun, one rank per GPU) every rank runs an independent replica
of the step.  The path has no exchange step, so there is no collective in the
data path.  Timing is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HOST_LEAD_CYCLES = 4_000_000   # ~2 ms of GPU sleep at ~2 GHz before each timed step or pass
METRIC = "int8 GEMM TOPS (% tensor peak); 4-bit GEMV weight GB/s (% HBM) at 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
INT8_M, INT8_K, INT8_N = 4096, 4608, 4608
WORKLOAD = ("qmm hot path: int8 GEMM u8xs8 M=4096 K=N=4608 (int8 out); q4 GEMV M=1 lm_head "
            "K=1024 N=151936 + 7 Qwen3-0.6B projections; q4 prefill M=512 (same 8 weights); "
            "q4 MUL_MAT_ID 128 experts top-8/17 T=512 gate/up/down")


def load_traffic():
    """DRAM traffic per call from committed ncu captures (profiles/traffic.json),
    kept only while every source the kernels are built from still hashes to what
    was profiled."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        d = json.load(f)
    out = {}
    for name, rec in d.get("kernels", {}).items():
        fresh = True
        for src, digest in rec.get("sources", {}).items():
            fp = os.path.join(ROOT, src)
            if not os.path.exists(fp) or hashlib.sha256(open(fp, "rb").read()).hexdigest() != digest:
                fresh = False
        if fresh:
            out[name] = rec["dram_bytes_per_launch"]
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class HotPath:
    """All device buffers of one step, and the list of library calls."""

    def __init__(self, q, I, dev):
        import torch
        self.q, self.dev = q, dev
        self.calls = []          # (name, fn, launches, work dict)
        # int8 GEMM
        c = I.int8_gemm_large()
        self.int8 = c
        self.A = c.A.to(dev)
        packed, _, col_sum = q.pack_b_int8(c.B.to(dev), c.b_type)
        self.packed, self.col_sum = packed, col_sum
        # static weights: packed and widened to f16 once, outside the timed region
        self.b16 = q.widen_b_int8(packed, c.K, c.N)
        self.bias, self.s_w = c.bias.to(dev), c.s_w.to(dev)
        self.s_x = torch.tensor([c.s_x], dtype=torch.float32, device=dev)
        self.out8 = torch.empty((c.M, c.N), dtype=torch.int8, device=dev)
        ws = q.int8_gemm_workspace_size(c.M, c.K, c.N)
        self.ws8 = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.calls.append(("int8_gemm_m4096", self.run_int8, self.int8_launches(),
                           {"ops": 2 * c.M * c.N * c.K,
                            "bytes": c.M * c.K + c.N * q.pack_b_int8_size(c.K, 1) + 4 * c.N * 3 + c.M * c.N}))
        # q4 dense weights (lm_head + 7 projections), M=1 and M=512
        shapes = [I.QWEN3_06B_LM_HEAD] + list(I.QWEN3_06B_PROJ)
        self.q4 = []
        self.q4_ws = {}
        for name, K, N in shapes:
            W = I.q4_weights(9 * 1000 + N % 997 + K, N, K).to(dev)
            tiles = q.pack_q4(W)
            del W
            x1 = I.q4_activations(9 * 7919 + 1, 1, K).to(dev)
            x512 = I.q4_activations(9 * 7919 + 512, 512, K).to(dev)
            y1 = torch.empty((1, N), dtype=torch.float32, device=dev)
            y512 = torch.empty((512, N), dtype=torch.float32, device=dev)
            self.q4.append((name, K, N, tiles, x1, x512, y1, y512))
            self.q4_ws[name] = torch.empty(max(256, q.q4_gemm_workspace_size(512, K, N)), dtype=torch.uint8,
                                           device=dev)
        for name, K, N, tiles, x1, _, y1, _ in self.q4:
            wb = tiles.numel()
            self.calls.append((f"q4_gemv_{name}_m1", self._q4(tiles, N, K, x1, y1), 1,
                               {"weight_bytes": wb, "bytes": wb + 2 * K + 4 * N, "flops": 2 * N * K}))
        for name, K, N, tiles, _, x512, _, y512 in self.q4:
            wb = tiles.numel()
            self.calls.append((f"q4_gemm_{name}_m512", self._q4(tiles, N, K, x512, y512, self.q4_ws[name]),
                               self.q4_launches(512),
                               {"flops": 2 * 512 * N * K, "weight_bytes": wb,
                                "bytes": wb + 2 * 512 * K + 4 * 512 * N}))
        # MoE
        self.moe = []
        for kind in ("gate", "up", "down"):
            m = I.moe_case(kind)
            tiles = torch.cat([q.pack_q4(m.W[e].to(dev)) for e in range(m.n_expert)])
            X = m.X.to(dev)
            ids = m.ids_buf.to(dev)
            Y = torch.empty((m.T, m.n_used, m.N), dtype=torch.float32, device=dev)
            wsb = torch.empty(q.q4_gemm_id_workspace_size(m.n_expert, m.n_used, m.T, m.K),
                              dtype=torch.uint8, device=dev)
            touched = int(torch.unique(m.ids_buf[:, :m.n_used]).numel())
            per = tiles.numel() // m.n_expert
            self.moe.append((kind, m, tiles, X, ids, Y, wsb))
            self.calls.append((f"q4_moe_{kind}", self._moe(m, tiles, X, ids, Y, wsb), self.moe_launches(m),
                               {"flops": 2 * m.T * m.n_used * m.N * m.K, "weight_bytes": touched * per,
                                "bytes": touched * per + X.numel() * 2 + Y.numel() * 4}))
        # the gate/up pair in one call: both weight sets over the gate case's src1 and ids
        (_, mg, tg, Xg, idsg, _, wsg), (_, _, tu, _, _, _, _) = self.moe[0], self.moe[1]
        self.Yg2 = torch.empty((mg.T, mg.n_used, mg.N), dtype=torch.float32, device=dev)
        self.Yu2 = torch.empty_like(self.Yg2)
        touched = int(torch.unique(mg.ids_buf[:, :mg.n_used]).numel())
        per = tg.numel() // mg.n_expert
        self.calls.append(("q4_moe_gateup", lambda: q.q4_gemm_id_pair(
            tg, tu, mg.n_expert, mg.N, mg.K, Xg, idsg, mg.ld_ids, mg.n_used, mg.T, Y_gate=self.Yg2, Y_up=self.Yu2,
            workspace=wsg, dev_status=self.status), self.moe_launches(mg),
            {"flops": 2 * 2 * mg.T * mg.n_used * mg.N * mg.K, "weight_bytes": 2 * touched * per,
             "bytes": 2 * touched * per + Xg.numel() * 2 + 2 * self.Yg2.numel() * 4}))
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()

    def int8_launches(self):
        # tensor-core route: A's widen prepass + GEMM; other routes: one kernel
        c = self.int8
        return 2 if self.q.int8_gemm_workspace_size(c.M, c.K, c.N) > 0 else 1

    def moe_launches(self, m):
        # routing grid, packing grid (f16 rows and their scales), then the grouped kernel
        return 3

    def q4_launches(self, M):
        # decode GEMV: one kernel; tensor-core route: f16 activation rows, then the GEMM
        return 1 if M <= 16 else 2

    def run_int8(self):
        c = self.int8
        self.q.int8_gemm(self.A, c.a_type, c.zA, self.packed, self.col_sum, c.N, c.b_type, c.zB,
                         "s8", bias=self.bias, s_x=self.s_x, s_w=self.s_w, s_y=c.s_y, zp_y=c.zp_y,
                         out=self.out8, workspace=self.ws8, dev_status=self.status, b16=self.b16)

    def run_int8_widen_each_call(self):
        """The same call without the one-time f16 copy: the packed weights are
        widened again on every call."""
        c = self.int8
        self.q.int8_gemm(self.A, c.a_type, c.zA, self.packed, self.col_sum, c.N, c.b_type, c.zB,
                         "s8", bias=self.bias, s_x=self.s_x, s_w=self.s_w, s_y=c.s_y, zp_y=c.zp_y,
                         out=self.out8, workspace=self.ws8, dev_status=self.status)

    def _q4(self, tiles, N, K, X, Y, ws=None):
        return lambda: self.q.q4_gemm(tiles, N, K, X, Y=Y, workspace=ws, dev_status=self.status)

    def _moe(self, m, tiles, X, ids, Y, ws):
        return lambda: self.q.q4_gemm_id(tiles, m.n_expert, m.N, m.K, X, ids, m.ld_ids, m.n_used,
                                         m.T, Y=Y, workspace=ws, dev_status=self.status)


def max_over_ranks(values, world, device):
    """Elementwise max of `values` over the ranks.  The replicas run the same
    work, so the job is as slow as its slowest rank: every timing is the
    maximum over ranks before any rate is derived from it."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replicas_rate(per_replica_rate, world):
    """Whole-job throughput of `world` replicas, each at the rate taken from
    the slowest rank's time (weak scaling: the work per GPU is fixed)."""
    return world * per_replica_rate


def run_ours(args, rank, world, dev):
    import torch
    import torch.distributed as dist
    from quantized_matmul_qmm_gb300 import build as B
    B.build()
    import quantized_matmul_qmm_gb300.qmm as q
    from quantized_matmul_qmm_gb300 import inputs as I

    hp = HotPath(q, I, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ncalls = len(hp.calls)

    def flush_l2():
        flush.zero_()
        flush_rd.max()   # reads 256 MiB: replaces the dirty lines with clean ones

    def step(evs=None):
        # the GPU idles ~2 ms (outside every timed bracket) while the host
        # enqueues the whole step, so no call's bracket waits on the host
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        for i, (_, fn, _, _) in enumerate(hp.calls):
            flush_l2()
            if evs is not None:
                evs[2 * i].record(stream)
            fn()
            if evs is not None:
                evs[2 * i + 1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(hp.status.item()) != 0:
        raise RuntimeError(f"device status {q.status_string(int(hp.status.item()))} in warm-up")
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    all_evs = []
    for _ in range(args.steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * ncalls)]
        step(evs)
        all_evs.append(evs)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    per_call = [0.0] * ncalls
    total = 0.0
    for evs in all_evs:
        for i in range(ncalls):
            ms = evs[2 * i].elapsed_time(evs[2 * i + 1])
            per_call[i] += ms
            total += ms
    red = max_over_ranks(per_call + [total], world, dev)
    per_call, total = red[:-1], red[-1]

    # end to end through the public API: pinned host A in, int8 result out
    c = hp.int8
    A_host = c.A.pin_memory()
    out_host = torch.empty((c.M, c.N), dtype=torch.int8).pin_memory()
    A_dev = torch.empty_like(hp.A)
    e2e_times = []
    for i in range(args.warmup + args.steps):
        flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        A_dev.copy_(A_host, non_blocking=True)
        q.int8_gemm(A_dev, c.a_type, c.zA, hp.packed, hp.col_sum, c.N, c.b_type, c.zB, "s8",
                    bias=hp.bias, s_x=hp.s_x, s_w=hp.s_w, s_y=c.s_y, zp_y=c.zp_y, out=hp.out8,
                    workspace=hp.ws8, dev_status=hp.status, b16=hp.b16)
        out_host.copy_(hp.out8, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_times.append(e0.elapsed_time(e1))
    e2e_ms = max_over_ranks([sum(e2e_times)], world, dev)[0] / args.steps
    if int(hp.status.item()) != 0:
        raise RuntimeError(f"device status {q.status_string(int(hp.status.item()))}")
    streams = run_gemv_streams(hp, q, args, dev, stream)
    if int(hp.status.item()) != 0:
        raise RuntimeError(f"device status {q.status_string(int(hp.status.item()))}")
    streams["w8"] = run_w8(q, I, args, dev, stream, hp.status, flush_l2)
    if int(hp.status.item()) != 0:
        raise RuntimeError(f"device status {q.status_string(int(hp.status.item()))}")
    streams["axis"] = run_axis_zp(q, hp, args, dev, stream, hp.status, flush_l2)
    if int(hp.status.item()) != 0:
        raise RuntimeError(f"device status {q.status_string(int(hp.status.item()))}")
    streams["q8"] = run_q8(q, I, args, dev, stream, hp.status, flush_l2)
    if int(hp.status.item()) != 0:
        raise RuntimeError(f"device status {q.status_string(int(hp.status.item()))}")
    streams["int8_small"] = run_int8_small(q, I, args, dev, stream, hp.status, flush_l2)
    alone, _ = _timer(args, stream, flush_l2)
    c8 = hp.int8
    us_w = alone(hp.run_int8_widen_each_call)
    streams["int8_gemm_m4096_widen_each_call"] = {
        "us": us_w, "TOPS": 2.0 * c8.M * c8.N * c8.K / (us_w * 1e-6) / 1e12,
        "note": "the step's int8 GEMM through qmm_int8_gemm: the packed weights widened again on every call "
                "(the step's call reads the f16 copy qmm_widen_b_int8 made once)"}
    streams["q4_small_batch"] = run_q4_small_batch(q, hp, args, dev, stream, hp.status)
    streams["probe"] = run_probe(q, args, dev, stream, hp.status)
    if int(hp.status.item()) != 0:
        raise RuntimeError(f"device status {q.status_string(int(hp.status.item()))}")
    return hp, per_call, total, clk, e2e_ms, streams


def run_gemv_streams(hp, q, args, dev, stream):
    """M=1 GEMV weight bandwidth on back-to-back launches, the way decode runs
    them: every launch streams weights that are cold in L2 because the launches
    cycle through rotating copies of the weights totalling >= 4x the L2 size.
      * lm_head: R copies of its 97 MB tile set, one launch per copy per pass;
      * the 7 projections: C copies of the set, all C x 7 launches captured in
        one CUDA graph, replayed once per pass.
    Each pass is timed with CUDA events; the per-launch (per-set) time is the
    pass time over R (C).  Returns medians over `args.steps` passes."""
    import math
    import statistics
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    name, K, N, tiles, x1, _, y1, _ = hp.q4[0]
    R = max(2, math.ceil(4 * l2 / tiles.numel()))
    lm_copies = [tiles] + [tiles.clone() for _ in range(R - 1)]
    proj = hp.q4[1:]
    set_bytes = sum(t.numel() for (_, _, _, t, _, _, _, _) in proj)
    C = max(2, math.ceil(4 * l2 / set_bytes))
    proj_copies = [[t if c == 0 else t.clone() for (_, _, _, t, _, _, _, _) in proj] for c in range(C)]

    def lm_pass():
        for t in lm_copies:
            q.q4_gemm(t, N, K, x1, Y=y1, dev_status=hp.status)

    def proj_pass():
        for cp in proj_copies:
            for t, (_, Kp, Np, _, xp, _, yp, _) in zip(cp, proj):
                q.q4_gemm(t, Np, Kp, xp, Y=yp, dev_status=hp.status)

    group_lists = [[(t, Np, Kp, xp, yp) for t, (_, Kp, Np, _, xp, _, yp, _) in zip(cp, proj)]
                   for cp in proj_copies]

    def group_pass():
        for gl in group_lists:
            q.q4_gemv_group(gl, dev_status=hp.status)

    proj_pass()                      # one-time per-device setup outside the capture
    group_pass()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        proj_pass()
    ggraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ggraph):
        group_pass()
    torch.cuda.synchronize()

    def timed(fn, n):
        out = []
        for i in range(args.warmup + n):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(HOST_LEAD_CYCLES)   # the host enqueues the pass ahead of the GPU
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                out.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) * 1e3 for a, b in out]

    lm_us = [t / R for t in timed(lm_pass, args.steps)]
    set_us = [t / C for t in timed(graph.replay, args.steps)]
    grp_us = [t / C for t in timed(ggraph.replay, args.steps)]
    del graph, ggraph, lm_copies, proj_copies, group_lists
    torch.cuda.synchronize()
    lm_med, set_med, grp_med = statistics.median(lm_us), statistics.median(set_us), statistics.median(grp_us)
    set_all_bytes = set_bytes + sum(2 * k + 4 * n for (_, k, n, _, _, _, _, _) in proj)
    return {
        "lm_head": {"us": lm_med, "copies": R, "weight_bytes": tiles.numel(),
                    "weight_GBs": tiles.numel() / (lm_med * 1e-6) / 1e9,
                    "GBs": (tiles.numel() + 2 * K + 4 * N) / (lm_med * 1e-6) / 1e9,
                    "launches_per_pass": R},
        "projection_set": {"us": set_med, "copies": C, "weight_bytes": set_bytes,
                           "weight_GBs": set_bytes / (set_med * 1e-6) / 1e9,
                           "GBs": (set_bytes + sum(2 * k + 4 * n for (_, k, n, _, _, _, _, _) in proj))
                                  / (set_med * 1e-6) / 1e9,
                           "launches_per_pass": 7 * C},
        "projection_set_group": {"us": grp_med, "copies": C, "weight_bytes": set_bytes,
                                 "weight_GBs": set_bytes / (grp_med * 1e-6) / 1e9,
                                 "GBs": set_all_bytes / (grp_med * 1e-6) / 1e9,
                                 "launches_per_pass": C},
        "l2_bytes": l2,
    }


def run_w8(q, I, args, dev, stream, status, flush_l2):
    """W8A16 (int8 weights, an fp32 scale for every 1,024 weights of a row, bf16
    activations), timed apart from the step:
      * lm_head M=1 decode GEMV, back-to-back launches over rotating copies of
        the codes totalling >= 4x the L2 size (as for the q4 GEMV);
      * the tensor-core route (codes widened to bf16, then the pair GEMM) on
        M=4096 K=N=4608 and on lm_head M=512, one call after an L2 flush.
    Medians over `args.steps` timed repetitions after `args.warmup`."""
    import math
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def timed(fn, flush):
        out = []
        for i in range(args.warmup + args.steps):
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            if flush:
                flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                out.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) * 1e3 for a, b in out)

    res = {}
    name, K, N = I.QWEN3_06B_LM_HEAD
    W = I.q4_weights(9 * 1000 + N % 997 + K, N, K).to(dev)
    codes, scales = q.pack_w8(W)
    del W
    wbytes = codes.numel() + scales.numel() * 4
    x1 = I.q4_activations(9 * 7919 + 1, 1, K).to(dev)
    y1 = torch.empty((1, N), dtype=torch.float32, device=dev)
    R = max(2, math.ceil(4 * l2 / wbytes))
    copies = [(codes, scales)] + [(codes.clone(), scales.clone()) for _ in range(R - 1)]

    def lm_pass():
        for c, sc in copies:
            q.w8_gemm(c, sc, N, K, x1, Y=y1, dev_status=status)

    us = timed(lm_pass, False) / R
    res["w8_gemv_lm_head_m1_stream"] = {"us": us, "copies": R, "launches": 1, "weight_bytes": wbytes,
                                       "weight_GBs": wbytes / (us * 1e-6) / 1e9,
                                       "GBs": (wbytes + 2 * K + 4 * N) / (us * 1e-6) / 1e9}
    del copies
    us = timed(lambda: q.w8_gemm(codes, scales, N, K, x1, Y=y1, dev_status=status), True)
    res["w8_gemv_lm_head_m1"] = {"us": us, "launches": 1, "weight_bytes": wbytes,
                                "weight_GBs": wbytes / (us * 1e-6) / 1e9,
                                "GBs": (wbytes + 2 * K + 4 * N) / (us * 1e-6) / 1e9}
    x512 = I.q4_activations(9 * 7919 + 512, 512, K).to(dev)
    y512 = torch.empty((512, N), dtype=torch.float32, device=dev)
    ws = torch.empty(q.w8_gemm_workspace_size(512, K, N), dtype=torch.uint8, device=dev)
    us = timed(lambda: q.w8_gemm(codes, scales, N, K, x512, Y=y512, workspace=ws, dev_status=status), True)
    res["w8_gemm_lm_head_m512"] = {"us": us, "launches": 2, "TFLOPS": 2 * 512 * N * K / (us * 1e-6) / 1e12,
                                   "weight_bytes": wbytes}
    del codes, scales, ws, y512, x512
    M, Kb, Nb = 4096, 4608, 4608
    W = I.q4_weights(4608, Nb, Kb).to(dev)
    codes, scales = q.pack_w8(W)
    del W
    X = I.q4_activations(4096, M, Kb).to(dev)
    Y = torch.empty((M, Nb), dtype=torch.float32, device=dev)
    ws = torch.empty(q.w8_gemm_workspace_size(M, Kb, Nb), dtype=torch.uint8, device=dev)
    us = timed(lambda: q.w8_gemm(codes, scales, Nb, Kb, X, Y=Y, workspace=ws, dev_status=status), True)
    res["w8_gemm_m4096"] = {"us": us, "launches": 2, "TFLOPS": 2 * M * Nb * Kb / (us * 1e-6) / 1e12,
                            "shape": f"M={M} K={Kb} N={Nb}"}
    del codes, scales, ws, X, Y
    torch.cuda.synchronize()
    return res


def run_q8(q, I, args, dev, stream, status, flush_l2):
    """Q8 tiles (the two 8-bit code layouts of the Q4NX chunk format), timed
    apart from the step like the W8A16 path:
      * lm_head M=1 decode GEMV in each layout, back-to-back launches over
        rotating copies of the tiles totalling >= 4x the L2 size;
      * lm_head M=512 through the tensor-core route (tiles decoded to f16,
        activation rows to scaled f16, then the pair GEMM), one call after an
        L2 flush.
    Medians over `args.steps` timed repetitions after `args.warmup`."""
    import math
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def timed(fn, flush):
        out = []
        for i in range(args.warmup + args.steps):
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            if flush:
                flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                out.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) * 1e3 for a, b in out)

    res = {}
    name, K, N = I.QWEN3_06B_LM_HEAD
    W = I.q4_weights(9 * 1000 + N % 997 + K, N, K).to(dev)
    x1 = I.q4_activations(9 * 7919 + 1, 1, K).to(dev)
    y1 = torch.empty((1, N), dtype=torch.float32, device=dev)
    for layout in (q.QMM_Q8_LAYOUT_KR, q.QMM_Q8_LAYOUT_SLAB16):
        tiles = q.pack_q8(W, layout)
        wbytes = tiles.numel()
        R = max(2, math.ceil(4 * l2 / wbytes))
        copies = [tiles] + [tiles.clone() for _ in range(R - 1)]

        def lm_pass():
            for t in copies:
                q.q8_gemm(t, layout, N, K, x1, Y=y1, dev_status=status)

        us = timed(lm_pass, False) / R
        res[f"q8_gemv_lm_head_m1_layout{layout}_stream"] = {
            "us": us, "copies": R, "launches": 1, "weight_bytes": wbytes,
            "weight_GBs": wbytes / (us * 1e-6) / 1e9, "GBs": (wbytes + 2 * K + 4 * N) / (us * 1e-6) / 1e9}
        del copies
        if layout == q.QMM_Q8_LAYOUT_KR:
            x512 = I.q4_activations(9 * 7919 + 512, 512, K).to(dev)
            y512 = torch.empty((512, N), dtype=torch.float32, device=dev)
            ws = torch.empty(q.q8_gemm_workspace_size(512, K, N), dtype=torch.uint8, device=dev)
            us = timed(lambda: q.q8_gemm(tiles, layout, N, K, x512, Y=y512, workspace=ws, dev_status=status), True)
            res["q8_gemm_lm_head_m512"] = {"us": us, "launches": 3,
                                           "TFLOPS": 2 * 512 * N * K / (us * 1e-6) / 1e12, "weight_bytes": wbytes}
            del x512, y512, ws
        del tiles
    del W
    torch.cuda.synchronize()
    return res


def _timer(args, stream, flush_l2):
    """Two ways to time a call: `alone(fn)` flushes L2 before each call and
    brackets it with CUDA events on the launching stream; `passes(fn, n)` runs
    a pass of n back-to-back launches after a ~2 ms host lead and divides.
    Both return the median over `args.steps` timed repetitions after
    `args.warmup`, in microseconds."""
    import torch

    def run(fn, flush):
        out = []
        for i in range(args.warmup + args.steps):
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            if flush:
                flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                out.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) * 1e3 for a, b in out)

    return (lambda fn: run(fn, True)), (lambda fn, n: run(fn, False) / n)


def run_probe(q, args, dev, stream, status):
    """Load-only HBM read bandwidth (qmm_probe_hbm_read) over rotating 128 MiB
    buffers totalling >= 4x L2, back to back, in both read styles the GEMVs
    use.  The larger of the two is the load-only roofline."""
    import math
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nb = 128 << 20
    R = max(4, math.ceil(4 * l2 / nb))
    bufs = [torch.ones(nb, dtype=torch.uint8, device=dev) for _ in range(R)]
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    _, passes = _timer(args, stream, None)
    res = {}
    for mode, name in ((0, "ld128"), (1, "bulk")):
        us = passes(lambda: [q.probe_hbm_read(b, mode, sink, status) for b in bufs], R)
        res[name] = {"us_per_buffer": us, "GBs": nb / (us * 1e-6) / 1e9}
    res["buffers"] = R
    res["buffer_bytes"] = nb
    res["GBs"] = max(res["ld128"]["GBs"], res["bulk"]["GBs"])
    del bufs
    torch.cuda.synchronize()
    return res


def run_int8_small(q, I, args, dev, stream, status, flush_l2):
    """The two small int8 workloads, timed apart from the step:
      * M=16 K=N=1024 (uint8 x int8, zA = 128 +- 8): int32 out and fp32 out,
        each one call after an L2 flush, and back to back over rotating copies
        of the packed weights (>= 4x L2, every launch reads them from HBM),
        captured in one CUDA graph;
      * the seven Qwen3-0.6B projections at M=32 (int8 per-tensor activations x
        packB weights, fp32 out): each alone after a flush, and the set of
        seven launches captured in one CUDA graph over rotating weight copies;
      * a mid-size M=128 K=N=4608 GEMM (the step's operands, first 128 rows),
        one call after a flush.
    TOPS = 2MNK / time; weight GB/s = packed weight bytes / time."""
    import math
    import torch
    alone, passes = _timer(args, stream, flush_l2)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}
    c = I.int8_gemm_small()
    A = c.A.to(dev)
    packed, _, col_sum = q.pack_b_int8(c.B.to(dev), c.b_type)
    s_w = c.s_w.to(dev)
    wb = packed.numel()
    outs = {"s32": torch.empty((c.M, c.N), dtype=torch.int32, device=dev),
            "f32": torch.empty((c.M, c.N), dtype=torch.float32, device=dev)}
    R = max(2, math.ceil(4 * l2 / wb))
    copies = [packed] + [packed.clone() for _ in range(R - 1)]
    for ot in ("s32", "f32"):
        sw = s_w if ot == "f32" else None
        call = lambda pk=packed, ot=ot, sw=sw: q.int8_gemm(A, c.a_type, c.zA, pk, col_sum, c.N, c.b_type, c.zB, ot,
                                                          s_w=sw, out=outs[ot], dev_status=status)
        us = alone(call)
        call(copies[0])
        torch.cuda.synchronize()
        g1 = torch.cuda.CUDAGraph()   # back to back without host launch gaps
        with torch.cuda.graph(g1):
            for pk in copies:
                call(pk)
        torch.cuda.synchronize()
        us_s = passes(g1.replay, R)
        del g1
        ops = 2.0 * c.M * c.N * c.K
        res[f"int8_m16_k1024_n1024_{ot}"] = {
            "us": us, "TOPS": ops / (us * 1e-6) / 1e12, "weight_GBs": wb / (us * 1e-6) / 1e9, "launches": 1,
            "stream": {"us": us_s, "copies": R, "TOPS": ops / (us_s * 1e-6) / 1e12,
                       "weight_GBs": wb / (us_s * 1e-6) / 1e9}}
    del copies
    # the projection set at M = 32
    projs = []
    for idx in range(7):
        cc = I.int8_qwen_projection(idx)
        pk, cs, cols = q.pack_b_int8(cc.B.to(dev), cc.b_type)
        projs.append((cc, cc.A.to(dev), pk, cs, cols, torch.tensor([cc.s_x], dtype=torch.float32, device=dev),
                      torch.empty((cc.M, cc.N), dtype=torch.float32, device=dev)))
    set_bytes = sum(p[2].numel() for p in projs)
    set_ops = sum(2.0 * p[0].M * p[0].N * p[0].K for p in projs)
    shapes = {}
    for cc, Ad, pk, cs, cols, sx, Y in projs:
        call = lambda cc=cc, Ad=Ad, pk=pk, cs=cs, cols=cols, sx=sx, Y=Y: q.int8_gemm(
            Ad, cc.a_type, cc.zA, pk, cols, cc.N, cc.b_type, cc.zB, "f32", s_x=sx, s_w=cs, out=Y, dev_status=status)
        us = alone(call)
        shapes[cc.name] = {"us": us, "K": cc.K, "N": cc.N, "TOPS": 2.0 * cc.M * cc.N * cc.K / (us * 1e-6) / 1e12,
                           "weight_GBs": pk.numel() / (us * 1e-6) / 1e9}
    C = max(2, math.ceil(4 * l2 / set_bytes))
    pcopies = [[p[2] if k == 0 else p[2].clone() for p in projs] for k in range(C)]

    def set_pass():
        for cp in pcopies:
            for pk, (cc, Ad, _, cs, cols, sx, Y) in zip(cp, projs):
                q.int8_gemm(Ad, cc.a_type, cc.zA, pk, cols, cc.N, cc.b_type, cc.zB, "f32", s_x=sx, s_w=cs, out=Y,
                            dev_status=status)

    group_lists = [[dict(A=Ad, a_type=cc.a_type, zA=cc.zA, packed=pk, col_sum=cols, N=cc.N, b_orig_type=cc.b_type,
                         zB=cc.zB, out_type="f32", s_x=sx, s_w=cs, out=Y)
                    for pk, (cc, Ad, _, cs, cols, sx, Y) in zip(cp, projs)] for cp in pcopies]

    def group_pass():
        for gl in group_lists:
            q.int8_gemm_group(gl, dev_status=status)

    set_pass()
    group_pass()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        set_pass()
    ggraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ggraph):
        group_pass()
    torch.cuda.synchronize()
    us_set = passes(graph.replay, C)
    us_grp = passes(ggraph.replay, C)
    res["int8_qwen3_projections_m32"] = {
        "per_shape": shapes,
        "graph": {"us_per_set": us_set, "copies": C, "launches_per_set": 7, "weight_bytes": set_bytes,
                  "TOPS": set_ops / (us_set * 1e-6) / 1e12, "weight_GBs": set_bytes / (us_set * 1e-6) / 1e9},
        "group_graph": {"us_per_set": us_grp, "copies": C, "launches_per_set": 1, "weight_bytes": set_bytes,
                        "TOPS": set_ops / (us_grp * 1e-6) / 1e12, "weight_GBs": set_bytes / (us_grp * 1e-6) / 1e9,
                        "note": "the seven projections as one qmm_int8_gemm_group launch per set"}}
    del graph, ggraph, pcopies, group_lists
    # mid-size M
    cl = I.int8_gemm_large()
    M = 128
    A128 = cl.A[:M].to(dev)
    pkl, _, csl = q.pack_b_int8(cl.B.to(dev), cl.b_type)
    out = torch.empty((M, cl.N), dtype=torch.int8, device=dev)
    bias, swl = cl.bias.to(dev), cl.s_w.to(dev)
    sxl = torch.tensor([cl.s_x], dtype=torch.float32, device=dev)
    us = alone(lambda: q.int8_gemm(A128, cl.a_type, cl.zA, pkl, csl, cl.N, cl.b_type, cl.zB, "s8", bias=bias,
                                   s_x=sxl, s_w=swl, s_y=cl.s_y, zp_y=cl.zp_y, out=out, dev_status=status))
    res["int8_m128_k4608_n4608"] = {"us": us, "TOPS": 2.0 * M * cl.N * cl.K / (us * 1e-6) / 1e12,
                                    "weight_GBs": pkl.numel() / (us * 1e-6) / 1e9, "launches": 1}
    torch.cuda.synchronize()
    return res


def run_q4_small_batch(q, hp, args, dev, stream, status):
    """q4 decode GEMV at M = 2, 8, 16 (lm_head), back to back over rotating
    weight copies totalling >= 4x L2, like the M = 1 measurement."""
    import math
    import torch
    _, passes = _timer(args, stream, None)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    name, K, N, tiles, _, x512, _, _ = hp.q4[0]
    R = max(2, math.ceil(4 * l2 / tiles.numel()))
    copies = [tiles] + [tiles.clone() for _ in range(R - 1)]
    res = {}
    for M in (2, 8, 16):
        X = x512[:M].contiguous()
        Y = torch.empty((M, N), dtype=torch.float32, device=dev)
        us = passes(lambda: [q.q4_gemm(t, N, K, X, Y=Y, dev_status=status) for t in copies], R)
        wb = tiles.numel()
        res[f"q4_gemv_lm_head_m{M}_stream"] = {"us": us, "copies": R, "weight_bytes": wb,
                                               "weight_GBs": wb / (us * 1e-6) / 1e9,
                                               "GBs": (wb + 2 * M * K + 4 * M * N) / (us * 1e-6) / 1e9,
                                               "TFLOPS": 2.0 * M * N * K / (us * 1e-6) / 1e12}
    del copies
    torch.cuda.synchronize()
    return res


def run_axis_zp(q, hp, args, dev, stream, status, flush_l2):
    """The int8 GEMM with per-axis zero points (one per row of A, one per
    column of B) on the step's M=4096 K=N=4608 operands, int8 out, one call
    after an L2 flush; median over `args.steps` after `args.warmup`."""
    import torch
    c = hp.int8
    g = torch.Generator().manual_seed(4096)
    zA = torch.randint(0, 256, (c.M,), generator=g, dtype=torch.int32).to(dev)
    zB = torch.randint(-8, 9, (c.N,), generator=g, dtype=torch.int32).to(dev)
    ws = torch.empty(q.int8_gemm_axis_zp_workspace_size(c.M, c.K, c.N), dtype=torch.uint8, device=dev)
    out = torch.empty((c.M, c.N), dtype=torch.int8, device=dev)
    times = []
    for i in range(args.warmup + args.steps):
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        q.int8_gemm_axis_zp(hp.A, c.a_type, zA, hp.packed, hp.col_sum, c.N, c.b_type, zB, "s8", bias=hp.bias,
                            s_x=hp.s_x, s_w=hp.s_w, s_y=c.s_y, zp_y=c.zp_y, out=out, workspace=ws,
                            dev_status=status)
        e1.record(stream)
        if i >= args.warmup:
            times.append((e0, e1))
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in times)
    return {"int8_gemm_axis_zp_m4096": {"us": us, "launches": 4, "TOPS": 2.0 * c.M * c.N * c.K / (us * 1e-6) / 1e12,
                                        "shape": f"M={c.M} K={c.K} N={c.N}, zero point per row of A and per column of B"}}


def _cpu_int8_rows(rows):
    """The oracle (as it stands) on the given rows of the M=4096 K=N=4608 GEMM;
    returns (int ops, seconds of oracle work)."""
    import numpy as np
    import oracle.qmm_oracle as O
    from quantized_matmul_qmm_gb300 import inputs as I
    c = I.int8_gemm_large()
    A = c.A[rows[0]:rows[1]].numpy().astype(np.int64)
    B = c.B.numpy().astype(np.int64)
    t0 = time.perf_counter()
    r = O.int8_gemm_y(A, c.a_type, c.zA, B, c.b_type, c.zB)
    O.int8_epilogue(r["Y"], "s8", c.bias.numpy(), c.s_x, c.s_w.numpy(), c.s_y, c.zp_y)
    return 2.0 * (rows[1] - rows[0]) * c.N * c.K, time.perf_counter() - t0


def _cpu_q4_rows(rows):
    """The oracle's q4 product for `rows` output rows of an lm_head-shaped
    weight (K=1024) at M=1; returns (weight bytes covered, seconds)."""
    import numpy as np
    import oracle.qmm_oracle as O
    from quantized_matmul_qmm_gb300 import inputs as I
    name, K, N = I.QWEN3_06B_LM_HEAD
    W = I.q4_weights(9 * 1000 + N % 997 + K, rows, K).numpy()   # a rows x K slice of the same distribution
    x = I.q4_activations(9 * 7919 + 1, 1, K).float().double().numpy()
    tiles = O.pack_q4(W)
    t0 = time.perf_counter()
    O.q4_gemm(tiles, rows, K, x)
    return tiles.size, time.perf_counter() - t0


def cpu_host():
    """Host cores and CPU model of this machine."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.TimeoutExpired):
        pass
    return cores, model


def cpu_baseline(rows_per_core: int, single_rows: int):
    """The CPU oracle as it stands, on this machine's host cores: one thread on
    `single_rows` rows of the int8 GEMM, then one process per core (spawned,
    so no CUDA state is inherited) on `rows_per_core` rows each, timed by the
    wall clock around the whole batch; and the q4 lm_head product on a sample
    of 4,096 output rows per core the same way."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    cores, model = cpu_host()
    ops1, dt1 = _cpu_int8_rows((0, single_rows))
    ctx = mp.get_context("spawn")
    with ProcessPoolExecutor(max_workers=cores, mp_context=ctx) as ex:
        # a first round warms the workers (imports, input generation)
        list(ex.map(_cpu_int8_rows, [(0, 1)] * cores))
        t0 = time.perf_counter()
        res = list(ex.map(_cpu_int8_rows, [(i * rows_per_core, (i + 1) * rows_per_core) for i in range(cores)]))
        wall = time.perf_counter() - t0
        ops = sum(r[0] for r in res)
        list(ex.map(_cpu_q4_rows, [32] * cores))
        t0 = time.perf_counter()
        q4 = list(ex.map(_cpu_q4_rows, [4096] * cores))
        q4_wall = time.perf_counter() - t0
    q4_bytes = sum(r[0] for r in q4)
    return {"value": ops / wall / 1e12, "unit": "TOPS", "cores": cores, "kind": "oracle",
            "cpu_model": model,
            "sample": f"{rows_per_core} rows of the M=4096 K=N=4608 int8 GEMM per core, one process per core, "
                      f"{cores * rows_per_core} rows in {wall:.1f} s wall (numpy int64)",
            "single_thread": {"value": ops1 / dt1 / 1e12, "unit": "TOPS", "cores": 1,
                              "sample": f"{single_rows} rows in {dt1:.1f} s"},
            "q4_gemv": {"value": q4_bytes / q4_wall / 1e9, "unit": "GB/s of q4 weights", "cores": cores,
                        "sample": f"lm_head-shaped q4 product at M=1 (K=1024), 4,096 output rows per core, "
                                  f"{cores * 4096} rows in {q4_wall:.1f} s wall (numpy fp64 decode-then-dense)"}}


def run_config(world):
    """The workload description both arms print."""
    return {"workload": WORKLOAD, "int8": f"u8xs8 M={INT8_M} K={INT8_K} N={INT8_N} int8 out",
            "l2": "flushed before every timed call (256 MiB write, then 256 MiB read); decode GEMVs "
                  "back to back over rotating weight copies >= 4x L2",
            "parallelism": f"replicas x{world}"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["qmm", "reference"], default="qmm")
    ap.add_argument("--cpu-rows", type=int, default=2, help="rows per host core of the oracle's CPU sample")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # the CPU oracle as the reference arm: rank 0 alone; each step is a
        # bounded sample of the int8 GEMM, one row per host core, one process
        # per core
        if rank != 0:
            return
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        cores, model = cpu_host()
        with ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as ex:
            for _ in range(args.warmup):
                list(ex.map(_cpu_int8_rows, [(i, i + 1) for i in range(cores)]))
            ops, secs = 0.0, 0.0
            for st in range(args.steps):
                t0 = time.perf_counter()
                res = list(ex.map(_cpu_int8_rows, [((st * cores + i) % INT8_M, (st * cores + i) % INT8_M + 1)
                                                   for i in range(cores)]))
                secs += time.perf_counter() - t0
                ops += sum(r[0] for r in res)
        value = ops / secs / 1e12
        sample = (f"{cores} of the 4096 rows of the M=4096 K=N=4608 int8 GEMM per step, one row per host core "
                  f"(one process each, numpy int64)")
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "int64", "data": "synthetic",
                "config": run_config(world),
                "cpu_baseline": {"value": value, "unit": "TOPS", "cores": cores, "kind": "oracle",
                                 "cpu_model": model, "sample": sample},
                "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hp, per_call, total, clk, e2e_ms, streams = run_ours(args, rank, world, dev)
    peaks, peak_kind = load_peaks()

    names = [c[0] for c in hp.calls]
    kern = {}
    for (name, _, launches, work), ms in zip(hp.calls, per_call):
        us = 1e3 * ms / args.steps
        d = {"us": round(us, 3), "launches": launches}
        if "ops" in work:
            d["TOPS"] = work["ops"] / (us * 1e-6) / 1e12
        if "flops" in work:
            d["TFLOPS"] = work["flops"] / (us * 1e-6) / 1e12
        if "weight_bytes" in work:
            d["weight_GBs"] = work["weight_bytes"] / (us * 1e-6) / 1e9
        d["GBs"] = work["bytes"] / (us * 1e-6) / 1e9
        kern[name] = d
    i8 = kern["int8_gemm_m4096"]
    tensor_peak = peaks["bf16_tflops"]
    hbm_peak = peaks["hbm_gbs"]
    traffic = load_traffic()
    value = replicas_rate(i8["TOPS"], world)
    lm = kern["q4_gemv_lm_head_m1"]
    st_lm, st_ps, st_pg = streams["lm_head"], streams["projection_set"], streams["projection_set_group"]
    probe = streams["probe"]
    roof = {"bound": "tensor", "achieved": i8["TOPS"], "peak": tensor_peak, "unit": "TFLOP/s",
            "frac": i8["TOPS"] / tensor_peak, "traffic": traffic.get("int8_gemm_m4096"),
            "kernel": "int8_gemm_m4096",
            "peak_source": f"{peak_kind} bf16 dense (the 16-bit tensor pipe the int8 GEMM runs on)"}
    rooflines = {}
    for name, d in kern.items():
        if name.startswith("int8_gemm") or (name.startswith("q4_gemm") and "m512" in name):
            ach = d.get("TOPS", d.get("TFLOPS"))
            rooflines[name] = {"bound": "tensor", "achieved": ach, "peak": tensor_peak, "unit": "TFLOP/s",
                               "frac": ach / tensor_peak, "traffic": traffic.get(name)}
        else:
            rooflines[name] = {"bound": "hbm", "achieved": d["GBs"], "peak": hbm_peak, "unit": "GB/s",
                               "frac": d["GBs"] / hbm_peak, "traffic": traffic.get(name)}
    rooflines["q4_gemv_lm_head_m1_stream"] = {"bound": "hbm", "achieved": st_lm["GBs"], "peak": hbm_peak,
                                              "unit": "GB/s", "frac": st_lm["GBs"] / hbm_peak,
                                              "traffic": traffic.get("q4_gemv_lm_head_m1")}
    rooflines["q4_gemv_projection_set_m1_graph"] = {"bound": "hbm", "achieved": st_ps["GBs"], "peak": hbm_peak,
                                                    "unit": "GB/s", "frac": st_ps["GBs"] / hbm_peak,
                                                    "traffic": None}
    rooflines["q4_gemv_projection_set_m1_group_graph"] = {
        "bound": "hbm", "achieved": st_pg["GBs"], "peak": hbm_peak, "unit": "GB/s", "frac": st_pg["GBs"] / hbm_peak,
        "traffic": traffic.get("q4_gemv_projection_set_m1_group_graph"), "note": "the 7 projections as one qmm_q4_gemv_group launch per set, sets in one CUDA graph"}
    w8 = streams["w8"]
    for name in ("w8_gemv_lm_head_m1_stream", "w8_gemv_lm_head_m1"):
        d = w8[name]
        rooflines[name] = {"bound": "hbm", "achieved": d["GBs"], "peak": hbm_peak, "unit": "GB/s",
                           "frac": d["GBs"] / hbm_peak, "traffic": traffic.get("w8_gemv_lm_head_m1")}
    for name in ("w8_gemm_lm_head_m512", "w8_gemm_m4096"):
        d = w8[name]
        rooflines[name] = {"bound": "tensor", "achieved": d["TFLOPS"], "peak": tensor_peak, "unit": "TFLOP/s",
                           "frac": d["TFLOPS"] / tensor_peak, "traffic": traffic.get(name)}
    for name, d in streams["axis"].items():
        rooflines[name] = {"bound": "tensor", "achieved": d["TOPS"], "peak": tensor_peak, "unit": "TFLOP/s",
                           "frac": d["TOPS"] / tensor_peak, "traffic": traffic.get(name)}
    q8 = streams["q8"]
    for name, d in q8.items():
        if "gemv" in name:
            rooflines[name] = {"bound": "hbm", "achieved": d["GBs"], "peak": hbm_peak, "unit": "GB/s",
                               "frac": d["GBs"] / hbm_peak, "traffic": traffic.get(name)}
        else:
            rooflines[name] = {"bound": "tensor", "achieved": d["TFLOPS"], "peak": tensor_peak, "unit": "TFLOP/s",
                               "frac": d["TFLOPS"] / tensor_peak, "traffic": traffic.get(name)}
    for name, d in rooflines.items():
        if d["bound"] == "hbm":
            d["peak_probe"] = probe["GBs"]
            d["frac_probe"] = d["achieved"] / probe["GBs"]
    small = streams["int8_small"]
    for name in ("int8_m16_k1024_n1024_s32", "int8_m16_k1024_n1024_f32"):
        d = small[name]["stream"]
        rooflines[name + "_stream"] = {"bound": "hbm", "achieved": d["weight_GBs"], "peak": hbm_peak, "unit": "GB/s",
                                       "frac": d["weight_GBs"] / hbm_peak, "peak_probe": probe["GBs"],
                                       "frac_probe": d["weight_GBs"] / probe["GBs"], "traffic": None,
                                       "note": "weight bytes only; back to back over rotating copies"}
    pg = small["int8_qwen3_projections_m32"]["graph"]
    rooflines["int8_qwen3_projections_m32_graph"] = {
        "bound": "hbm", "achieved": pg["weight_GBs"], "peak": hbm_peak, "unit": "GB/s",
        "frac": pg["weight_GBs"] / hbm_peak, "peak_probe": probe["GBs"], "frac_probe": pg["weight_GBs"] / probe["GBs"],
        "traffic": None, "note": "weight bytes only; 7 launches per set in one CUDA graph, rotating copies"}
    pgg = small["int8_qwen3_projections_m32"]["group_graph"]
    rooflines["int8_qwen3_projections_m32_group_graph"] = {
        "bound": "hbm", "achieved": pgg["weight_GBs"], "peak": hbm_peak, "unit": "GB/s",
        "frac": pgg["weight_GBs"] / hbm_peak, "peak_probe": probe["GBs"], "frac_probe": pgg["weight_GBs"] / probe["GBs"],
        "traffic": traffic.get("int8_qwen3_projections_m32_group_graph"), "note": "weight bytes only; one grouped launch per set in one CUDA graph, rotating copies"}
    for name, d in streams["q4_small_batch"].items():
        rooflines[name] = {"bound": "hbm", "achieved": d["GBs"], "peak": hbm_peak, "unit": "GB/s",
                           "frac": d["GBs"] / hbm_peak, "peak_probe": probe["GBs"],
                           "frac_probe": d["GBs"] / probe["GBs"], "traffic": traffic.get(name)}
    c = hp.int8
    launches = sum(l for (_, _, l, _) in hp.calls) * args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": run_config(world),
        "roofline": roof,
        "rooflines": rooflines,
        "gemv": {"value": replicas_rate(st_lm["weight_GBs"], world), "unit": "GB/s", "kernel": "q4_gemv_lm_head_m1",
                 "frac_hbm": st_lm["GBs"] / hbm_peak, "peak_source": peak_kind,
                 "frac_probe": st_lm["GBs"] / probe["GBs"], "probe_GBs": probe["GBs"],
                 "method": f"lm_head M=1, back-to-back launches over {st_lm['copies']} rotating weight copies "
                           f"(>= 4x the {streams['l2_bytes'] >> 20} MiB L2), median over passes",
                 "projection_set_graph": {"weight_GBs": world * st_ps["weight_GBs"],
                                          "frac_hbm": st_ps["GBs"] / hbm_peak, "frac_probe": st_ps["GBs"] / probe["GBs"],
                                          "us_per_set": st_ps["us"], "copies": st_ps["copies"],
                                          "launches_per_set": 7},
                 "projection_set_group_graph": {"weight_GBs": world * st_pg["weight_GBs"],
                                                "frac_hbm": st_pg["GBs"] / hbm_peak,
                                                "frac_probe": st_pg["GBs"] / probe["GBs"],
                                                "us_per_set": st_pg["us"], "copies": st_pg["copies"],
                                                "launches_per_set": 1},
                 "single_call": {"weight_GBs": world * lm["weight_GBs"], "frac_hbm": lm["GBs"] / hbm_peak,
                                 "us": lm["us"], "note": "one launch timed alone after an L2 flush"}},
        "kernels": kern,
        "w8a16": {"note": "int8 weights with an fp32 scale for every 1,024 weights of a row, bf16 activations; "
                          "timed apart from the step (median, L2 flushed before each single call)",
                  **w8},
        "int8_axis_zp": {"note": "per-axis zero points: the exact GEMM to int32 in the workspace, row sums, "
                                 "then one correction + output pass; timed apart from the step", **streams["axis"]},
        "q8": {"note": "8-bit tiles (bf16 scale per row and 32 columns) in the chunk format's two code layouts; "
                       "timed apart from the step (median, L2 flushed before each single call)",
               **q8},
        "hbm_probe": {"note": "load-only reads of rotating 128 MiB buffers (>= 4x L2), back to back; the larger "
                              "of the two read styles is the load-only roofline (peak_probe)", **probe},
        "int8_small": {"note": "the M=16 and M=32 int8 workloads and a mid-size M=128 GEMM, timed apart from the step",
                       **small},
        "int8_gemm_m4096_widen_each_call": streams["int8_gemm_m4096_widen_each_call"],
        "q4_small_batch": {"note": "q4 decode GEMV at M = 2, 8, 16 on lm_head, back to back over rotating weight copies",
                           **streams["q4_small_batch"]},
        "e2e": {"value": replicas_rate(2.0 * c.M * c.N * c.K / (e2e_ms * 1e-3) / 1e12, world), "unit": "TOPS",
                "h2d_bytes_per_step": c.M * c.K, "d2h_bytes_per_step": c.M * c.N},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.cpu_rows, 4)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

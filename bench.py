#!/usr/bin/env python
"""Benchmark of the dense fp32 GEMM and packed 2-bit GEMV / skinny GEMM path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mm|reference]

Prints ONE JSON line (rank 0).  One step is one pass of the whole hot path:
  0. the GPT-2-small MLP up-projection at 64 tokens, 64 x 768 x 3072 fp32 NN,
     one mm_gemm_f32 call with L2 flushed before it;
  1. square 2048^3 fp32 GEMM in the NN, NT and TN layouts (L2 flushed first
     by writing a 512 MiB buffer, since the 48 MiB of operands fit in L2);
  2. the 2-bit 12,288 x 1,536 GEMV over a rotation of 64 distinct matrices
     (288 MiB of codes, larger than the 129 MB L2), back to back, twice: as 64
     independent calls (programmatic dependent launch, no call waits for the
     previous one) and as a dependent chain (call i+1 reads as its x the first
     3 KB that call i wrote, so it waits for call i before reading x; only its
     weight loads start early);
  3. the ternary 16-layer encoder block: 16 x (222x768 -> 3072, 222x3072 -> 768);
  4. the 4-bit 12,288 x 1,536 GEMV and the transposed 2-bit 1,536 x 12,288 GEMV,
     each over a 64-matrix rotation of independent calls;
  5. the training-shape set: 8192 x 8192 x 2048 forward and its two backward
     products, through the split entry point (automatic split, one workspace).
Each phase is captured once as a CUDA graph and replayed; every replay is timed
with CUDA events on the stream it runs on.  The headline value is the 2048^3
GEMM throughput (TFLOP/s); the GEMV weight bandwidth (GB/s: 4,718,592 bytes of
weights per call over the per-call time, the measure defined on the Kernel 0112
page, whose runs are batches of back-to-back dispatches) is reported beside it.

Multi-GPU (torchrun): every rank runs the same step on its own GPU with its own
inputs (replicas, weak scaling, no collective on the data path); times are
max-reduced over ranks and `value` counts the work of all ranks.

--impl reference times the CPU oracle (plain fp64 C triple loops) on the same
workload on this host's cores, on a bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import math
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "2048³ fp32 GEMM TFLOP/s; 2-bit 12288×1536 GEMV weight GB/s vs HBM peak"
GEMV_WEIGHT_BYTES = 12288 * 1536 // 4           # 4,718,592
GEMV_TOTAL_BYTES = GEMV_WEIGHT_BYTES + 12288 * 2 + 1536 * 2 + 12288 * 4
GEMV4_WEIGHT_BYTES = 12288 * 1536 // 2          # 9,437,184
GEMV4_TOTAL_BYTES = GEMV4_WEIGHT_BYTES + 12288 * 2 + 1536 * 2 + 12288 * 4
GEMVT_TOTAL_BYTES = GEMV_WEIGHT_BYTES + 1536 * 2 + 12288 * 2 + 1536 * 4   # 1536 x 12288: same weight bytes
GEMM_FLOP = 2.0 * 2048 ** 3
TRAIN_FLOP = 3 * 2.0 * 8192 * 8192 * 2048  # forward + the two backward products, 274.9 GFLOP each
MLP_M, MLP_N, MLP_K = 8192, 3072, 768  # GPT-2 small MLP up-projection, 8 x 1024 tokens
MLP_FLOP = 2.0 * MLP_M * MLP_N * MLP_K  # 38.7 GFLOP (the bias and GELU are O(MN), not counted)
C1_M, C1_N, C1_K = 64, 3072, 768  # GPT-2 small MLP up-projection at 64 tokens, one call
C1_FLOP = 2.0 * C1_M * C1_N * C1_K  # 302 MFLOP
C1_BYTES = 4 * (C1_M * C1_K + C1_K * C1_N + C1_M * C1_N)  # 10.42 MB: A and B read once, C written
C1_CALLS = 8  # distinct problems per step, one mm_gemm_f32 call each, all cold after the L2 flush
TERN_FLOP_PER_LAYER = 2 * (2.0 * 222 * 3072 * 768)
ATTN_HEADS, ATTN_T, ATTN_D = 32, 512, 64  # causal self-attention, B = 4 x H = 8 heads
# algorithmic flops of a forward + backward: the forward's S = Q K^T and O = P V, the backward's
# dV, dP, dQ, dK, each 2 D flops per allowed (query, key) pair (T (T + 1) / 2 of them, causal)
ATTN_FLOP = 6 * 2.0 * ATTN_HEADS * (ATTN_T * (ATTN_T + 1) // 2) * ATTN_D
N_GEMV = 64
GEMV_B_LAUNCHES = 8  # the rotation as this many back-to-back strided-batched launches per step
# each launch writes its own y and reads nothing another writes, so it is launched independent
# (programmatic dependent launch without the wait): the next launch's CTAs take the SMs that the
# current one's last CTAs leave idle; measured, 4 launches: 0.957 -> 0.927 us per matrix (74 -> 76%
# of HBM), 8 launches: 0.945 -> 0.911 (75 -> 78%)
GEMV_B_OPTS = dict(dequant=6, pdl=1, independent=1)
N_LAYERS = 16
WORKLOAD = ("gpt2_mlp_up_64x768x3072_fp32_nn + square_2048_fp32_gemm_nn_nt_tn + gemv2bit_12288x1536_rotation64 + "
            "ternary_encoder_16x(222x768x3072,222x3072x768) + gemv4bit_12288x1536_rotation64 + "
            "gemv2bit_1536x12288_rotation64 + training_set_8192x2048x8192_fwd_dA_dB")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["mm", "reference"], default="mm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gemm-path", type=int, default=0)
    return ap.parse_args(argv)


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend):
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
    return rank, world


def reduce_max(value: float, device=None) -> float:
    """Max of `value` over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def rank_replica(rank: int) -> int:
    """Each rank draws its own inputs (weak scaling): rank r runs replica r of every workload,
    whose random streams share no draw with any other replica's."""
    from dense_packed_bit_gb300 import synth
    if not 0 <= rank < synth.MAX_REPLICAS:
        raise ValueError(f"rank {rank}: the input recipes hold {synth.MAX_REPLICAS} replicas")
    return rank


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() in ("active", "1", "0x1"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- peaks

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


def fp32_simt_peak_tflops(sms: int, mhz: float) -> float:
    # 128 FP32 lanes per SM, 2 flop per FMA
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def traffic_for(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it still matches the source."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if not parts or parts[0].startswith("#") or parts[0] != kernel_key:
            continue
        src = os.path.join(ROOT, parts[1])
        if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != parts[2]:
            return None
        return int(parts[3])
    return None


# ---------------------------------------------------------------- workload

class Workload:
    def __init__(self, device, rank, args):
        import torch
        from dense_packed_bit_gb300 import synth
        self.dev = device
        rep = rank_replica(rank)
        # SHA-256 of every workload's inputs as drawn (codes, scales, activations, operands), so
        # that a change of the inputs shows in the report
        sha = {k: synth.Digest() for k in ("gpt2_mlp_up_64", "square_2048", "gemv2_rotation64", "gemv4_rotation64",
                                           "gemv2_t_rotation64", "ternary_encoder", "training_set",
                                           "gpt2_mlp_bias_gelu", "gpt2_attention")}
        self.c1 = []
        for j in range(C1_CALLS):
            c1 = synth.gpt2_mlp_up_64x768x3072(replica=rep * C1_CALLS + j)
            assert (c1.M, c1.N, c1.K) == (C1_M, C1_N, C1_K)
            sha["gpt2_mlp_up_64"].update(c1.A, c1.B)
            self.c1.append(dict(case=c1, A=torch.from_numpy(c1.A).to(device), B=torch.from_numpy(c1.B).to(device),
                                C=torch.empty((C1_M, C1_N), dtype=torch.float32, device=device)))
        self.gemm = []
        for layout in ("nn", "nt", "tn"):
            c = synth.square_2048(layout, replica=rep)
            A, B = c.A, c.B
            sha["square_2048"].update(A, B)
            self.gemm.append(dict(case=c, layout=layout, A=torch.from_numpy(A).to(device),
                                  B=torch.from_numpy(B).to(device),
                                  C=torch.empty((c.M, c.N), dtype=torch.float32, device=device),
                                  C_ffma=torch.empty((c.M, c.N), dtype=torch.float32, device=device),
                                  hA=A, hB=B))
        import dense_packed_bit_gb300 as mm
        # the FFMA phase runs through the split entry point: its stream-K tail's workspace
        self.ffma_ws_floats = mm.mm_gemm_f32_splitk_workspace_ex(2048, 2048, 2048, 0, path=mm.MM_GEMM_FFMA)
        self.ffma_ws = torch.empty(max(self.ffma_ws_floats, 4), dtype=torch.float32, device=device)
        # the rotation as one contiguous [64, 12288, 384] buffer: the per-call phases take views,
        # the batched phase the whole buffer
        self.gemv_codes_all = torch.empty((N_GEMV, 12288, 384), dtype=torch.uint8, device=device)
        self.gemv_scales_all = torch.empty((N_GEMV, 12288), dtype=torch.int16, device=device)
        self.gemv_codes, self.gemv_scales = [], []
        x = None
        for i in range(N_GEMV):
            c = synth.gemv_2bit_12288x1536(i, replica=rep)
            sha["gemv2_rotation64"].update(c.codes, c.scales)
            self.gemv_codes_all[i].copy_(torch.from_numpy(c.codes))
            self.gemv_scales_all[i].copy_(torch.from_numpy(c.scales.view("int16")))
            self.gemv_codes.append(self.gemv_codes_all[i])
            self.gemv_scales.append(self.gemv_scales_all[i])
            x = c.X
            self.gemv_cb = c.codebook
        self.gemv_yb = torch.empty((GEMV_B_LAUNCHES, N_GEMV, 12288), dtype=torch.float32, device=device)
        sha["gemv2_rotation64"].update(x)
        self.gemv_x = torch.from_numpy(x.reshape(-1)).to(device)
        self.gemv_y = torch.empty((N_GEMV, 12288), dtype=torch.float32, device=device)
        self.gemv_yc = torch.zeros((N_GEMV, 12288), dtype=torch.float32, device=device)  # the chain's outputs
        self.gemv4_codes, self.gemv4_scales = [], []
        for i in range(N_GEMV):
            c = synth.gemv_4bit_12288x1536(i, replica=rep)
            sha["gemv4_rotation64"].update(c.codes, c.scales)
            self.gemv4_codes.append(torch.from_numpy(c.codes).to(device))
            self.gemv4_scales.append(torch.from_numpy(c.scales).to(device))
            x4 = c.X
            self.gemv4_cb = c.codebook
        sha["gemv4_rotation64"].update(x4)
        self.gemv4_x = torch.from_numpy(x4.reshape(-1)).to(device)
        self.gemv4_y = torch.empty((N_GEMV, 12288), dtype=torch.float32, device=device)
        self.gemvt_codes, self.gemvt_scales = [], []
        for i in range(N_GEMV):
            c = synth.gemv_2bit_1536x12288(i, replica=rep)
            sha["gemv2_t_rotation64"].update(c.codes, c.scales)
            self.gemvt_codes.append(torch.from_numpy(c.codes).to(device))
            self.gemvt_scales.append(torch.from_numpy(c.scales).to(device))
            xt = c.X
        sha["gemv2_t_rotation64"].update(xt)
        self.gemvt_x = torch.from_numpy(xt.reshape(-1)).to(device)
        self.gemvt_y = torch.empty((N_GEMV, 1536), dtype=torch.float32, device=device)
        self.tern = []
        for layer in range(N_LAYERS):
            for proj in ("up", "down"):
                c = synth.ternary_encoder_layer(layer, proj, replica=rep)
                sha["ternary_encoder"].update(c.codes, c.scales, c.X)
                self.tern.append(dict(case=c, codes=torch.from_numpy(c.codes).to(device),
                                      scales=torch.from_numpy(c.scales).to(device),
                                      X=torch.from_numpy(c.X).to(device),
                                      Y=torch.empty((c.X.shape[0], c.rows), dtype=torch.float32, device=device)))
        at = synth.gpt2_attention_4x8x512x64(replica=rep)
        assert (at.heads, at.T, at.D) == (ATTN_HEADS, ATTN_T, ATTN_D)
        sha["gpt2_attention"].update(at.Q, at.K, at.V, at.dO)
        self.attn = dict(case=at, **{n: torch.from_numpy(getattr(at, n)).to(device) for n in ("Q", "K", "V", "dO")},
                         **{n: torch.empty((ATTN_HEADS, ATTN_T, ATTN_D), dtype=torch.float32, device=device)
                            for n in ("O", "dQ", "dK", "dV")},
                         L=torch.empty((ATTN_HEADS, ATTN_T), dtype=torch.float32, device=device))
        # training-shape set: forward C = A B, dA = dC B^T, dB = A^T dC (N(0, 0.02)), through the
        # split entry point with its automatic choice and one shared workspace
        self.train = list(synth.training_set_8192_all(replica=rep))
        sha["training_set"].update(self.train[0].A, self.train[0].B, self.train[1].A)  # A, B, dC
        tA = torch.from_numpy(self.train[0].A).to(device)
        tB = torch.from_numpy(self.train[0].B).to(device)
        tdC = torch.from_numpy(self.train[1].A).to(device)
        import dense_packed_bit_gb300 as mm
        self.train_ops = []
        need = 0
        for c, (a, b) in zip(self.train, ((tA, tB), (tdC, tB), (tA, tdC))):
            out = torch.empty((c.M, c.N), dtype=torch.float32, device=device)
            self.train_ops.append((c, a, b, out))
            need = max(need, mm.mm_gemm_f32_splitk_workspace(c.M, c.N, c.K, 0))
        self.train_ws = torch.empty(max(need, 4), dtype=torch.float32, device=device)
        self.train_ws_floats = need
        # GPT-2 small's MLP up-projection with its bias and GELU fused, 8 sequences of 1024 tokens
        mlp = synth.gpt2_mlp_bias_gelu_8192x768x3072(replica=rep)
        sha["gpt2_mlp_bias_gelu"].update(mlp.A, mlp.B, mlp.bias)
        self.inputs_sha256 = {k: d.hexdigest() for k, d in sha.items()}
        assert (mlp.M, mlp.N, mlp.K) == (MLP_M, MLP_N, MLP_K)
        self.mlp_case = mlp
        self.mlp_x = torch.from_numpy(mlp.A).to(device)
        self.mlp_w = torch.from_numpy(mlp.B).to(device)
        self.mlp_b = torch.from_numpy(mlp.bias).to(device)
        self.mlp_y = torch.empty((MLP_M, MLP_N), dtype=torch.float32, device=device)
        self.mlp_ws_floats = mm.mm_gemm_f32_splitk_workspace(MLP_M, MLP_N, MLP_K, 0)
        self.mlp_ws = torch.empty(max(self.mlp_ws_floats, 4), dtype=torch.float32, device=device)
        self.flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
        self.args = args


# independent calls: the fp4 tensor-core decode, 15 tiles of 127 rows per CTA (7 CTAs per call, ~20 calls
# in flight over four streams); measured 1.31 us per call against 1.38 for the staged SIMT decode
GEMV_INDEP = dict(dequant=6, rows_per_lane=15, pdl=1, independent=1)
GEMV_CHAINED = dict(dequant=2, staging=1, rows_per_lane=1, pdl=1, weights_static=1)
GEMV_INDEP_STREAMS = 4  # independent calls rotate over four streams inside the graph
GEMV4_INDEP = dict(staging=1, blocks=1, pdl=1, independent=1)
# the transposed 1536 x 12288 shape (13 tiles of 127 rows, 48 stages each): the fp4 decode, three
# tiles per CTA (5 CTAs per call), over four streams; measured 1.66 us per call against 1.87 for the
# automatic (SIMT affine) decode
GEMVT_INDEP = dict(dequant=6, rows_per_lane=3, pdl=1, independent=1)
# encoder layers run as a dependent chain: each product waits for the previous kernel before
# reading X or writing Y; its weights are loaded and decoded before that wait
TERN_OPTS = dict(pdl=1, weights_static=1)


def capture_phases(w: Workload, stream):
    """CUDA graphs of each phase (launch-bound loops replay without host launch cost).

    gemm   : the three 2048^3 products (NN, NT, TN)
    gemv   : the 64-matrix rotation as independent calls (no call reads another's output;
             each kernel skips the wait on its predecessor and overlaps it completely),
             alternating between two streams so that two launch queues feed the GPU
    gemv_c : the same rotation as a dependent chain (each call waits for the previous
             kernel before reading x, only its weight loads start early)
    tern   : the 16-layer ternary encoder block (32 skinny GEMMs)
    gemv4  : the 64-matrix rotation of 4-bit matrices as independent calls over two streams
    """
    import torch
    import dense_packed_bit_gb300 as mm
    a = w.args

    def gemm():
        for g in w.gemm:
            c = g["case"]
            mm.mm_gemm_f32_ex(c.transA, c.transB, c.M, c.N, c.K, g["A"], g["A"].shape[1], g["B"],
                              g["B"].shape[1], g["C"], c.N, path=a.gemm_path)

    def gemm_ffma():
        # the same three products on the FFMA path (the TMA-staged register-blocked kernel), with
        # its stream-K tail (the automatic split of mm_gemm_f32_splitk_ex for this path)
        for g in w.gemm:
            c = g["case"]
            mm.mm_gemm_f32_splitk_ex(c.transA, c.transB, c.M, c.N, c.K, g["A"], g["A"].shape[1], g["B"],
                                     g["B"].shape[1], g["C_ffma"], c.N, 0, w.ffma_ws, w.ffma_ws_floats,
                                     path=mm.MM_GEMM_FFMA)

    side = torch.cuda.Stream(device=stream.device)
    sides = [side] + [torch.cuda.Stream(device=stream.device) for _ in range(GEMV_INDEP_STREAMS - 2)]

    def gemv(opts, nstreams=1):
        def f():
            cur = torch.cuda.current_stream()
            sts = [cur] + sides[:nstreams - 1]
            for s in sts[1:]:
                s.wait_stream(cur)
            for i in range(N_GEMV):
                mm.mm_gemv_packed2_ex(w.gemv_codes[i], w.gemv_scales[i], w.gemv_x, w.gemv_y[i], 12288, 1536,
                                      w.gemv_cb, sts[i % len(sts)], **opts)
            for s in sts[1:]:
                cur.wait_stream(s)
        return f

    def gemv_chain():
        # a dependent chain: call 0 reads the workload's x, call i+1 reads as its 1,536 fp16
        # activations the first 3,072 bytes (768 fp32 outputs) that call i wrote
        for i in range(N_GEMV):
            x = w.gemv_x if i == 0 else w.gemv_yc[i - 1][:768].view(torch.int16)
            mm.mm_gemv_packed2_ex(w.gemv_codes[i], w.gemv_scales[i], x, w.gemv_yc[i], 12288, 1536, w.gemv_cb,
                                  **GEMV_CHAINED)

    def c1():
        for g in w.c1:
            mm.mm_gemm_f32(0, 0, C1_M, C1_N, C1_K, g["A"], C1_K, g["B"], C1_N, g["C"], C1_N)

    def gemv_batched():
        for j in range(GEMV_B_LAUNCHES):
            mm.mm_gemv_packed2_strided_batched_ex(w.gemv_codes_all, 12288 * 384, w.gemv_scales_all, 12288, w.gemv_x, 0,
                                                  w.gemv_yb[j], 12288, N_GEMV, 12288, 1536, w.gemv_cb, **GEMV_B_OPTS)

    def gemv4():
        cur = torch.cuda.current_stream()
        side.wait_stream(cur)
        for i in range(N_GEMV):
            st = side if i % 2 else cur
            mm.mm_gemv_packed4_ex(w.gemv4_codes[i], w.gemv4_scales[i], w.gemv4_x, w.gemv4_y[i], 12288, 1536,
                                  w.gemv4_cb, st, **GEMV4_INDEP)
        cur.wait_stream(side)

    def gemvt():
        cur = torch.cuda.current_stream()
        sts = [cur] + sides[:GEMV_INDEP_STREAMS - 1]
        for s in sts[1:]:
            s.wait_stream(cur)
        for i in range(N_GEMV):
            mm.mm_gemv_packed2_ex(w.gemvt_codes[i], w.gemvt_scales[i], w.gemvt_x, w.gemvt_y[i], 1536, 12288,
                                  w.gemv_cb, sts[i % len(sts)], **GEMVT_INDEP)
        for s in sts[1:]:
            cur.wait_stream(s)

    def train():
        for c, a, b, out in w.train_ops:
            mm.mm_gemm_f32_splitk(c.transA, c.transB, c.M, c.N, c.K, a, a.shape[1], b, b.shape[1], out, c.N, 0,
                                  w.train_ws, w.train_ws_floats)

    def attn():
        a = w.attn
        scale = 1.0 / math.sqrt(ATTN_D)
        mm.mm_attention_fwd(a["Q"], a["K"], a["V"], a["O"], a["L"], ATTN_HEADS, ATTN_T, ATTN_D, 1, scale)
        mm.mm_attention_bwd(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["L"], a["dQ"], a["dK"], a["dV"], ATTN_HEADS,
                            ATTN_T, ATTN_D, 1, scale)

    def mlp():
        mm.mm_gemm_f32_bias_act_splitk(0, 0, MLP_M, MLP_N, MLP_K, w.mlp_x, MLP_K, w.mlp_w, MLP_N, w.mlp_b,
                                       mm.MM_ACT_GELU_TANH, w.mlp_y, MLP_N, 0, w.mlp_ws, w.mlp_ws_floats)

    def tern():
        for t in w.tern:
            c = t["case"]
            mm.mm_gemm_packed2_ex(t["codes"], t["scales"], t["X"], t["Y"], c.X.shape[0], c.rows, c.cols, c.codebook,
                                  **TERN_OPTS)

    graphs = {}
    for name, fn in (("c1", c1), ("gemm", gemm), ("gemm_ffma", gemm_ffma), ("gemv", gemv(GEMV_INDEP, GEMV_INDEP_STREAMS)), ("gemv_c", gemv_chain),
                     ("tern", tern), ("gemv4", gemv4), ("gemvt", gemvt), ("train", train), ("mlp", mlp),
                     ("gemv_b", gemv_batched), ("attn", attn)):
        with torch.cuda.stream(stream):
            fn()  # warm the kernels' one-time setup outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs[name] = g
    return graphs


LAUNCHES_PER_STEP = C1_CALLS + 3 + 3 + 4 * N_GEMV + 2 * N_LAYERS + 3 + 1 + GEMV_B_LAUNCHES + 3  # C1, 2048^3, GEMVs, encoder, training set, MLP, batched, attention


PHASES = ("c1", "gemm", "gemm_ffma", "gemv", "gemv_c", "tern", "gemv4", "gemvt", "train", "mlp", "gemv_b", "attn")
L2_COLD = ("c1", "gemm", "gemm_ffma", "attn")  # phases whose operands fit in L2: a 512 MiB write evicts them first


def run_step(w: Workload, graphs, ev, stream):
    """One pass of the hot path; ev maps each phase to a (start, end) event pair."""
    for name in PHASES:
        if name in L2_COLD:
            w.flush.fill_(1.0)  # evict the operands from L2 (torch kernel, outside the events)
        ev[name][0].record(stream)
        graphs[name].replay()
        ev[name][1].record(stream)


def new_events():
    import torch
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    return {name: mk() for name in PHASES}


def e2e_gemm(w: Workload, steps: int, stream):
    """2048^3 GEMMs through the C ABI with host buffers: H2D of A and B from pinned
    memory, the three GEMMs, D2H of C, all inside the timed region.

    The copies run on their own streams, so that the inputs of the next product cross
    while the current one computes and its C comes back during the next: each product
    has its own device buffers, and events order every copy after the last use of the
    buffer it overwrites (a product's H2D after the previous step's GEMM of that product
    has read A and B; its GEMM after its H2D and after the previous step's D2H of C)."""
    import torch
    import dense_packed_bit_gb300 as mm
    host = []
    for g in w.gemm:
        hA = torch.from_numpy(g["hA"]).pin_memory()
        hB = torch.from_numpy(g["hB"]).pin_memory()
        hC = torch.empty(g["C"].shape, dtype=torch.float32).pin_memory()
        host.append((hA, hB, hC))
    h2d = sum(a.numel() * 4 + b.numel() * 4 for a, b, _ in host)
    d2h = sum(c.numel() * 4 for _, _, c in host)
    up = torch.cuda.Stream(device=stream.device)
    down = torch.cuda.Stream(device=stream.device)
    n = len(w.gemm)
    ev = {k: [torch.cuda.Event() for _ in range(n)] for k in ("in", "gemm", "out")}
    started = [False] * n

    def once():
        for j, (g, (hA, hB, hC)) in enumerate(zip(w.gemm, host)):
            c = g["case"]
            with torch.cuda.stream(up):
                if started[j]:
                    up.wait_event(ev["gemm"][j])  # the previous GEMM of this product has read A, B
                g["A"].copy_(hA, non_blocking=True)
                g["B"].copy_(hB, non_blocking=True)
                ev["in"][j].record(up)
            stream.wait_event(ev["in"][j])
            if started[j]:
                stream.wait_event(ev["out"][j])  # the previous C of this product has left
            mm.mm_gemm_f32(c.transA, c.transB, c.M, c.N, c.K, g["A"], g["A"].shape[1], g["B"], g["B"].shape[1],
                           g["C"], c.N, stream)
            ev["gemm"][j].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev["gemm"][j])
                hC.copy_(g["C"], non_blocking=True)
                ev["out"][j].record(down)
            started[j] = True

    with torch.cuda.stream(stream):
        once()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            once()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    return {"value": 3 * GEMM_FLOP * steps / dt / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "H2D, GEMMs and D2H on three streams: a product's inputs cross while the previous one computes"}


# ---------------------------------------------------------------- CPU oracle baseline

CPU_SAMPLE_MAX_PRODUCTS = 15  # the oracle's timed sample: at most 5 rounds of NN, NT, TN
PARITY_TOL = 1e-5  # |C - C_exact| <= 1e-5 * sum_k |a_ik b_kj|, the bound of every GEMM parity test


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and v.strip():
                return v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip() in ("model name", "Model") and v.strip():
                    return v.strip()
    except OSError:
        pass
    import platform
    return platform.machine() or "unknown"


def phase_stats(times_ms) -> dict:
    """Mean, median, min and max of one phase's per-step times (ms)."""
    t = sorted(float(x) for x in times_ms)
    if not t:
        return {}
    return {"ms_mean": sum(t) / len(t), "ms_median": statistics.median(t), "ms_min": t[0], "ms_max": t[-1]}


def parity_ratio(got, ref, T) -> float:
    """max over outputs of |got - ref| / T, with T = sum_k |term_k| per output (inf for a
    non-finite output, or for an error where T = 0)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    T = np.asarray(T, dtype=np.float64)
    if got.shape != ref.shape or not np.all(np.isfinite(got)):
        return float("inf")
    err = np.abs(got - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(T > 0, err / T, np.where(err > 0, np.inf, 0.0))
    return float(r.max()) if r.size else 0.0


def cpu_oracle_sample(seconds_target: float = 15.0, gpu_gemm=None):
    """Time the fp64 oracle on the 2048^3 NN/NT/TN products (all host cores).

    gpu_gemm: None, or {layout: the GPU's C for that product, on the host}; each is then
    compared with the oracle's product, every output, and the worst |err| / sum|terms| is
    reported beside the timing."""
    import oracle
    from dense_packed_bit_gb300 import synth
    oracle.build()
    threads = oracle.default_threads()
    cases = [synth.square_2048(layout) for layout in ("nn", "nt", "tn")]  # drawn before timing
    flop = 0.0
    dt = 0.0  # time inside the oracle calls only (no input drawing, no parity comparison)
    n_done = 0
    parity = {}
    while True:
        for layout, c in zip(("nn", "nt", "tn"), cases):
            t0 = time.perf_counter()
            ref, T = oracle.gemm(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B, threads=threads)
            dt += time.perf_counter() - t0
            flop += GEMM_FLOP
            n_done += 1
            if gpu_gemm is not None and layout in gpu_gemm and layout not in parity:
                parity[layout] = parity_ratio(gpu_gemm[layout], ref, T)
        if dt > seconds_target or n_done >= CPU_SAMPLE_MAX_PRODUCTS:
            break
    # one core: the first 128 rows of the NN product
    c = cases[0]
    rows1 = min(128, c.M)
    t1 = time.perf_counter()
    oracle.gemm(c.transA, c.transB, rows1, c.N, c.K, c.A[:rows1], c.B, threads=1)
    dt1 = time.perf_counter() - t1
    out = {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"{n_done} full 2048^3 products (NN, NT, TN in turn), fp64 accumulation, "
                     f"{dt:.1f} s inside the oracle calls",
           "cpu_model": cpu_model(),
           "value_1thread": 2.0 * rows1 * c.N * c.K / dt1 / 1e12,
           "sample_1thread": f"the first {rows1} rows of the NN product on one core, {dt1:.2f} s"}
    if gpu_gemm is not None:
        out["parity"] = {"what": "max over all 2048^2 outputs of |C_gpu - C_oracle| / sum_k |a_ik b_kj|, "
                                 "the bench's own products (mm_gemm_f32, the last e2e step)",
                         "tol": PARITY_TOL, "square_2048": parity,
                         "ok": bool(parity) and all(v <= PARITY_TOL for v in parity.values())}
    return out


def _sample_coords(rng, M, N, n_lines=2, n_random=2000):
    """Whole first / last / random rows and columns plus random outputs of an M x N result."""
    rows = [0, M - 1] + [int(v) for v in rng.integers(0, M, n_lines)]
    cols = [0, N - 1] + [int(v) for v in rng.integers(0, N, n_lines)]
    ii = np.concatenate([np.repeat(rows, N), np.tile(np.arange(M), len(cols)), rng.integers(0, M, n_random)])
    jj = np.concatenate([np.tile(np.arange(N), len(rows)), np.repeat(cols, M), rng.integers(0, N, n_random)])
    return ii, jj


def bench_parity(w) -> dict:
    """The outputs the timed phases left on the GPU (the last replay of each), compared with the
    fp64 oracle on the host: worst |y - y_ref| / sum_k |term_k| per workload, against 1e-5.

    c1 (the first and last of its calls), gemv (64 independent calls), gemv_b (the batched launch), gemv4, gemv_t: every output.
    gemv_c (the dependent chain): call 0 on the workload's x, and each later call whose x, the
    bits of the previous call's first 768 outputs read as fp16, holds only finite values.
    ternary: every output of layers 0 and 15, 2,000 sampled outputs of the other products.
    training_set: 4 whole rows and 4 whole columns and 2,000 random outputs per product.
    gpt2_mlp_up (bias + GELU): the first and last 64 rows, against its own bound
    1.13e-5 T + 2^-20 (1 + |z|), reported as a fraction of that bound.
    """
    import oracle
    oracle.build()
    rng = np.random.default_rng(2026)
    out = {}
    t0 = time.perf_counter()
    worst, n = 0.0, 0
    for g in (w.c1[0], w.c1[-1]):
        c = g["case"]
        ref, T = oracle.gemm(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B)
        worst = max(worst, parity_ratio(g["C"].cpu().numpy(), ref, T))
        n += ref.size
    out["gpt2_mlp_up_64"] = {"worst": worst, "outputs": n, "problems": f"the first and last of the {C1_CALLS} calls"}

    codes = w.gemv_codes_all.cpu().numpy()
    scales = w.gemv_scales_all.cpu().numpy().view(np.uint16)
    x = w.gemv_x.cpu().numpy().view(np.uint16)
    y, yb, yc = w.gemv_y.cpu().numpy(), w.gemv_yb[-1].cpu().numpy(), w.gemv_yc.cpu().numpy()
    # the batched launches of a step compute the same rotation: every one must hold the same bits
    yb_all = w.gemv_yb.cpu().numpy()
    batched_same = bool(all(np.array_equal(yb_all[j].view(np.uint32), yb.view(np.uint32))
                            for j in range(GEMV_B_LAUNCHES)))
    worst = worst_b = 0.0
    chain_worst, chain_checked = 0.0, 0
    for i in range(N_GEMV):
        ref, T = oracle.packed_gemm(codes[i], scales[i], x, 12288, 1536, w.gemv_cb)
        worst = max(worst, parity_ratio(y[i], ref[0], T[0]))
        worst_b = max(worst_b, parity_ratio(yb[i], ref[0], T[0]))
        xi = x if i == 0 else yc[i - 1][:768].view(np.uint16)
        if i == 0:
            chain_worst, chain_checked = parity_ratio(yc[0], ref[0], T[0]), 1
        elif np.all(np.isfinite(xi.view(np.float16))):
            rc, Tc = oracle.packed_gemm(codes[i], scales[i], xi, 12288, 1536, w.gemv_cb)
            chain_worst = max(chain_worst, parity_ratio(yc[i], rc[0], Tc[0]))
            chain_checked += 1
    out["gemv2_rotation64"] = {"worst": worst, "outputs": N_GEMV * 12288}
    out["gemv2_batched"] = {"worst": worst_b if batched_same else float("inf"), "outputs": N_GEMV * 12288,
                            "launches_bit_identical": batched_same}
    out["gemv2_chain"] = {"worst": chain_worst, "calls_checked": chain_checked,
                          "note": "later calls read the previous call's fp32 bits as fp16; calls whose x "
                                  "holds inf or NaN patterns are not compared"}

    worst = 0.0
    x4 = w.gemv4_x.cpu().numpy().view(np.uint16)
    y4 = w.gemv4_y.cpu().numpy()
    for i in range(N_GEMV):
        ref, T = oracle.packed4_gemm(w.gemv4_codes[i].cpu().numpy(), w.gemv4_scales[i].cpu().numpy().view(np.uint16),
                                     x4, 12288, 1536, w.gemv4_cb)
        worst = max(worst, parity_ratio(y4[i], ref[0], T[0]))
    out["gemv4_rotation64"] = {"worst": worst, "outputs": N_GEMV * 12288}

    worst = 0.0
    xt = w.gemvt_x.cpu().numpy().view(np.uint16)
    yt = w.gemvt_y.cpu().numpy()
    for i in range(N_GEMV):
        ref, T = oracle.packed_gemm(w.gemvt_codes[i].cpu().numpy(), w.gemvt_scales[i].cpu().numpy().view(np.uint16),
                                    xt, 1536, 12288, w.gemv_cb)
        worst = max(worst, parity_ratio(yt[i], ref[0], T[0]))
    out["gemv2_t_rotation64"] = {"worst": worst, "outputs": N_GEMV * 1536}

    worst, n_out = 0.0, 0
    for j, t in enumerate(w.tern):
        c = t["case"]
        Y = t["Y"].cpu().numpy()
        if j // 2 in (0, N_LAYERS - 1):
            ref, T = oracle.packed_gemm(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
            worst = max(worst, parity_ratio(Y, ref, T))
            n_out += Y.size
        else:
            mi = rng.integers(0, Y.shape[0], 2000)
            ri = rng.integers(0, Y.shape[1], 2000)
            ref, T = oracle.packed_gemm_at(c.codes, c.scales, c.X, c.cols, c.codebook, mi, ri)
            worst = max(worst, parity_ratio(Y[mi, ri], ref, T))
            n_out += len(mi)
    out["ternary_encoder"] = {"worst": worst, "outputs": n_out}

    worst, n_out = 0.0, 0
    for c, _, _, o in w.train_ops:
        ii, jj = _sample_coords(rng, c.M, c.N)
        ref, T = oracle.gemm_at(c.transA, c.transB, c.K, c.A, c.B, ii, jj)
        C = o.cpu().numpy()
        worst = max(worst, parity_ratio(C[ii, jj], ref, T))
        n_out += len(ii)
    out["training_set"] = {"worst": worst, "outputs": n_out}

    worst, n_out = 0.0, 0
    for g in w.gemm:
        c = g["case"]
        ii, jj = _sample_coords(rng, c.M, c.N)
        ref, T = oracle.gemm_at(c.transA, c.transB, c.K, g["hA"], g["hB"], ii, jj)
        worst = max(worst, parity_ratio(g["C_ffma"].cpu().numpy()[ii, jj], ref, T))
        n_out += len(ii)
    out["square_2048_ffma"] = {"worst": worst, "outputs": n_out}

    # bias + GELU: its bound is 1.13e-5 T + 2^-20 (1 + |z|); the ratio is err / that bound, scaled by
    # 1e-5 so that it compares with the same tolerance as the others
    mlp = w.mlp_case
    Ym = w.mlp_y.cpu().numpy()
    worst = 0.0
    for r0 in (0, MLP_M - 64):
        ref, T, Z = oracle.gemm_bias_act(0, 0, 64, MLP_N, MLP_K, mlp.A[r0:r0 + 64], mlp.B, mlp.bias, 1)
        bound = 1.13 * T + 2.0 ** -20 * (1.0 + np.abs(Z)) / PARITY_TOL
        worst = max(worst, parity_ratio(Ym[r0:r0 + 64], ref, bound))
    out["gpt2_mlp_up_bias_gelu"] = {"worst": worst, "outputs": 128 * MLP_N,
                                    "note": "|err| / (1.13 T + 2^-20 (1 + |z|) / 1e-5)"}

    # attention: heads 0 and 31 in full, O, L and the three gradients, each against its bound scale
    # times the head's tolerance 1e-5 + 2 gamma_D A (the fp32 scores' rounding, passed on by the
    # softmax), reported as a fraction of 1e-5 like the others
    at = w.attn["case"]
    hs = [0, ATTN_HEADS - 1]
    scale = float(np.float32(1.0 / math.sqrt(ATTN_D)))
    Qa, Ka = np.abs(at.Q[hs].astype(np.float64)), np.abs(at.K[hs].astype(np.float64))
    A = scale * np.max(np.einsum("hid,hkd->hik", Qa, Ka), axis=(1, 2))
    tol = (1e-5 + 2.0 * ATTN_D * 2.0 ** -24 * A).reshape(-1, 1, 1)
    Or, Lr, TO = oracle.attention_fwd(at.Q[hs], at.K[hs], at.V[hs], at.causal, scale)
    rq, rk, rv, tq, tk, tv = oracle.attention_bwd(at.Q[hs], at.K[hs], at.V[hs], at.dO[hs], at.causal, scale)
    got = {n: w.attn[n].cpu().numpy()[hs] for n in ("O", "L", "dQ", "dK", "dV")}
    worst = 0.0
    for n, ref, T in (("O", Or, TO), ("dQ", rq, tq), ("dK", rk, tk), ("dV", rv, tv)):
        worst = max(worst, parity_ratio(got[n], ref, T * tol / PARITY_TOL))
    worst = max(worst, parity_ratio(got["L"], Lr, (1.0 + np.abs(Lr)) * tol[:, :, 0] / PARITY_TOL))
    out["gpt2_attention"] = {"worst": worst, "outputs": int(2 * ATTN_T * (4 * ATTN_D + 1)),
                             "note": "heads 0 and 31: |err| / (T (1e-5 + 2 gamma_D A) / 1e-5)"}
    ok = all(v["worst"] <= PARITY_TOL for v in out.values())
    return {"what": "max |y_gpu - y_oracle| / sum_k |term_k| over the outputs the timed phases left, per workload",
            "tol": PARITY_TOL, "ok": bool(ok), "workloads": out, "seconds": time.perf_counter() - t0}


# ---------------------------------------------------------------- main arms

def main_reference(args):
    rank, world, _ = dist_env()
    if world > 1:
        dist_init("gloo")
        if rank != 0:
            return 0
    import oracle
    from dense_packed_bit_gb300 import synth
    oracle.build()
    threads = oracle.default_threads()
    # bounded sample per step: the first 128 rows of each 2048^3 product
    rows = 128
    cases = [synth.square_2048(l) for l in ("nn", "nt", "tn")]
    # the sampled rows of op(A), cut out before timing
    row_A = [c.A[:, :rows].copy() if c.transA else c.A[:rows] for c in cases]

    def step():
        fl = 0.0
        for c, A in zip(cases, row_A):
            oracle.gemm(c.transA, c.transB, rows, c.N, c.K, A, c.B, threads=threads)
            fl += 2.0 * rows * c.N * c.K
        return fl

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += step()
    dt = time.perf_counter() - t0
    val = fl / dt / 1e12
    sample = f"first {rows} rows of each 2048^3 product (NN, NT, TN) per step, fp64 oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "square_2048_fp32_gemm_nn_nt_tn (row sample)", "rows_per_product": rows},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model()},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


def main_mm(args):
    import torch
    import dense_packed_bit_gb300 as mm
    from dense_packed_bit_gb300 import build as mmbuild

    rank, world, local = dist_env()
    if rank == 0:
        mmbuild.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    rank, world = dist_init("nccl")
    if world > 1:
        barrier(dev)
        mmbuild.build()  # other ranks pick up the library rank 0 built
    mm.load_library()

    w = Workload(dev, rank, args)
    stream = torch.cuda.Stream(device=dev)
    graphs = capture_phases(w, stream)
    ev_steps = [new_events() for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            run_step(w, graphs, new_events(), stream)
        mm.mm_check_device_error(stream)
        torch.cuda.synchronize()

        clocks = ClockSampler(dev.index)
        clocks.start()
        barrier(dev)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for s in range(args.steps):
            run_step(w, graphs, ev_steps[s], stream)
        torch.cuda.synchronize()
        barrier(dev)
        wall = time.perf_counter() - t0
        clk = clocks.stop()
        mm.mm_check_device_error(stream)

    def total_s(name):
        return reduce_max(sum(ev[name][0].elapsed_time(ev[name][1]) for ev in ev_steps) / 1e3, dev)

    # per-phase spread over the timed steps on this rank (the headline figures use the totals)
    phases = {name: phase_stats([ev[name][0].elapsed_time(ev[name][1]) for ev in ev_steps]) for name in PHASES}

    c1_total_s = total_s("c1")
    c1_call_s = c1_total_s / args.steps / C1_CALLS
    gemm_total_s = total_s("gemm")
    gemm_ffma_total_s = total_s("gemm_ffma")
    gemv_total_s = total_s("gemv")
    gemvc_total_s = total_s("gemv_c")
    tern_total_s = total_s("tern")
    gemv4_total_s = total_s("gemv4")
    gemvt_total_s = total_s("gemvt")
    train_total_s = total_s("train")
    mlp_total_s = total_s("mlp")
    gemvb_total_s = total_s("gemv_b")
    attn_total_s = total_s("attn")
    per_mat_gemvb_s = gemvb_total_s / (args.steps * GEMV_B_LAUNCHES * N_GEMV)
    wall = reduce_max(wall, dev)

    gemm_tflops = world * 3 * GEMM_FLOP * args.steps / gemm_total_s / 1e12
    per_call_gemv_s = gemv_total_s / (args.steps * N_GEMV)
    per_call_gemvc_s = gemvc_total_s / (args.steps * N_GEMV)
    gemv_gbs = world * GEMV_WEIGHT_BYTES / per_call_gemv_s / 1e9
    tern_tflops = world * N_LAYERS * TERN_FLOP_PER_LAYER * args.steps / tern_total_s / 1e12
    per_call_gemv4_s = gemv4_total_s / (args.steps * N_GEMV)
    per_call_gemvt_s = gemvt_total_s / (args.steps * N_GEMV)
    step_ms = (c1_total_s + gemm_total_s + gemm_ffma_total_s + gemv_total_s + gemvc_total_s + tern_total_s + gemv4_total_s + gemvt_total_s +
               train_total_s + mlp_total_s + gemvb_total_s + attn_total_s) / args.steps * 1e3

    peaks, peaks_src = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    fp32_peak_max = fp32_simt_peak_tflops(sms, peaks.get("sm_max_mhz", 2070.0))
    gemm_per_gpu = 3 * GEMM_FLOP * args.steps / gemm_total_s / 1e12
    if args.gemm_path in (mm.MM_GEMM_AUTO, mm.MM_GEMM_TF32X3):
        # three tf32 MMAs per fp32 multiply-add: the fp32-equivalent tensor peak is a third of tf32's
        tf32_peak = peaks["bf16_tflops"] * (1.1 / 2.25)
        roof = {"bound": "tensor", "achieved": gemm_per_gpu, "peak": tf32_peak / 3.0, "unit": "TFLOP/s",
                "frac": gemm_per_gpu / (tf32_peak / 3.0), "traffic": traffic_for("gemm_tf32x3_ws"),
                "kernel": "gemm_tf32x3_ws_kernel",
                "peak_source": (f"{peaks_src} bf16 burst {peaks['bf16_tflops']:.0f} TFLOP/s x nominal tf32/bf16 "
                                f"ratio 1.1/2.25, divided by the 3 MMAs of the split"),
                "frac_of_fp32_simt_peak": gemm_per_gpu / fp32_peak_max}
        if clk.get("sm_mhz"):
            # the tensor peak scales with the SM clock: the measured bf16 burst ran at the clock
            # MEASURED_PEAKS records under load, this kernel at the clock sampled during the run
            ref_mhz = peaks.get("clocks_under_load", {}).get("sm_mhz_median") or peaks.get("sm_max_mhz", 2070.0)
            roof["frac_at_sampled_clock"] = gemm_per_gpu / (tf32_peak / 3.0 * clk["sm_mhz"] / ref_mhz)
            roof["sampled_clock_note"] = (f"peak rescaled from the {ref_mhz:.0f} MHz of the bf16 measurement to the "
                                          f"{clk['sm_mhz']:.0f} MHz sampled here")
        roof["ncu_tensor_active"] = "85.4% of cycles on the SMs holding a tile (profiles/gemm_tf32x3_ws_pair_square2048_nn.md)"
    else:
        roof = {"bound": "alu", "achieved": gemm_per_gpu, "peak": fp32_peak_max, "unit": "TFLOP/s",
                "frac": gemm_per_gpu / fp32_peak_max, "traffic": traffic_for("gemm_ffma"),
                "kernel": "gemm_ffma_kernel",
                "peak_source": f"{sms} SMs x 128 FP32 lanes x 2 flop x {peaks.get('sm_max_mhz', 2070.0):.0f} MHz"}
        if clk.get("sm_mhz"):
            roof["frac_at_sampled_clock"] = gemm_per_gpu / fp32_simt_peak_tflops(sms, clk["sm_mhz"])

    out = {
        "metric": METRIC, "value": gemm_tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "gpt2_mlp_up_64": "64x768x3072 fp32 NN, U[-1,1), one mm_gemm_f32 call per problem, 8 distinct problems per step",
                   "gemm": "2048x2048x2048 fp32 NN+NT+TN, N(0,0.02)",
                   "gemv": "12288x1536 2-bit, 64-matrix rotation (288 MiB > L2), codebook {-2,-1,0,1}",
                   "ternary": "16 layers, M=222, up 768->3072 and down 3072->768, a dependent chain with PDL",
                   "gemv_t": "1536x12288 2-bit, 64-matrix rotation (288 MiB > L2)",
                   "training_set": "8192x8192x2048 NN, dA=dC.B^T 8192x2048x8192, dB=A^T.dC 2048x8192x8192, N(0,0.02)",
                   "l2": "512 MiB buffer written before the 64x768x3072 and the 2048^3 phases of every step; "
                         "GEMV rotations exceed L2",
                   "gemv_opts": {"independent": GEMV_INDEP, "independent_streams": GEMV_INDEP_STREAMS,
                                 "chained": GEMV_CHAINED,
                                 "chain": "call i+1 reads as x the first 768 fp32 outputs of call i, as fp16 bits"},
                   "launch": "each phase replayed as a CUDA graph",
                   "gemm_path": args.gemm_path, "parallelism": f"replicas x{world}"},
        "gemm_ms_per_step": gemm_total_s / args.steps * 1e3,
        "square_2048_ffma": {"metric": "fp32 GEMM TFLOP/s, 2048^3 NN + NT + TN on the FFMA path "
                                       "(mm_gemm_f32_splitk_ex, MM_GEMM_FFMA, automatic split: TMA-staged 8x8 "
                                       "register blocks, packed f32x2 FMAs, stream-K tail)",
                             "workspace_floats": w.ffma_ws_floats,
                             "value": world * 3 * GEMM_FLOP * args.steps / gemm_ffma_total_s / 1e12, "unit": "TFLOP/s",
                             "us_per_product": gemm_ffma_total_s / args.steps / 3 * 1e6,
                             "roofline": {"bound": "alu", "kernel": "gemm_ffma_kernel",
                                          "achieved": 3 * GEMM_FLOP * args.steps / gemm_ffma_total_s / 1e12,
                                          "peak": fp32_peak_max, "unit": "TFLOP/s",
                                          "frac": 3 * GEMM_FLOP * args.steps / gemm_ffma_total_s / 1e12 / fp32_peak_max,
                                          "traffic": traffic_for("gemm_ffma"),
                                          "peak_source": f"{sms} SMs x 128 FP32 lanes x 2 flop x "
                                                         f"{peaks.get('sm_max_mhz', 2070.0):.0f} MHz",
                                          "note": "256 tiles of 128 x 128 at one CTA per SM are 1.68 waves on 152 "
                                                  "SMs: the first 152 tiles run whole, the k-steps of the other 104 "
                                                  "are cut evenly over 152 CTAs (stream-K tail), whose partial tiles "
                                                  "ffma_sk_reduce_kernel adds in K order"}},
        "gpt2_mlp_up_64": {"metric": "fp32 GEMM TFLOP/s, 64 x 768 x 3072 NN (one mm_gemm_f32 call, L2 flushed)",
                           "value": world * C1_FLOP / c1_call_s / 1e12, "unit": "TFLOP/s",
                           "us_per_call": c1_call_s * 1e6,
                           "calls": f"{C1_CALLS} distinct seeded problems per step, back to back in one graph "
                                    "after the L2 flush (every operand cold)",
                           "roofline": {"bound": "hbm", "kernel": "gemm_skinny_tc_kernel",
                                        "achieved": C1_BYTES / c1_call_s / 1e9,
                                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                        "frac": C1_BYTES / c1_call_s / 1e9 / peaks["hbm_gbs"],
                                        "traffic": traffic_for("gemm_skinny_tc"), "peak_source": peaks_src,
                                        "hbm_floor_us": C1_BYTES / peaks["hbm_gbs"] / 1e3,
                                        "fp32_floor_us": C1_FLOP / fp32_peak_max / 1e6,
                                        "frac_of_fp32_simt_peak": C1_FLOP / c1_call_s / 1e12 / fp32_peak_max,
                                        "note": "302 MFLOP over 10.42 MB (A, B read once, C written): 29 flop per "
                                                "byte, below the 3xTF32 ridge (316 TFLOP/s / 6.8 TB/s = 47), so "
                                                "HBM bounds the tensor-core kernel; a single cold 11 us call is "
                                                "latency-bound (DRAM latency of its first slabs, the cluster "
                                                "reduction), far from either floor"}},
        "gemv": {"metric": "2-bit 12288x1536 GEMV weight GB/s", "value": gemv_gbs, "unit": "GB/s",
                 "us_per_call": per_call_gemv_s * 1e6,
                 "mode": f"64 independent back-to-back calls over the rotation, {GEMV_INDEP_STREAMS} streams",
                 "kernel": "gemv2_mxf4_kernel (codes as packed e2m1 in tensor memory, x as 14 exact e2m1 digit "
                           "pieces, tcgen05.mma kind::mxf4), 15 tiles of 127 rows per CTA",
                 "chained": {"value": world * GEMV_WEIGHT_BYTES / per_call_gemvc_s / 1e9, "unit": "GB/s",
                             "us_per_call": per_call_gemvc_s * 1e6,
                             "mode": "each call waits for the previous kernel before reading x"},
                 "roofline": {"bound": "hbm", "achieved": GEMV_TOTAL_BYTES / per_call_gemv_s / 1e9,
                              "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": GEMV_TOTAL_BYTES / per_call_gemv_s / 1e9 / peaks["hbm_gbs"],
                              "weight_frac": GEMV_WEIGHT_BYTES / per_call_gemv_s / 1e9 / peaks["hbm_gbs"],
                              "traffic": traffic_for("gemv2_mxf4_single"), "peak_source": peaks_src},
                 "batched": {"value": world * GEMV_WEIGHT_BYTES / per_mat_gemvb_s / 1e9, "unit": "GB/s",
                             "us_per_matrix": per_mat_gemvb_s * 1e6,
                             "mode": f"the 64-matrix rotation (288 MiB) as one mm_gemv_packed2_strided_batched "
                                     f"launch, {GEMV_B_LAUNCHES} launches back to back per step, one shared x, each "
                                     f"into its own y, launched independent (programmatic dependent launch)",
                             "opts": GEMV_B_OPTS,
                             "kernel": "gemv2_mxf4_kernel (automatic: codes as packed e2m1 in tensor memory, x as "
                                       "14 exact e2m1 digit pieces, tcgen05.mma kind::mxf4)",
                             "roofline": {"bound": "hbm", "achieved": GEMV_TOTAL_BYTES / per_mat_gemvb_s / 1e9,
                                          "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                          "frac": GEMV_TOTAL_BYTES / per_mat_gemvb_s / 1e9 / peaks["hbm_gbs"],
                                          "weight_frac": GEMV_WEIGHT_BYTES / per_mat_gemvb_s / 1e9 / peaks["hbm_gbs"],
                                          "traffic": traffic_for("gemv2_mxf4_batched"), "peak_source": peaks_src}}},
        "gpt2_attention": {"metric": "causal attention forward + backward TFLOP/s (algorithmic), 32 heads x 512 x 64",
                           "value": world * ATTN_FLOP * args.steps / attn_total_s / 1e12, "unit": "TFLOP/s",
                           "us_per_step": attn_total_s / args.steps * 1e6,
                           "kernels": "attn_fwd_kernel, attn_bwd_dkdv_kernel, attn_bwd_dq_kernel (fp32 FFMA)",
                           "roofline": {"bound": "alu", "achieved": ATTN_FLOP * args.steps / attn_total_s / 1e12,
                                        "peak": fp32_peak_max, "unit": "TFLOP/s",
                                        "frac": ATTN_FLOP * args.steps / attn_total_s / 1e12 / fp32_peak_max,
                                        "traffic": traffic_for("attn_fwd"),
                                        "peak_source": f"{sms} SMs x 128 FP32 lanes x 2 flop x "
                                                       f"{peaks.get('sm_max_mhz', 2070.0):.0f} MHz",
                                        "note": "algorithmic flops: S, O forward, dV, dP, dQ, dK backward over the "
                                                "allowed (causal) pairs; the kernels also recompute S and dP for "
                                                "the dQ pass and compute the diagonal tiles in full"}},
        "ternary": {"value": tern_tflops, "unit": "TFLOP/s", "ms_per_block": tern_total_s / args.steps * 1e3,
                    "us_per_product": tern_total_s / args.steps / (2 * N_LAYERS) * 1e6,
                    "kernel": "gemm_packed2_tcr_kernel (automatic token tile and cluster split)", "opts": TERN_OPTS,
                    "roofline": {"bound": "tensor", "achieved": tern_tflops / world,
                                 "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                 "frac": tern_tflops / world / peaks["bf16_tflops"],
                                 "peak_source": f"{peaks_src} bf16 burst (fp16 runs at the bf16 rate)",
                                 "traffic": {"up": traffic_for("gemm_packed2_tcr_up"),
                                             "down": traffic_for("gemm_packed2_tcr_down")},
                                 "note": "1 GFLOP products: latency bound (MMA issue chain, stage hand-offs, "
                                         "cluster reduction), not tensor-throughput bound"}},
        "gemv4": {"metric": "4-bit 12288x1536 GEMV weight GB/s (normal-quantile 16-entry codebook)",
                  "value": world * GEMV4_WEIGHT_BYTES / per_call_gemv4_s / 1e9, "unit": "GB/s",
                  "us_per_call": per_call_gemv4_s * 1e6,
                  "mode": "64 independent back-to-back calls over the rotation, two streams",
                  "opts": GEMV4_INDEP,
                  "roofline": {"bound": "hbm", "achieved": GEMV4_TOTAL_BYTES / per_call_gemv4_s / 1e9,
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": GEMV4_TOTAL_BYTES / per_call_gemv4_s / 1e9 / peaks["hbm_gbs"],
                               "traffic": traffic_for("gemv4_lut"), "peak_source": peaks_src}},
        "gemv_t": {"metric": "2-bit 1536x12288 GEMV weight GB/s (transposed shape)",
                   "value": world * GEMV_WEIGHT_BYTES / per_call_gemvt_s / 1e9, "unit": "GB/s",
                   "us_per_call": per_call_gemvt_s * 1e6,
                   "mode": "64 independent back-to-back calls over the rotation, four streams",
                   "kernel": "gemv2_mxf4_kernel, 3 tiles of 127 rows per CTA",
                   "opts": GEMVT_INDEP,
                   "roofline": {"bound": "hbm", "achieved": GEMVT_TOTAL_BYTES / per_call_gemvt_s / 1e9,
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": GEMVT_TOTAL_BYTES / per_call_gemvt_s / 1e9 / peaks["hbm_gbs"],
                                "traffic": traffic_for("gemv2_mxf4_t"), "peak_source": peaks_src}},
        "training_set": {"metric": "fp32 GEMM TFLOP/s, 8192x8192x2048 forward + dA (NT) + dB (TN)",
                         "value": world * TRAIN_FLOP * args.steps / train_total_s / 1e12, "unit": "TFLOP/s",
                         "ms_per_set": train_total_s / args.steps * 1e3,
                         "path": "mm_gemm_f32_splitk, automatic split (plain for the forward product, stream-K for dA and dB)"},
        "gpt2_mlp_up": {"metric": "fp32 GEMM TFLOP/s with bias + GELU (tanh form) fused in the epilogue",
                        "value": world * MLP_FLOP * args.steps / mlp_total_s / 1e12, "unit": "TFLOP/s",
                        "us_per_call": mlp_total_s / args.steps * 1e6,
                        "shape": f"{MLP_M}x{MLP_N}x{MLP_K} NN (8 x 1024 tokens, 768 -> 3072), N(0,1) x N(0,0.02)",
                        "path": "mm_gemm_f32_bias_act_splitk, automatic split (stream-K: 384 pair tiles on 76 pairs)"},
        "roofline": roof,
        "phases": phases,
        "clocks": clk,
        # the FFMA phase's products add a reduce launch each when their stream-K tail runs
        "gpu_launches": (LAUNCHES_PER_STEP + (3 if w.ffma_ws_floats else 0)) * args.steps,
        "wall_s": wall,
    }
    if rank == 0:
        out["e2e"] = e2e_gemm(w, max(2, args.steps // 2), stream)
        if world == 1 and not args.no_cpu_baseline:
            try:
                gpu_gemm = {g["layout"]: g["C"].cpu().numpy() for g in w.gemm}
            except Exception as e:  # the parity check is a report item: it must not cost the line
                print(f"bench: GEMM outputs not read back for the parity check: {e}", file=sys.stderr)
                gpu_gemm = None
            out["cpu_baseline"] = cpu_oracle_sample(gpu_gemm=gpu_gemm)
            try:
                bp = bench_parity(w)
                out["cpu_baseline"]["parity"]["workloads"] = bp["workloads"]
                out["cpu_baseline"]["parity"]["ok"] = bool(out["cpu_baseline"]["parity"]["ok"] and bp["ok"])
                out["cpu_baseline"]["parity"]["what"] += ("; and per workload, the outputs the timed phases left "
                                                          "(see workloads)")
                out["cpu_baseline"]["parity"]["seconds_workloads"] = bp["seconds"]
            except Exception as e:  # a report item: it must not cost the line
                print(f"bench: workload parity not computed: {e}", file=sys.stderr)
        out["inputs_sha256"] = w.inputs_sha256
        print(json.dumps(out), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return main_reference(args)
    return main_mm(args)


if __name__ == "__main__":
    sys.exit(main())

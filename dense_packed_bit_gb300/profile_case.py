"""Run one hot-path kernel a few times on one workload, for profiler captures.

    python -m dense_packed_bit_gb300.profile_case gemm --layout nn --size 2048 --reps 3
    python -m dense_packed_bit_gb300.profile_case gemm --size 2048 --path 1 --misalign 1   (lda = ldb = ldc = n + 1)
    python -m dense_packed_bit_gb300.profile_case c1 --reps 3 [--path 1 --tile 4 --split 8]   (64 x 768 x 3072 NN)
    python -m dense_packed_bit_gb300.profile_case c1 --reps 3 --path 2 --split 4   (workspace K slices + reduce)
    python -m dense_packed_bit_gb300.profile_case c1 --reps 3 --path 2 --tile 4 --split 0   (few rows, tensor cores)
    python -m dense_packed_bit_gb300.profile_case gemv --reps 3 [--split 8 --rows 4 --warps 8 --dequant 2 --independent 1]
    python -m dense_packed_bit_gb300.profile_case gemv --reps 3 --split 0 --rows 1 --warps 0 --dequant 2 --staging 1
    python -m dense_packed_bit_gb300.profile_case gemv --reps 3 --misalign 1   (codes one byte off 16-byte alignment)
    python -m dense_packed_bit_gb300.profile_case gemv4 --reps 3 [--staging 1 --rows 1 --independent 1]
    python -m dense_packed_bit_gb300.profile_case ternary --reps 1 [--tile 2] [--pdl 2: pdl + static weights]
    python -m dense_packed_bit_gb300.profile_case gemv_batched --reps 2 --matrices 16 [--dequant 6 --tiles 0]
    python -m dense_packed_bit_gb300.profile_case gemv_t --reps 3 --matrices 8   (1,536 x 12,288, automatic)
    python -m dense_packed_bit_gb300.profile_case gemv_t --reps 3 --matrices 4 --dequant 6 --rows 3   (fp4 decode)
    python -m dense_packed_bit_gb300.profile_case attn --reps 2   (causal attention 32 x 512 x 64, forward + backward)

One warm-up launch precedes the `reps` launches.  No timing is done here:
numbers come from the profiler or from bench.py.
"""
from __future__ import annotations

import argparse
import sys


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["gemm", "c1", "gemv", "gemv4", "ternary", "gemv_batched", "gemv_t", "attn"])
    ap.add_argument("--layout", default="nn", choices=["nn", "nt", "tn"])
    ap.add_argument("--size", type=int, default=2048)
    ap.add_argument("--path", type=int, default=0)
    ap.add_argument("--tile", type=int, default=0, help="gemm --path 1 --tile 5: the FFMA kernel's stream-K tail")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--matrices", type=int, default=64)
    ap.add_argument("--split", type=int, default=8)
    ap.add_argument("--rows", type=int, default=4)
    ap.add_argument("--warps", type=int, default=4)
    ap.add_argument("--pdl", type=int, default=1)
    ap.add_argument("--dequant", type=int, default=0)
    ap.add_argument("--independent", type=int, default=0)
    ap.add_argument("--staging", type=int, default=None, help="gemv: default 0; gemv4: default automatic")
    ap.add_argument("--misalign", type=int, default=0, help="gemm: leading dimensions n + 1; gemv: codes at an odd address")
    ap.add_argument("--tiles", type=int, default=0, help="batched fp4 decode: 127-row tiles per CTA (0: automatic)")
    a = ap.parse_args(argv)

    import torch

    import dense_packed_bit_gb300 as mm
    from dense_packed_bit_gb300 import build, synth

    build.build()
    mm.load_library()
    dev = torch.device("cuda:0")
    if a.op == "gemm":
        n = a.size
        tA, tB = {"nn": (0, 0), "nt": (0, 1), "tn": (1, 0)}[a.layout]
        ld = n + 1 if a.misalign else n
        A = torch.zeros((n, ld), dtype=torch.float32, device=dev)
        B = torch.zeros((n, ld), dtype=torch.float32, device=dev)
        A[:, :n] = torch.from_numpy(synth.normal_f32(1, (n, n), 0.02)).to(dev)
        B[:, :n] = torch.from_numpy(synth.normal_f32(2, (n, n), 0.02)).to(dev)
        C = torch.empty((n, ld), dtype=torch.float32, device=dev)
        if a.path == 1 and a.tile == 5:
            # the FFMA kernel with its stream-K tail (mm_gemm_f32_splitk_ex, automatic split)
            wsf = mm.mm_gemm_f32_splitk_workspace_ex(n, n, n, 0, path=1)
            ws = torch.empty((max(wsf, 1),), dtype=torch.float32, device=dev)
            for _ in range(1 + a.reps):
                mm.mm_gemm_f32_splitk_ex(tA, tB, n, n, n, A, ld, B, ld, C, ld, 0, ws, wsf, path=1)
        for _ in range(0 if (a.path == 1 and a.tile == 5) else 1 + a.reps):
            mm.mm_gemm_f32_ex(tA, tB, n, n, n, A, ld, B, ld, C, ld, path=a.path, tile=a.tile)
    elif a.op == "c1":
        c = synth.gpt2_mlp_up_64x768x3072()
        A, B = torch.from_numpy(c.A).to(dev), torch.from_numpy(c.B).to(dev)
        C = torch.empty((c.M, c.N), dtype=torch.float32, device=dev)
        workspace_split = a.path == 2 and a.tile != 4 and a.split > 1
        if workspace_split:
            wsf = mm.mm_gemm_f32_splitk_workspace(c.M, c.N, c.K, a.split)
            ws = torch.empty((max(wsf, 1),), dtype=torch.float32, device=dev)
            for _ in range(1 + a.reps):
                mm.mm_gemm_f32_splitk(0, 0, c.M, c.N, c.K, A, c.K, B, c.N, C, c.N, a.split, ws, wsf)
        for _ in range(0 if workspace_split else 1 + a.reps):
            mm.mm_gemm_f32_ex(0, 0, c.M, c.N, c.K, A, c.K, B, c.N, C, c.N, path=a.path, tile=a.tile,
                              splitk=a.split if a.tile == 4 and a.path in (1, 2) else 0)
    elif a.op == "attn":
        c = synth.gpt2_attention_4x8x512x64()
        Q, K, V, dO = (torch.from_numpy(getattr(c, n)).to(dev) for n in ("Q", "K", "V", "dO"))
        O, dQ, dK, dV = (torch.empty_like(Q) for _ in range(4))
        L = torch.empty((c.heads, c.T), dtype=torch.float32, device=dev)
        for _ in range(1 + a.reps):
            mm.mm_attention_fwd(Q, K, V, O, L, c.heads, c.T, c.D, c.causal, 0.125)
            mm.mm_attention_bwd(Q, K, V, O, dO, L, dQ, dK, dV, c.heads, c.T, c.D, c.causal, 0.125)
    elif a.op == "gemv":
        codes, scales = [], []
        for i in range(a.matrices):
            c = synth.gemv_2bit_12288x1536(i)
            if a.misalign:
                buf = torch.empty((c.codes.size + 1,), dtype=torch.uint8, device=dev)
                buf[1:] = torch.from_numpy(c.codes.reshape(-1)).to(dev)
                codes.append(buf[1:])
            else:
                codes.append(torch.from_numpy(c.codes).to(dev))
            scales.append(torch.from_numpy(c.scales).to(dev))
        x = torch.from_numpy(c.X.reshape(-1)).to(dev)
        y = torch.empty((a.matrices, 12288), dtype=torch.float32, device=dev)
        for r in range(1 + a.reps):
            i = r % a.matrices
            mm.mm_gemv_packed2_ex(codes[i], scales[i], x, y[i], 12288, 1536, c.codebook, split=a.split,
                                  rows_per_lane=a.rows, warps=a.warps, dequant=a.dequant, pdl=a.pdl,
                                  weights_static=a.pdl and not a.independent, independent=a.independent,
                                  staging=a.staging or 0)
    elif a.op == "gemv_t":
        codes, scales = [], []
        for i in range(a.matrices):
            c = synth.gemv_2bit_1536x12288(i)
            codes.append(torch.from_numpy(c.codes).to(dev))
            scales.append(torch.from_numpy(c.scales).to(dev))
        x = torch.from_numpy(c.X.reshape(-1)).to(dev)
        y = torch.empty((a.matrices, 1536), dtype=torch.float32, device=dev)
        for r in range(1 + a.reps):
            i = r % a.matrices
            # --dequant 6: the fp4 decode with --rows tiles of 127 rows per CTA; else the automatic decode
            opts = dict(dequant=6, rows_per_lane=a.rows) if a.dequant == 6 else {}
            mm.mm_gemv_packed2_ex(codes[i], scales[i], x, y[i], 1536, 12288, c.codebook, pdl=1, independent=1, **opts)
    elif a.op == "gemv4":
        codes, scales = [], []
        for i in range(a.matrices):
            c = synth.gemv_4bit_12288x1536(i)
            codes.append(torch.from_numpy(c.codes).to(dev))
            scales.append(torch.from_numpy(c.scales).to(dev))
        x = torch.from_numpy(c.X.reshape(-1)).to(dev)
        y = torch.empty((a.matrices, 12288), dtype=torch.float32, device=dev)
        for r in range(1 + a.reps):
            i = r % a.matrices
            mm.mm_gemv_packed4_ex(codes[i], scales[i], x, y[i], 12288, 1536, c.codebook, pdl=a.pdl,
                                  independent=a.independent, staging=-1 if a.staging is None else a.staging,
                                  blocks=a.rows if a.staging else 0)
    elif a.op == "gemv_batched":
        n = a.matrices
        codes = torch.empty((n, 12288, 384), dtype=torch.uint8, device=dev)
        scales = torch.empty((n, 12288), dtype=torch.int16, device=dev)
        for i in range(n):
            c = synth.gemv_2bit_12288x1536(i)
            codes[i].copy_(torch.from_numpy(c.codes))
            scales[i].copy_(torch.from_numpy(c.scales.view("int16")))
        x = torch.from_numpy(c.X.reshape(-1)).to(dev)
        y = torch.empty((n, 12288), dtype=torch.float32, device=dev)
        for _ in range(1 + a.reps):
            mm.mm_gemv_packed2_strided_batched_ex(codes, 12288 * 384, scales, 12288, x, 0, y, 12288, n, 12288, 1536,
                                                  c.codebook, dequant=a.dequant, rows_per_lane=a.tiles)
    else:
        layers = []
        for layer in range(16):
            for proj in ("up", "down"):
                c = synth.ternary_encoder_layer(layer, proj)
                layers.append((c, torch.from_numpy(c.codes).to(dev), torch.from_numpy(c.scales).to(dev),
                               torch.from_numpy(c.X).to(dev),
                               torch.empty((c.X.shape[0], c.rows), dtype=torch.float32, device=dev)))
        for _ in range(1 + a.reps):
            for c, dc, ds, dX, dY in layers:
                if a.tile or a.pdl == 2:
                    mm.mm_gemm_packed2_ex(dc, ds, dX, dY, c.X.shape[0], c.rows, c.cols, c.codebook, tile=a.tile,
                                          pdl=int(a.pdl == 2), weights_static=int(a.pdl == 2))
                else:
                    mm.mm_gemm_packed2(dc, ds, dX, dY, c.X.shape[0], c.rows, c.cols, c.codebook)
    mm.mm_check_device_error()
    torch.cuda.synchronize()
    print("ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())

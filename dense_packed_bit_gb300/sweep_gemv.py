"""Split-width sweep of the 2-bit GEMV decodes on the 12,288 x 1,536 rotation.

    python -m dense_packed_bit_gb300.sweep_gemv [--matrices 64] [--reps 15] [--json out.json]
    python -m dense_packed_bit_gb300.sweep_gemv --streams-sweep [--reps 15]

"Kernel 0112", section "The four variants", sweeps how many threads share one
row's dot product (4, 16, 32).  This sweeps the same knob, and the ones around
it, for every decode of mm_gemv_packed2_ex:

  register loads (affine and select decodes): lanes per row (split) x rows per
  lane x warps per CTA;
  TMA-staged affine: 128-row blocks per CTA (eight warps split K);
  mma.sync decodes: warps per row x 16-row blocks per warp, or 64-row blocks per
  CTA when staged;
  fp8 mma.sync, tcgen05 fp8 and tcgen05 fp4 decodes: row blocks or 127-row tiles per CTA;
  the batched fp4 launch: tiles per CTA.

Each configuration runs the 64 distinct seeded matrices (288 MiB, more than L2)
as independent calls alternating over two streams (programmatic dependent launch,
`independent=1`), captured in a CUDA graph and replayed `reps` times; the median
replay gives microseconds per call and weight GB/s (4,718,592 code bytes per
call) against the copy bandwidth in MEASURED_PEAKS.json when present.  A
configuration the library refuses is listed as such.  Timing only: parity of
every decode is the test suite's job.

--streams-sweep: independent calls of the decodes the bench times, spread over 2, 4
or 8 streams, by 127-row tiles per CTA (fp4 tensor-core decode, 12,288 x 1,536 and
the transposed 1,536 x 12,288), 128-row blocks per CTA (TMA-staged SIMT decode) and
64-row blocks per CTA (4-bit table decode, 32 matrices of 9 MiB); fraction of HBM on
all the call's bytes.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

CODE_BYTES = 12288 * 384
TOTAL_BYTES = CODE_BYTES + 12288 * 2 + 1536 * 2 + 12288 * 4


def configs():
    out = []
    for dq, name in ((2, "regload affine"), (1, "regload select")):
        for split in (4, 8, 16):
            for rows in (1, 2, 4):
                for warps in (4, 8):
                    out.append((name, dict(dequant=dq, staging=0, split=split, rows_per_lane=rows, warps=warps)))
    for blocks in (1, 2, 3, 4, 6):
        out.append(("staged affine", dict(dequant=2, staging=1, rows_per_lane=blocks)))
    for split in (1, 2, 3, 4, 6):
        for rows in (1, 2, 4):
            out.append(("mma.sync", dict(dequant=3, staging=0, split=split, rows_per_lane=rows, warps=split * 2)))
    for blocks in (1, 2, 4, 8):
        out.append(("mma.sync staged", dict(dequant=3, staging=1, rows_per_lane=blocks)))
    for blocks in (1, 2, 4, 8):
        out.append(("fp8 mma.sync", dict(dequant=4, rows_per_lane=blocks)))
    for tiles in (1, 2, 4):
        out.append(("tcgen05 fp8", dict(dequant=5, rows_per_lane=tiles)))
    for tiles in (1, 2, 4):
        out.append(("tcgen05 mxf4", dict(dequant=6, rows_per_lane=tiles)))
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--matrices", type=int, default=64)
    ap.add_argument("--reps", type=int, default=15)
    ap.add_argument("--json", default=None)
    ap.add_argument("--streams-sweep", action="store_true")
    a = ap.parse_args(argv)
    if a.streams_sweep:
        return streams_sweep(a.reps)

    import numpy as np
    import torch

    import dense_packed_bit_gb300 as mm
    from dense_packed_bit_gb300 import build, synth

    build.build()
    mm.load_library()
    dev = torch.device("cuda:0")
    n = a.matrices
    codes = torch.empty((n, 12288, 384), dtype=torch.uint8, device=dev)
    scales = torch.empty((n, 12288), dtype=torch.int16, device=dev)
    for i in range(n):
        c = synth.gemv_2bit_12288x1536(i)
        codes[i].copy_(torch.from_numpy(c.codes))
        scales[i].copy_(torch.from_numpy(c.scales.view("int16")))
    cb = c.codebook
    x = torch.from_numpy(c.X.reshape(-1)).to(dev)
    y = torch.empty((n, 12288), dtype=torch.float32, device=dev)
    hbm = None
    peaks_path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        hbm = json.load(open(peaks_path)).get("hbm_gbs")
    stream = torch.cuda.Stream(device=dev)
    side = torch.cuda.Stream(device=dev)

    def timed(fn):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        mm.mm_check_device_error()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        ts = []
        for _ in range(a.reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):  # a graph replays on the current stream
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / n)
        mm.mm_check_device_error()
        return float(np.median(ts))

    def independent(opts):
        def f():
            cur = torch.cuda.current_stream()
            side.wait_stream(cur)
            for i in range(n):
                s = cur if i % 2 == 0 else side
                mm.mm_gemv_packed2_ex(codes[i], scales[i], x, y[i], 12288, 1536, cb, s, pdl=1, independent=1, **opts)
            cur.wait_stream(side)
        return f

    def batched(tiles):
        def f():
            mm.mm_gemv_packed2_strided_batched_ex(codes, 12288 * 384, scales, 12288, x, 0, y, 12288, n, 12288, 1536,
                                                  cb, dequant=mm.MM_DEQ_MXF4, rows_per_lane=tiles)
        return f

    rows = []
    runs = [(name, opts, independent(opts)) for name, opts in configs()]
    runs += [("batched mxf4", dict(tiles_per_cta=t), batched(t)) for t in (0, 4, 8, 12, 16, 24)]
    for name, opts, fn in runs:
        try:
            us = timed(fn)
        except mm.MMError as e:
            rows.append(dict(decode=name, opts=opts, refused=str(e)))
            print(f"{name:16s} {json.dumps(opts):70s} refused: {e}", flush=True)
            continue
        gbs = CODE_BYTES / (us * 1e-6) / 1e9
        r = dict(decode=name, opts=opts, us_per_call=round(us, 3), weight_gbs=round(gbs, 1))
        if hbm:
            r["frac_hbm_total_bytes"] = round(TOTAL_BYTES / (us * 1e-6) / 1e9 / hbm, 3)
        rows.append(r)
        print(f"{name:16s} {json.dumps(opts):70s} {us:7.3f} us  {gbs:7.0f} GB/s"
              + (f"  {r['frac_hbm_total_bytes']:.3f} of HBM" if hbm else ""), flush=True)
    if a.json:
        json.dump(rows, open(a.json, "w"), indent=1)
    return 0


def streams_sweep(reps):
    import numpy as np
    import torch

    import dense_packed_bit_gb300 as mm
    from dense_packed_bit_gb300 import build, synth

    build.build()
    mm.load_library()
    dev = torch.device("cuda:0")
    hbm = 6772.5
    peaks_path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        hbm = json.load(open(peaks_path)).get("hbm_gbs") or hbm
    streams = [torch.cuda.Stream(device=dev) for _ in range(8)]
    main_st = streams[0]

    def timed(fn, n):
        try:
            with torch.cuda.stream(main_st):
                fn()
        except mm.MMError:
            torch.cuda.synchronize()
            return float("nan")
        torch.cuda.synchronize()
        mm.mm_check_device_error()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main_st):
            fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(main_st):
                e0.record(main_st)
                g.replay()
                e1.record(main_st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / n)
        mm.mm_check_device_error()
        return float(np.median(ts))

    def indep(call, n, ns):
        def f():
            cur = torch.cuda.current_stream()
            sts = [cur] + streams[1:ns]
            for s in sts[1:]:
                s.wait_stream(cur)
            for i in range(n):
                call(i, sts[i % ns])
            for s in sts[1:]:
                cur.wait_stream(s)
        return f

    def load(fn, n):
        cs = [fn(i) for i in range(n)]
        codes = torch.stack([torch.from_numpy(c.codes) for c in cs]).to(dev)
        scales = torch.stack([torch.from_numpy(c.scales.view("int16")) for c in cs]).to(dev)
        return codes, scales, torch.from_numpy(cs[0].X.reshape(-1)).to(dev), cs[0].codebook

    def report(label, us, nbytes):
        print(f"{label:52s} {us:7.3f} us/call  {nbytes / us / 1e3 / hbm:.3f} of HBM", flush=True)

    n = 64
    total2 = 12288 * 384 + 12288 * 2 + 1536 * 2 + 12288 * 4
    codes, scales, x, cb = load(synth.gemv_2bit_12288x1536, n)
    y = torch.empty((n, 12288), dtype=torch.float32, device=dev)
    for ns in (2, 4, 8):
        for t in (6, 8, 10, 12, 15, 20, 25, 33, 49):
            call = lambda i, s, t=t: mm.mm_gemv_packed2_ex(codes[i], scales[i], x, y[i], 12288, 1536, cb, s, pdl=1,
                                                           independent=1, dequant=6, rows_per_lane=t)
            report(f"12288x1536 fp4 decode, {t} tiles/CTA, {ns} streams", timed(indep(call, n, ns), n), total2)
        for b in (2, 3, 4, 6):
            call = lambda i, s, b=b: mm.mm_gemv_packed2_ex(codes[i], scales[i], x, y[i], 12288, 1536, cb, s, pdl=1,
                                                           independent=1, dequant=2, staging=1, rows_per_lane=b)
            report(f"12288x1536 staged SIMT, {b} blocks/CTA, {ns} streams", timed(indep(call, n, ns), n), total2)
    del codes, scales
    codes, scales, x, cb = load(synth.gemv_2bit_1536x12288, n)
    y = torch.empty((n, 1536), dtype=torch.float32, device=dev)
    total_t = 1536 * 3072 + 1536 * 2 + 12288 * 2 + 1536 * 4
    for ns in (4, 8):
        for t in (1, 2, 3, 4, 5, 7):
            call = lambda i, s, t=t: mm.mm_gemv_packed2_ex(codes[i], scales[i], x, y[i], 1536, 12288, cb, s, pdl=1,
                                                           independent=1, dequant=6, rows_per_lane=t)
            report(f"1536x12288 fp4 decode, {t} tiles/CTA, {ns} streams", timed(indep(call, n, ns), n), total_t)
    del codes, scales
    n4 = 32
    codes, scales, x, cb = load(synth.gemv_4bit_12288x1536, n4)
    y = torch.empty((n4, 12288), dtype=torch.float32, device=dev)
    total4 = 12288 * 768 + 12288 * 2 + 1536 * 2 + 12288 * 4
    for ns in (2, 4, 8):
        for b in (1, 2, 3):
            call = lambda i, s, b=b: mm.mm_gemv_packed4_ex(codes[i], scales[i], x, y[i], 12288, 1536, cb, s,
                                                           staging=1, blocks=b, pdl=1, independent=1)
            report(f"12288x1536 4-bit table, {b} blocks/CTA, {ns} streams", timed(indep(call, n4, ns), n4), total4)
    return 0


if __name__ == "__main__":
    sys.exit(main())

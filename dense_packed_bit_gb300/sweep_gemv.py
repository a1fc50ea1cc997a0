"""Split-width sweep of the 2-bit GEMV decodes on the 12,288 x 1,536 rotation.

    python -m dense_packed_bit_gb300.sweep_gemv [--matrices 64] [--reps 15] [--json out.json]

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
    a = ap.parse_args(argv)

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


if __name__ == "__main__":
    sys.exit(main())

"""Shape sweep of the ternary 16-layer encoder block as the bench chains it.

    python -m dense_packed_bit_gb300.sweep_tern [--reps 20]

"More Stumbling, This Time in the Browser", section "This time, in a browser":
the encoder's 16 layers each multiply 2 x 111 = 222 token rows by an up
(3072 x 768) and a down (768 x 3072) ternary matrix.  The 32 products run as one
dependent chain (programmatic dependent launch, weights promised static), as in
the bench, for each pair of (tokens per tile, CTAs of the cluster splitting K)
of the tensor-memory kernel (tile 3) for the up and the down projection;
(0, 0) is the automatic choice.  Median of `reps` graph replays, microseconds per
block.  Timing only: parity is the test suite's job.
"""
from __future__ import annotations

import argparse
import sys

UP = [(0, 0), (80, 2), (224, 1), (224, 2), (224, 4), (112, 1), (112, 2), (80, 1), (48, 1), (64, 2)]
DOWN = [(0, 0), (112, 8), (224, 8), (112, 4), (224, 4), (80, 4), (80, 8), (64, 4), (64, 8)]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=20)
    a = ap.parse_args(argv)

    import numpy as np
    import torch

    import dense_packed_bit_gb300 as mm
    from dense_packed_bit_gb300 import build, synth

    build.build()
    mm.load_library()
    dev = torch.device("cuda:0")
    prods = []
    for layer in range(16):
        for proj in ("up", "down"):
            c = synth.ternary_encoder_layer(layer, proj)
            prods.append(dict(c=c, proj=proj, codes=torch.from_numpy(c.codes).to(dev),
                              scales=torch.from_numpy(c.scales).to(dev), X=torch.from_numpy(c.X).to(dev),
                              Y=torch.empty((c.X.shape[0], c.rows), dtype=torch.float32, device=dev)))
    st = torch.cuda.Stream(device=dev)

    def run(up, down):
        for t in prods:
            c = t["c"]
            ntok, split = up if t["proj"] == "up" else down
            kw = dict(tile=3, splitk=split, ntok=ntok) if ntok else {}
            mm.mm_gemm_packed2_ex(t["codes"], t["scales"], t["X"], t["Y"], c.X.shape[0], c.rows, c.cols,
                                  c.codebook, pdl=1, weights_static=1, **kw)

    def timed(up, down):
        try:
            with torch.cuda.stream(st):
                run(up, down)
            torch.cuda.synchronize()
            mm.mm_check_device_error()
        except mm.MMError:
            torch.cuda.synchronize()
            return None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            run(up, down)
        ts = []
        for _ in range(a.reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(st):
                e0.record(st)
                g.replay()
                e1.record(st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        mm.mm_check_device_error()
        return float(np.median(ts))

    for up in UP:
        for down in DOWN:
            us = timed(up, down)
            print(f"up (ntok, S) = {up}, down (ntok, S) = {down}: "
                  + (f"{us:.1f} us per block" if us is not None else "refused"), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())

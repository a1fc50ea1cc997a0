"""Dependent GEMV chains: each call's activations are bytes the previous call wrote.

"Kernel 0112", section "What the kernel costs in a whole token": a token runs its
weight-reading kernels one after another, each reading what the one before it
wrote.  The chained launch mode serves exactly that: with programmatic dependent
launch a GEMV may start, and with weights_static load its weights, while the
previous kernel still runs; it must not read x, nor write y, before that kernel
has finished.  These tests give every GEMV kernel that has a chained mode three
calls on one stream:

  call 1 reads x1 from buffer P and writes y1;
  call 2 reads x2 from buffer Q and writes y2 over P        (write after read: call 1's x);
  call 3 reads as x3 the first bytes of P, i.e. y2's bits   (read after write: call 2's y),
         and writes y3 over Q                               (write after read: call 2's x).

Integer activations in {-1, 0, 1}, an integer codebook and unit scales make y1 and
y2 integers below 2^11 in magnitude, which the oracle gives exactly and whose fp32
bits read as finite fp16 values; call 3's expectation is the oracle's product on
exactly those bits.  A call that read its x before its predecessor finished
writing it, or wrote its y while its predecessor still read that memory, returns
a different y.  The chain runs three times in a row on the same buffers.
"""
import numpy as np
import pytest

import dense_packed_bit_gb300 as mm
from dense_packed_bit_gb300 import synth
from gpu_util import check_bound, check_exact, empty_f32, to_dev, to_host

pytestmark = pytest.mark.gpu

CB2 = synth.CODEBOOK_2BIT
CB4_INT = np.arange(-8, 8, dtype=np.float32)   # integer 16-entry codebook: exact integer outputs


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_packed_bit_gb300 import build
    build.build()
    mm.load_library()


# (name, field bits, rows, cols, options of the chained call)
VARIANTS = [
    ("staged_affine", 2, 12288, 1536, dict(dequant=2, staging=1)),
    ("regload_affine", 2, 12288, 1536, dict(dequant=2, staging=0)),
    ("select", 2, 12288, 1536, dict(dequant=1)),
    ("mma_sync", 2, 12288, 1536, dict(dequant=3, staging=0)),
    ("mma_sync_staged", 2, 12288, 1536, dict(dequant=3, staging=1)),
    ("fp8_mma_sync", 2, 12288, 1536, dict(dequant=4)),
    ("tcgen05", 2, 12288, 1536, dict(dequant=5)),
    ("mxf4", 2, 12288, 1536, dict(dequant=6)),
    ("transposed", 2, 1536, 12288, dict()),
    ("mxf4_transposed", 2, 1536, 12288, dict(dequant=6)),
    ("staged_4bit", 4, 12288, 1536, dict(staging=1)),
    ("generic_4bit", 4, 12288, 1536, dict(staging=0)),
]


def _codes(bits, rows, cols, seed):
    rb = (cols * bits + 7) // 8
    return synth.random_bytes(seed, rows * rb).reshape(rows, rb)


def _call(bits, codes, scales, x, y, rows, cols, cb, opts):
    if bits == 2:
        mm.mm_gemv_packed2_ex(codes, scales, x, y, rows, cols, cb, **opts)
    else:
        mm.mm_gemv_packed4_ex(codes, scales, x, y, rows, cols, cb, **opts)


def _oracle(oracle, bits, codes, scales, x, rows, cols, cb):
    f = oracle.packed_gemm if bits == 2 else oracle.packed4_gemm
    ref, T = f(codes, scales, x.reshape(1, cols), rows, cols, cb)
    return ref[0], T[0]


@pytest.mark.parametrize("weights_static", [0, 1])
@pytest.mark.parametrize("variant", VARIANTS, ids=[v[0] for v in VARIANTS])
def test_gemv_chain_reads_and_writes_after_its_predecessor(oracle, variant, weights_static):
    import torch
    name, bits, rows, cols, base = variant
    cb = CB2 if bits == 2 else CB4_INT
    opts = dict(base, pdl=1, weights_static=weights_static)
    rng = np.random.default_rng(rows + cols + bits)
    codes = [_codes(bits, rows, cols, 500 + 10 * bits + i) for i in range(3)]
    ones = np.full(rows, 0x3C00, np.uint16)
    x1 = rng.integers(-1, 2, size=cols).astype(np.float16).view(np.uint16)
    x2 = rng.integers(-1, 2, size=cols).astype(np.float16).view(np.uint16)
    # P holds x1, then y2, whose first 2 * cols bytes are read as x3; Q holds x2, then y3
    nfl = max(rows, (cols + 1) // 2)
    P, Q = empty_f32((nfl,)), empty_f32((nfl,))
    y1 = empty_f32((rows,))
    dc = [to_dev(c) for c in codes]
    ds = to_dev(ones)
    x1_t = torch.from_numpy(x1.view(np.int16)).to(P.device)
    x2_t = torch.from_numpy(x2.view(np.int16)).to(P.device)
    Px = P.view(torch.int16)[:cols]
    Qx = Q.view(torch.int16)[:cols]
    ref1, _ = _oracle(oracle, bits, codes[0], ones, x1, rows, cols, cb)
    ref2, _ = _oracle(oracle, bits, codes[1], ones, x2, rows, cols, cb)
    assert np.all(np.abs(ref2) < 2048), "y2 must read as finite fp16 values"
    for rep in range(3):
        P.fill_(float("nan"))
        Q.fill_(float("nan"))
        Px.copy_(x1_t)
        Qx.copy_(x2_t)
        _call(bits, dc[0], ds, Px, y1, rows, cols, cb, opts)
        _call(bits, dc[1], ds, Qx, P[:rows], rows, cols, cb, opts)
        _call(bits, dc[2], ds, Px, Q[:rows], rows, cols, cb, opts)
        mm.mm_check_device_error()
        check_exact(to_host(y1), ref1, f"{name}: call 1 read x1 before call 2 overwrote it")
        Ph = to_host(P)
        check_exact(Ph[:rows], ref2, f"{name}: call 2")
        # x3 = the first 2 * cols bytes of P as call 3 found them: y2's bits (and, when y2 is
        # shorter than x3, the tail of x1's buffer left as it was)
        x3 = Ph.view(np.uint16)[:cols].copy()
        assert np.all(np.isfinite(x3.view(np.float16)))
        ref3, T3 = _oracle(oracle, bits, codes[2], ones, x3, rows, cols, cb)
        worst = check_bound(to_host(Q)[:rows], ref3, T3, f"{name}: call 3 read call 2's y (repeat {rep})")
    print(f"{name} weights_static={weights_static}: call 3 worst |err|/T = {worst:.3e}")


@pytest.mark.parametrize("weights_static", [0, 1])
def test_batched_fp4_chain_reads_and_writes_after_its_predecessor(oracle, weights_static):
    # the same three-call chain through the strided-batched fp4 launch (two matrices per call,
    # a shared x): with programmatic dependent launch each batched kernel may start while the
    # previous one runs, and must still read x and write y only after it
    import torch
    batch, rows, cols = 2, 12288, 1536
    rb = cols // 4
    opts = dict(dequant=mm.MM_DEQ_MXF4, pdl=1, weights_static=weights_static)
    rng = np.random.default_rng(77 + weights_static)
    codes = [np.stack([_codes(2, rows, cols, 900 + 10 * i + b) for b in range(batch)]) for i in range(3)]
    ones = np.full((batch, rows), 0x3C00, np.uint16)
    x1 = rng.integers(-1, 2, size=cols).astype(np.float16).view(np.uint16)
    x2 = rng.integers(-1, 2, size=cols).astype(np.float16).view(np.uint16)
    nfl = max(batch * rows, (cols + 1) // 2)
    P, Q = empty_f32((nfl,)), empty_f32((nfl,))
    y1 = empty_f32((batch * rows,))
    dc = [to_dev(c) for c in codes]
    ds = to_dev(ones)
    x1_t = torch.from_numpy(x1.view(np.int16)).to(P.device)
    x2_t = torch.from_numpy(x2.view(np.int16)).to(P.device)
    Px = P.view(torch.int16)[:cols]
    Qx = Q.view(torch.int16)[:cols]

    def call(i, x, y):
        mm.mm_gemv_packed2_strided_batched_ex(dc[i], rows * rb, ds, rows, x, 0, y, rows, batch, rows, cols, CB2,
                                              **opts)

    ref1 = [_oracle(oracle, 2, codes[0][b], ones[b], x1, rows, cols, CB2)[0] for b in range(batch)]
    ref2 = [_oracle(oracle, 2, codes[1][b], ones[b], x2, rows, cols, CB2)[0] for b in range(batch)]
    assert np.all(np.abs(ref2[0]) < 2048), "y2 must read as finite fp16 values"
    for rep in range(3):
        P.fill_(float("nan"))
        Q.fill_(float("nan"))
        Px.copy_(x1_t)
        Qx.copy_(x2_t)
        call(0, Px, y1)
        call(1, Qx, P[:batch * rows])
        call(2, Px, Q[:batch * rows])
        mm.mm_check_device_error()
        y1h, Ph, Qh = to_host(y1), to_host(P), to_host(Q)
        for b in range(batch):
            check_exact(y1h[b * rows:(b + 1) * rows], ref1[b], f"batched call 1, matrix {b}")
            check_exact(Ph[b * rows:(b + 1) * rows], ref2[b], f"batched call 2, matrix {b}")
        x3 = Ph.view(np.uint16)[:cols].copy()
        assert np.all(np.isfinite(x3.view(np.float16)))
        for b in range(batch):
            ref3, T3 = _oracle(oracle, 2, codes[2][b], ones[b], x3, rows, cols, CB2)
            check_bound(Qh[b * rows:(b + 1) * rows], ref3, T3, f"batched call 3, matrix {b} (repeat {rep})")


def test_batched_fp4_independent_launches_same_bits():
    # back-to-back batched launches with independent = 1 (no wait on the previous kernel), each
    # into its own y: the same bits as plain launches
    import torch
    batch, rows, cols = 8, 4000, 1536
    rb = cols // 4
    codes = np.stack([_codes(2, rows, cols, 950 + b) for b in range(batch)])
    scales = synth.uniform_f16_bits(951, (batch, rows), 0.005, 0.05)
    x = synth.normal_f16_bits(952, (cols,))
    dc, ds, dx = to_dev(codes), to_dev(scales), to_dev(x)
    plain = empty_f32((batch, rows))
    mm.mm_gemv_packed2_strided_batched_ex(dc, rows * rb, ds, rows, dx, 0, plain, rows, batch, rows, cols, CB2,
                                          dequant=mm.MM_DEQ_MXF4)
    ref = to_host(plain)
    for opts in (dict(pdl=1), dict(pdl=1, weights_static=1), dict(pdl=1, independent=1)):
        ys = [empty_f32((batch, rows)) for _ in range(4)]
        for y in ys:
            mm.mm_gemv_packed2_strided_batched_ex(dc, rows * rb, ds, rows, dx, 0, y, rows, batch, rows, cols, CB2,
                                                  dequant=mm.MM_DEQ_MXF4, **opts)
        mm.mm_check_device_error()
        for j, y in enumerate(ys):
            assert np.array_equal(to_host(y).view(np.uint32), ref.view(np.uint32)), f"{opts}: launch {j}"

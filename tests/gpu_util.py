"""Helpers for the GPU parity tests: device transfers and the acceptance check.

The acceptance bound for every output is |y - y_ref| <= 1e-5 * T where
T = sum_k |term_k| (both from the fp64 oracle); bit-exact cases compare the
fp32 result with the fp64 oracle value, which must then be an fp32 number.

Guard bands: every output that empty_f32 allocates sits between GUARD floats of
a sentinel NaN on each side, and to_host checks both bands bit for bit when it
reads the output back, so a kernel that writes before or past its output fails
the test that launched it.
"""
import numpy as np

TOL = 1e-5
GUARD = 64                 # sentinel floats before and after every output (256 bytes)
SENTINEL = 0x7FC0DEAD      # a quiet NaN whose payload no kernel writes (below 2^31: an int32)


def torch_dev():
    import torch
    assert torch.cuda.is_available(), "GPU test needs CUDA"
    return torch.device("cuda:0")


def to_dev(a: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(torch_dev())


def empty_f32(shape, fill=float("nan"), device=None):
    """A contiguous fp32 output of `shape` filled with `fill` (default: the sentinel NaN),
    inside a buffer with GUARD sentinel floats before and after it."""
    import torch
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.int32,
                     device=device if device is not None else torch_dev())
    out = buf[GUARD:GUARD + n].view(torch.float32).reshape(shape)
    if not (isinstance(fill, float) and np.isnan(fill)):
        out.fill_(fill)
    out._guard = (buf, n)  # lives and dies with the output
    return out


def check_guard(t):
    """Assert the guard bands around an output from empty_f32 are untouched (no-op for others)."""
    entry = getattr(t, "_guard", None)
    if entry is None:
        return
    buf, n = entry
    before = buf[:GUARD].cpu().numpy().view(np.uint32)
    after = buf[GUARD + n:].cpu().numpy().view(np.uint32)
    for name, band in (("before", before), ("after", after)):
        bad = np.flatnonzero(band != SENTINEL)
        if bad.size:
            off = (bad - GUARD) if name == "before" else bad
            raise AssertionError(f"output of {n} floats: {bad.size} words written {name} it "
                                 f"(offsets {off[:5].tolist()}{' from its start' if name == 'before' else ' past its end'})")


def to_host(t) -> np.ndarray:
    import torch
    if t.is_cuda:
        torch.cuda.synchronize()
    check_guard(t)
    return t.cpu().numpy()


def check_bound(got, ref, T, what=""):
    """Assert |got - ref| <= 1e-5 * T elementwise; returns the worst err / T."""
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > TOL * T
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(i), float(got[tuple(i)]), float(ref[tuple(i)]), float(T[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} outputs outside 1e-5*T, e.g. {detail}")
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(T > 0, err / T, 0.0)
    return float(r.max()) if r.size else 0.0


def check_exact(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert np.array_equal(got, ref), f"{what}: not bit-exact, max |diff| {np.max(np.abs(got - ref))}"

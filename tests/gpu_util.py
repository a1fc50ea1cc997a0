"""Helpers for the GPU parity tests: device transfers and the acceptance check.

The acceptance bound for every output is |y - y_ref| <= 1e-5 * T where
T = sum_k |term_k| (both from the fp64 oracle); bit-exact cases compare the
fp32 result with the fp64 oracle value, which must then be an fp32 number.
"""
import numpy as np

TOL = 1e-5


def torch_dev():
    import torch
    assert torch.cuda.is_available(), "GPU test needs CUDA"
    return torch.device("cuda:0")


def to_dev(a: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(torch_dev())


def empty_f32(shape, fill=float("nan")):
    import torch
    return torch.full(shape, fill, dtype=torch.float32, device=torch_dev())


def to_host(t) -> np.ndarray:
    import torch
    torch.cuda.synchronize()
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

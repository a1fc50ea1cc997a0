"""The guard bands of the GPU tests' output helper, exercised on CPU tensors.

A GPU test can only rely on the guard check if the check itself is right: it
must pass for an output whose own elements are all written, and fail for a
single word written just before or just past the output.
"""
import numpy as np
import pytest

from gpu_util import GUARD, SENTINEL, check_guard, empty_f32, to_host

torch = pytest.importorskip("torch")
CPU = torch.device("cpu")


def test_output_layout_and_fill():
    t = empty_f32((3, 5), device=CPU)
    assert t.shape == (3, 5) and t.dtype == torch.float32 and t.is_contiguous()
    h = to_host(t)
    assert np.all(np.isnan(h)) and np.all(h.view(np.uint32) == SENTINEL)
    z = empty_f32((7,), 0.0, device=CPU)
    assert np.all(to_host(z) == 0.0)


def test_fully_written_output_passes():
    t = empty_f32((4, 9), device=CPU)
    t.copy_(torch.arange(36, dtype=torch.float32).reshape(4, 9))
    assert np.array_equal(to_host(t), np.arange(36, dtype=np.float32).reshape(4, 9))


@pytest.mark.parametrize("where", [-1, -GUARD, 0, GUARD - 1])
def test_write_outside_the_output_is_caught(where):
    t = empty_f32((10,), device=CPU)
    buf, n = t._guard
    t.fill_(1.0)
    # one word before the output (where < 0) or past its end (where >= 0)
    idx = GUARD + where if where < 0 else GUARD + n + where
    buf[idx] = 0
    with pytest.raises(AssertionError, match="before" if where < 0 else "past its end"):
        to_host(t)


def test_views_and_foreign_tensors_are_not_checked():
    t = empty_f32((6,), device=CPU)
    check_guard(t[1:])                      # a view carries no guard: no check, no error
    check_guard(torch.zeros(3))
    check_guard(np.zeros(3))

"""Failure detection on the GPU, without a fault.

A bounded device wait that runs out must reach the host as MM_ERR_TIMEOUT, be
cleared by reading it, and leave the context usable for the next call.  The
probe waits on an mbarrier phase that expects one arrival and gets none (a flag
that nothing sets) through the same wait helper every pipelined kernel uses,
with a limit of a few milliseconds; nothing traps, faults or hangs, and the
host refuses limits above 0.1 s.
"""
import numpy as np
import pytest

import dense_packed_bit_gb300 as mm
from dense_packed_bit_gb300 import synth
from gpu_util import check_bound, empty_f32, to_dev, to_host

pytestmark = pytest.mark.gpu

MS = 1_000_000  # ns


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_packed_bit_gb300 import build
    build.build()
    mm.load_library()
    mm.mm_check_device_error()  # start from a clear error word


def _out():
    import torch
    return torch.full((2,), -1, dtype=torch.int64, device="cuda:0")


def _timeout_reported(stream=None):
    with pytest.raises(mm.MMError) as ei:
        mm.mm_check_device_error(stream)
    assert ei.value.status == mm.MM_ERR_TIMEOUT, str(ei.value)
    assert "probe" in str(ei.value)


def test_completed_wait_reports_ok():
    out = _out()
    mm.mm_probe_bounded_wait(1, 5 * MS, out)
    mm.mm_check_device_error()
    done, waited = to_host(out).tolist()
    assert done == 1
    assert 0 <= waited < 5 * MS


@pytest.mark.parametrize("limit", [20_000, 2 * MS])
def test_wait_that_runs_out_reports_timeout_once(limit):
    out = _out()
    mm.mm_probe_bounded_wait(0, limit, out)
    _timeout_reported()
    done, waited = to_host(out).tolist()
    assert done == 0
    assert limit < waited < limit + 50 * MS     # ran out after the limit, and not much later
    mm.mm_check_device_error()                  # reading cleared the word


def test_timeout_on_a_side_stream():
    import torch
    s = torch.cuda.Stream()
    out = _out()
    s.wait_stream(torch.cuda.current_stream())  # the fill of `out` comes before the probe's write
    with torch.cuda.stream(s):
        mm.mm_probe_bounded_wait(0, MS, out, stream=s)
    _timeout_reported(stream=s)
    assert to_host(out).tolist()[0] == 0


def test_context_usable_after_timeout(oracle):
    mm.mm_probe_bounded_wait(0, MS, None)
    _timeout_reported()
    # the next GEMM and GEMV run normally and match the oracle
    c = synth.gpt2_mlp_up_64x768x3072()
    dC = empty_f32((c.M, c.N))
    mm.mm_gemm_f32(c.transA, c.transB, c.M, c.N, c.K, to_dev(c.A), c.K, to_dev(c.B), c.N, dC, c.N)
    mm.mm_check_device_error()
    ref, T = oracle.gemm(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B)
    check_bound(to_host(dC), ref, T, c.name)
    g = synth.gemv_2bit_12288x1536(0)
    y = empty_f32((g.rows,))
    mm.mm_gemv_packed2(to_dev(g.codes), to_dev(g.scales), to_dev(g.X.reshape(-1)), y, g.rows, g.cols, g.codebook)
    mm.mm_check_device_error()
    yref, yT = oracle.packed_gemm(g.codes, g.scales, g.X, g.rows, g.cols, g.codebook)
    check_bound(to_host(y), yref.reshape(-1), yT.reshape(-1), g.name)


def test_probe_is_asynchronous_and_ordered():
    # two probes on one stream: the word holds the first timeout until it is read; a completed
    # wait queued after it does not clear it
    out = _out()
    mm.mm_probe_bounded_wait(0, MS, None)
    mm.mm_probe_bounded_wait(1, MS, out)
    _timeout_reported()
    assert to_host(out).tolist()[0] == 1
    mm.mm_check_device_error()

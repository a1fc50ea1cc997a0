"""Host-side logic of bench.py that needs no GPU: the parity figure it reports beside the
CPU baseline, and the input digests of its workloads."""
import math
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from dense_packed_bit_gb300 import synth  # noqa: E402


def test_parity_ratio_hand_cases():
    ref = np.array([[1.0, -2.0], [0.0, 4.0]])
    T = np.array([[2.0, 4.0], [0.0, 8.0]])
    assert bench.parity_ratio(ref.astype(np.float32), ref, T) == 0.0
    got = ref.copy()
    got[1, 1] += 8e-5                      # 1e-5 of its T
    assert math.isclose(bench.parity_ratio(got, ref, T), 1e-5, rel_tol=1e-9)
    got = ref.copy()
    got[1, 0] = 1e-30                      # an error where T = 0
    assert bench.parity_ratio(got, ref, T) == math.inf
    got = ref.copy()
    got[0, 0] = np.nan
    assert bench.parity_ratio(got, ref, T) == math.inf
    assert bench.parity_ratio(ref[:1], ref, T) == math.inf          # wrong shape
    assert bench.parity_ratio(np.zeros((0, 2)), np.zeros((0, 2)), np.zeros((0, 2))) == 0.0


def _small_square(layout, replica=0):
    tA, tB = {"nn": (0, 0), "nt": (0, 1), "tn": (1, 0)}[layout]
    return synth.gemm_case(f"square_64_{layout}", tA, tB, 64, 48, 80, "normal", 40, replica=replica)


def _fp32_product(c):
    A = c.A.T if c.transA else c.A
    B = c.B.T if c.transB else c.B
    return (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float32)


def test_cpu_baseline_reports_parity_of_given_outputs(monkeypatch):
    # the recipe shrunk to 64 x 48 x 80 so that the oracle runs in milliseconds
    monkeypatch.setattr(synth, "square_2048", _small_square)
    good = {l: _fp32_product(_small_square(l)) for l in ("nn", "nt", "tn")}
    res = bench.cpu_oracle_sample(seconds_target=0.0, gpu_gemm=good)
    p = res["parity"]
    assert p["ok"] is True and set(p["square_2048"]) == {"nn", "nt", "tn"}
    assert all(v <= 1e-6 for v in p["square_2048"].values())   # fp32 rounding of an fp64 product
    assert res["kind"] == "oracle" and res["cores"] >= 1 and res["value"] > 0

    bad = dict(good)
    bad["nt"] = good["nt"].copy()
    bad["nt"][5, 7] += 0.5
    p = bench.cpu_oracle_sample(seconds_target=0.0, gpu_gemm=bad)["parity"]
    assert p["ok"] is False and p["square_2048"]["nt"] > 1e-5 and p["square_2048"]["nn"] <= 1e-6

    assert "parity" not in bench.cpu_oracle_sample(seconds_target=0.0)


def test_cpu_baseline_sample_is_bounded(monkeypatch):
    # with no time bound reached, the sample stops at its product cap, in whole NN/NT/TN rounds,
    # and draws each product's inputs once (before timing), not once per product
    drawn = []

    def counting(layout, replica=0):
        drawn.append(layout)
        return _small_square(layout, replica)

    monkeypatch.setattr(synth, "square_2048", counting)
    res = bench.cpu_oracle_sample(seconds_target=1e9)
    assert bench.CPU_SAMPLE_MAX_PRODUCTS % 3 == 0
    assert res["sample"].startswith(f"{bench.CPU_SAMPLE_MAX_PRODUCTS} full")
    assert sorted(drawn) == ["nn", "nt", "tn"]


def test_digest_incremental_equals_whole():
    a, b = synth.uniform_f32(3, (4, 5)), synth.random_bytes(4, 33)
    assert synth.Digest().update(a).update(b).hexdigest() == synth.digest(a, b)
    assert synth.digest(a, b) != synth.digest(b, a)
    assert synth.digest(a) != synth.digest(a.reshape(5, 4))          # the shape is hashed too


def test_phase_stats():
    st = bench.phase_stats([3.0, 1.0, 2.0, 10.0])
    assert st == {"ms_mean": 4.0, "ms_median": 2.5, "ms_min": 1.0, "ms_max": 10.0}
    assert bench.phase_stats([]) == {}


def test_cpu_model_is_a_string():
    m = bench.cpu_model()
    assert isinstance(m, str) and m


def test_cpu_baseline_one_core_figure(monkeypatch):
    monkeypatch.setattr(synth, "square_2048", _small_square)
    res = bench.cpu_oracle_sample(seconds_target=0.0)
    assert res["value_1thread"] > 0 and "one core" in res["sample_1thread"]
    assert isinstance(res["cpu_model"], str)


def test_rank_replica_bounds():
    assert [bench.rank_replica(r) for r in range(8)] == list(range(8))
    for bad in (-1, synth.MAX_REPLICAS):
        with pytest.raises(ValueError):
            bench.rank_replica(bad)

"""Stored calibration (lambda, codebooks) of each workload.

The files under tests/golden/calib are written by tests/golden/make_calib.py,
which calls only the oracle.  Here: shapes and dtypes, and a bit-exact
regeneration of the tiny workload's calibration.
"""
import importlib.util
import os

import numpy as np
import pytest

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _make_calib():
    spec = importlib.util.spec_from_file_location("make_calib", os.path.join(GOLDEN, "make_calib.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("i", sorted(W.WORKLOADS))
def test_artifact_shapes(i):
    w = W.WORKLOADS[i]
    z = np.load(os.path.join(GOLDEN, "calib", f"cfg{i}.npz"))
    assert z["lam"].dtype == np.float32 and z["lam"].shape == (w.num_kv_heads, 128)
    assert np.all(z["lam"] > 0)
    assert z["ck"].dtype == np.float16 and z["ck"].shape == (2 ** w.k_bits, w.k_sub)
    assert z["cv"].dtype == np.float16 and z["cv"].shape == (2 ** w.v_bits, w.v_sub)
    assert np.all(np.isfinite(z["ck"].astype(np.float32)))
    # Lloyd objective never increases
    for o in (z["obj_k"], z["obj_v"]):
        assert len(o) == W.KMEANS_ITERS + 1 and np.all(np.diff(o) <= 1e-9 * o[0])


def test_tiny_workload_calibration_regenerates_bit_exactly():
    mk = _make_calib()
    c = mk.calibrate(W.WORKLOADS[0])
    z = np.load(os.path.join(GOLDEN, "calib", "cfg0.npz"))
    for key in ("lam", "ck", "cv", "obj_k", "obj_v"):
        assert np.array_equal(c[key], z[key]), key


def test_lambda_is_sqrt_of_calibration_max():
    w = W.WORKLOADS[0]
    k_cal, _ = W.calibration(w)
    z = np.load(os.path.join(GOLDEN, "calib", "cfg0.npz"))
    expect = np.sqrt(np.abs(k_cal.astype(np.float64)).max(axis=0)).astype(np.float32)
    assert np.array_equal(z["lam"], expect)

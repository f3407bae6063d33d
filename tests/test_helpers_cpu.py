"""The certified VQ index comparison used by the GPU parity tests, checked on
the CPU with a simulated device result (the oracle's own fp32-rounded Z)."""
import numpy as np
import pytest

import oracle
from pipeline_activation_compression_gb300 import synth
from tests.helpers import check_vq_indices, gpu_residuals


def _sim(n=300):
    w = synth.WORKLOADS["vq_d1024_r128"]
    b = synth.make_boundary(w, n_tokens=n)
    W = synth.widen
    Z = oracle.compress(W(b["X"]), b["tids"], W(b["A"]), W(b["E"]), W(b["P"]))
    Z32 = Z.astype(np.float32)
    C = b["C"]
    # what an exact device would pick for its fp32 residuals
    Cd = W(C)
    idx = np.zeros((n, w.R, w.G), dtype=np.int64)
    for g in range(w.G):
        v = Z32[:, g * w.gd:(g + 1) * w.gd].copy()
        for rho in range(w.R):
            D = ((v.astype(np.float64)[:, None, :] - Cd[rho, g][None]) ** 2).sum(-1)
            idx[:, rho, g] = np.argmin(D, axis=1)
            v = (v - Cd[rho, g][idx[:, rho, g]].astype(np.float32)).astype(np.float32)
    return w, b, Z, Z32, idx


def test_exact_device_passes():
    w, b, Z, Z32, idx = _sim()
    rep = check_vq_indices(idx.astype(np.uint8), Z32, Z, b["C"])
    assert rep["mismatches"] <= 2


def test_wrong_index_is_caught():
    w, b, Z, Z32, idx = _sim()
    bad = idx.copy()
    bad[7, 0, 1] = (bad[7, 0, 1] + 1) % w.K
    with pytest.raises(AssertionError):
        check_vq_indices(bad.astype(np.uint8), Z32, Z, b["C"])


def test_residuals_follow_choices():
    w, b, Z, Z32, idx = _sim(50)
    V = gpu_residuals(Z32, b["C"], idx)
    Cd = synth.widen(b["C"])
    assert np.allclose(V[:, 1, 2], Z[:, 2 * w.gd:3 * w.gd] - Cd[0, 2][idx[:, 0, 2]], atol=1e-5)

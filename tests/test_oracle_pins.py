"""The fp64 oracle against what the MAPL paper and mathematics fix (CPU)."""
import numpy as np
import pytest

import oracle
from pipeline_activation_compression_gb300 import synth, polar
from tests import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


@pytest.mark.parametrize("name", ["tiny_d64_r16", "proj_d1024_r128", "vq_d1024_r128", "vq_d2048_r256"])
def test_generator_orthonormal(name):
    pins.check_generator(name, n_tokens=256)


def test_generator_statistics():
    w = synth.WORKLOADS["vq_d1024_r128"]
    b = synth.make_boundary(w, n_tokens=4096)
    t = b["tids"]
    assert t.dtype == np.int32 and t.min() >= 0 and t.max() < w.V
    # truncated Zipf(1.1): P(0)/P(1) = 2^1.1
    c0, c1 = np.sum(t == 0), np.sum(t == 1)
    assert 1.6 < c0 / c1 < 2.8
    E = synth.widen(b["E"])
    assert abs(E.std() - 0.02) < 0.001
    # X minus its (stored) anchor: unit-RMS rank-250 signal plus 0.05 noise
    X = synth.widen(b["X"])
    res = X - E[t] @ synth.widen(b["P"])
    assert abs(np.sqrt(np.mean(res ** 2)) - np.sqrt(1 + 0.05 ** 2)) < 0.02
    s = np.linalg.svd(res[:2048], compute_uv=False)
    energy = np.cumsum(s ** 2) / np.sum(s ** 2)
    assert energy[249] > 0.99 and energy[200] < 0.99
    # bf16 storage is exact round-to-nearest-even
    x = np.array([1.0, 1.00390625, 1.005859375, -3.3e-3, 0.0], dtype=np.float32)
    bits = synth.bf16_bits(x)
    assert list(bits[:3]) == [0x3F80, 0x3F80, 0x3F81]


def test_generator_deterministic_and_prefix_stable():
    a = synth.make_boundary("tiny_d64_r16")
    b = synth.make_boundary("tiny_d64_r16")
    for k in a:
        assert np.array_equal(a[k], b[k])
    c = synth.make_boundary("proj_d1024_r64", n_tokens=100)
    d = synth.make_boundary("proj_d1024_r64", n_tokens=300)
    assert np.array_equal(c["A"], d["A"]) and np.array_equal(c["E"], d["E"])


def test_polar_coefficients_equioscillate():
    """Polar Express: p_t is the minimax odd quintic on [l, u]; its error
    alternates in sign with equal size at l, two interior points and u, and
    the schedule tends to the quintic with p(1)=1, p'(1)=p''(1)=0."""
    a, b, c, E = polar.minimax_odd_quintic(1e-3, 1.0)
    x = np.linspace(1e-3, 1.0, 200001)
    e = 1 - (a * x + b * x ** 3 + c * x ** 5)
    assert abs(np.max(np.abs(e)) - E) < 1e-9
    ext = [e[0], e[-1], e.min(), e.max()]
    assert abs(ext[0] - E) < 1e-9 and abs(ext[1] + E) < 1e-9
    assert abs(ext[2] + E) < 1e-9 and abs(ext[3] - E) < 1e-9
    sched = polar.polar_express_schedule(8, 1e-3)
    assert np.allclose(sched[-1], polar.NEWTON_SCHULZ_QUINTIC, atol=1e-6)
    # composed map sends [1e-3, 1] close to 1 after 6 steps
    t = np.geomspace(1e-3, 1, 50)
    for (a, b, c) in sched[:6]:
        t = a * t + b * t ** 3 + c * t ** 5
    assert np.max(np.abs(t - 1)) < 1e-3


def test_codebook_sigmas_match_oracle_measurement():
    """The stored per-round codebook std equals the RMS of what each round
    quantises, as measured with the oracle on a 4096-token sample."""
    import json, os
    path = os.path.join(os.path.dirname(__file__), "golden", "codebook_rms.json")
    with open(path) as f:
        meas = json.load(f)
    for name, vals in meas.items():
        w = synth.WORKLOADS[name]
        assert np.allclose(w.code_sigma, vals["sigma"], rtol=0, atol=5e-4), name

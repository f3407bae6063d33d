"""The planted-tie codebooks used by the GPU tie tests, checked with the
oracle alone: each planted decision is the exact tie or the near tie it is
meant to be (CPU)."""
import dataclasses

import numpy as np
import pytest

from pipeline_activation_compression_gb300 import synth
from tests.ties import describe, plant_ties


@pytest.mark.parametrize("name,n", [("vq_d1024_r128", 400), ("vq_d2048_r128", 300)])
def test_planted_ties_are_ties(name, n):
    w = synth.WORKLOADS[name]
    b = synth.make_boundary(w, n_tokens=n)
    C, info, Z = plant_ties(w, b)
    rows = describe(C, info, Z)
    assert len(rows) == w.R * w.G * 48
    for rho, g, tok, kind, a, bb, k, rel, flag in rows:
        assert k in (a, bb), (rho, g, tok, kind)
        if kind == "dup":
            assert k == min(a, bb) and rel == 0.0 and flag
        else:
            assert flag and 1e-9 < rel < 1e-6, (rho, g, tok, rel)

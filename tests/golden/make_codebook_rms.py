"""Measure the per-round codebook std of the bf16 VQ workloads with the oracle.

The workload recipe draws round-rho code entries from N(0, sigma_rho), sigma_rho
being the RMS of what round rho quantises.  This script measures both numbers
with the fp64 oracle on the first 4096 tokens of each workload and writes
``codebook_rms.json`` beside itself; the generator stores the rounded values.

Run: python tests/golden/make_codebook_rms.py
"""
import dataclasses
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from pipeline_activation_compression_gb300 import synth  # noqa: E402

N_SAMPLE = 4096


def measure(name):
    w = synth.WORKLOADS[name]
    b = synth.make_boundary(dataclasses.replace(w, code_sigma=(1.0, 1.0)), n_tokens=N_SAMPLE)
    Z = oracle.compress(synth.widen(b["X"]), b["tids"], synth.widen(b["A"]),
                        synth.widen(b["E"]), synth.widen(b["P"]))
    s1 = float(np.sqrt(np.mean(Z ** 2)))
    b = synth.make_boundary(dataclasses.replace(w, code_sigma=(s1, 1.0)), n_tokens=N_SAMPLE)
    C = synth.widen(b["C"])
    res = oracle.rvq_encode(Z, C[:1])
    s2 = float(np.sqrt(np.mean(res["residual"] ** 2)))
    return [round(s1, 4), round(s2, 4)]


if __name__ == "__main__":
    out = {n: {"sigma": measure(n), "n_sample": N_SAMPLE}
           for n, w in synth.WORKLOADS.items() if w.vq and w.dtype == "bf16"}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "codebook_rms.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
    print(json.dumps(out))

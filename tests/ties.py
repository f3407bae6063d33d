"""Codebooks with planted exact and near ties (test input construction).

§3.5 quantises each group's residual to its nearest code.  Random codebooks
almost never put two codes at (nearly) the same distance, so the two rare
branches of a nearest-code search -- exact ties, which must go to the lowest
index, and gaps so small that fp32 distances cannot order them -- would stay
untested.  ``plant_ties`` rewrites part of a workload's codebook so that, for
chosen tokens, every round's decision is one of:

* ``dup``:  the nearest code appears twice (the copy at a lower or a higher
  index); both copies are at exactly the same distance, so the lowest index
  must win;
* ``near``: the two nearest codes are bf16(v) with one coordinate set to
  either of two adjacent bf16 values, chosen (by search over every bf16
  value near that coordinate) so that their squared distances differ by
  0.5e-7 to 2e-7 of ||v||^2.

Only the oracle (fp64) is used to place the codes: round 0 uses the oracle's
Z, a later round the residual the oracle leaves after the earlier rounds.
Each round plants its ties in tokens of its own.
"""
from __future__ import annotations

import numpy as np

import oracle
from pipeline_activation_compression_gb300 import synth


def _bf16_line() -> np.ndarray:
    """Every finite bf16 value, ascending, as float64."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        v = synth.widen(bits)
    v = np.unique(v[np.isfinite(v)])
    return v


_LINE = None


def _near_pair(v, target):
    """Two adjacent bf16 values (a, b) for one coordinate j of v such that
    the squared distances of the codes bf16(v) with coordinate j set to a or
    to b differ by about ``target`` while both stay as close to v as the
    search allows.  Returns (j, a, b)."""
    global _LINE
    if _LINE is None:
        _LINE = _bf16_line()
    best = None
    span = 0.25 * np.sqrt(float(v @ v) / v.size) + 1e-30
    for j, x in enumerate(v):
        lo = np.searchsorted(_LINE, x - span)
        hi = np.searchsorted(_LINE, x + span)
        a = _LINE[lo:hi - 1]
        b = _LINE[lo + 1:hi]
        gap = np.abs((x - a) ** 2 - (x - b) ** 2)
        cost = np.minimum((x - a) ** 2, (x - b) ** 2)
        ok = (gap > 0.5 * target) & (gap < 2.0 * target)
        if not np.any(ok):
            continue
        k = np.argmin(np.where(ok, cost, np.inf))
        if best is None or cost[k] < best[0]:
            best = (cost[k], j, float(a[k]), float(b[k]))
    assert best is not None, "no bf16 pair gives the requested gap"
    return best[1], best[2], best[3]


def plant_ties(w, b, n_near=32, n_dup=16, seed=3):
    """Return (C_bits, info).  ``info[(rho, g)]`` lists (token, kind, slots)
    with the code slots planted for that token."""
    rng = np.random.default_rng(seed)
    W = synth.widen
    Z = oracle.compress(W(b["X"]), b["tids"], W(b["A"]), W(b["E"]), W(b["P"]))
    C = W(b["C"]).copy()
    R, G, K, gd = C.shape
    N = Z.shape[0]
    need = 2 * (n_near + n_dup)
    assert need <= K, "codebook too small for the planted ties"
    # a separate set of tokens per round: a later round plants its ties in
    # residuals of ordinary size (what a random round-0 code leaves), not in
    # the tiny residual a planted round-0 code leaves
    per = n_near + n_dup
    assert R * per <= N, "too few tokens for the planted ties"
    order = rng.permutation(N)
    kinds = ["near"] * n_near + ["dup"] * n_dup
    info = {}
    u = Z.copy()
    for rho in range(R):
        toks = order[rho * per:(rho + 1) * per]
        for g in range(G):
            cols = slice(g * gd, (g + 1) * gd)
            slots = rng.permutation(K)[:need].reshape(-1, 2)
            entries = []
            for j, (n, kind) in enumerate(zip(toks, kinds)):
                v = u[n, cols]
                lo, hi = int(min(slots[j])), int(max(slots[j]))
                first, second = (lo, hi) if j % 2 == 0 else (hi, lo)
                ca = W(synth.bf16_bits(v.astype(np.float32)))
                if kind == "near":
                    # one coordinate set to either of two adjacent bf16
                    # values: the squared distances differ by ~1e-7 ||v||^2
                    i, a, bv = _near_pair(v, 1e-7 * float(v @ v))
                    ca[i] = a
                    cb = ca.copy()
                    cb[i] = bv
                    C[rho, g, first] = ca
                    C[rho, g, second] = cb
                else:
                    C[rho, g, first] = ca
                    C[rho, g, second] = ca
                entries.append((int(n), kind, (first, second)))
            info[(rho, g)] = entries
            # the residual the oracle carries into the next round
            res = oracle.rvq_encode(u[:, cols], C[rho:rho + 1, g:g + 1])
            u[:, cols] = res["residual"]
    return synth.bf16_bits(C.astype(np.float32)), info, Z


def describe(C_bits, info, Z):
    """Oracle view of the planted decisions: per (rho, g) and kind, the
    relative gaps and whether the planted pair holds the two nearest codes."""
    C = synth.widen(C_bits)
    enc = oracle.rvq_encode(Z, C)
    out = []
    for (rho, g), entries in info.items():
        for n, kind, (a, bb) in entries:
            rel = enc["gap"][n, rho, g] / enc["vnorm2"][n, rho, g]
            out.append((rho, g, n, kind, a, bb, int(enc["idx"][n, rho, g]), float(rel),
                        bool(enc["flag"][n, rho, g])))
    return out

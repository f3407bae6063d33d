"""Seeded synthetic inputs for the MAPL boundary codec.

This module only draws random numbers and stores them in their storage dtype.
It is shared by the fp64 oracle tests and by the CUDA path's tests and bench,
so it deliberately holds none of the codec's own arithmetic (no projection, no
quantisation, no reconstruction): every tensor here is an *input*.

Workload recipe (stated in full so it can be re-derived):

* ``tids``: int32.  Uniform on [0, V) for the tiny workload; otherwise a
  truncated Zipf(1.1) law, P(id = k) proportional to (k+1)^-1.1 for k in
  [0, V), sampled by inverse CDF (id 0 is the most frequent token).
* ``A`` in St(d, r): Q factor of the thin QR of a d x r N(0,1) matrix, signs
  fixed so that diag(R) > 0.  ``P`` (r x d, orthonormal rows): transpose of the
  Q factor of an independent d x r draw.  Same for the receiving stage's P'.
* ``E`` / ``E'`` (V x r): N(0, 0.02) entries (0.02 is a standard deviation).
* ``X`` (N x d): the sending stage's anchor rows ``E[tids] P`` plus a rank-R
  signal ``S W / rms(S W)`` (S: N x R, W: R x d, both N(0,1)) plus
  ``0.05 * N(0,1)`` noise.  The tiny workload instead uses
  ``E[tids] P + S W + 0.01 * N(0,1)`` with S: N x r N(0,1), W: r x d N(0,1)/8.
  The anchor term is part of how the synthetic activation is *made*; the codec
  later has to remove it.
* Codebooks ``C`` (R x G x K x gd): round rho entries are N(0, sigma_rho).
  For the tiny workload sigma = 0.5 for every round.  For the bf16 VQ
  workloads sigma_rho is the RMS of what round rho quantises (the projected
  residual for rho = 0, the round-1 residual for rho = 1); those two numbers
  were measured once with the fp64 oracle on a 4096-token sample of each
  workload by ``tests/golden/make_codebook_rms.py`` and are stored below.
* First boundary (``make_first_boundary``): the anchor is a full V x d token
  embedding ``E_emb`` with N(0, 1) entries; ``X = E_emb[tids]`` + the same
  kind of unit-RMS rank-R signal + ``0.05 * N(0,1)`` noise, drawn from a
  stream of their own; tids, A and C are those of ``make_boundary``.
* SPEL gradients: N(0, 1e-3) entries, a fresh draw each step.

Storage: fp32 workloads keep every tensor in float32.  bf16 workloads round
X, A, P, E, P', E' and C to bfloat16 once (round to nearest even) and keep the
bit patterns as uint16; ``widen`` turns them back into exact float64 values.

Every tensor draws from its own child of ``numpy.random.SeedSequence(seed)``
in a fixed order, so changing one size never changes another tensor's values.
"""
from __future__ import annotations

import dataclasses
import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "SPEL_WORKLOADS", "SpelWorkload", "make_boundary",
    "make_first_boundary", "make_spel", "spel_gradients", "bf16_bits", "bf16_to_f64", "widen",
]

# order of the SeedSequence children; never reorder (it would change inputs)
_STREAMS = ("tids", "E", "P", "A", "E_next", "P_next", "S", "W", "noise",
            "C", "G", "m0")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    d: int
    r: int
    V: int
    B: int
    T: int
    dtype: str                 # "f32" or "bf16" storage / compute dtype
    G: int = 0                 # VQ groups (0: no VQ, Z is the payload)
    R: int = 0                 # residual rounds
    K: int = 0                 # codes per group per round
    signal_rank: int = 250
    tids_law: str = "zipf"     # "zipf" or "uniform"
    tiny_recipe: bool = False  # the tiny workload's own X formula
    code_sigma: tuple = ()     # per-round codebook std

    @property
    def N(self) -> int:
        return self.B * self.T

    @property
    def vq(self) -> bool:
        return self.G > 0

    @property
    def gd(self) -> int:
        return self.r // self.G if self.G else 0


# Per-round codebook std for the bf16 VQ workloads (see module docstring).
_SIGMA_D1024_R128 = (0.9929, 0.9813)
_SIGMA_D2048_R128 = (1.0008, 0.8235)
_SIGMA_D2048_R256 = (1.0022, 0.9899)

WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_d64_r16", d=64, r=16, V=512, B=4, T=32, dtype="f32",
                 G=1, R=2, K=16, tids_law="uniform", tiny_recipe=True,
                 code_sigma=(0.5, 0.5)),
        Workload("proj_d1024_r64", 1024, 64, 32000, 8, 2048, "bf16"),
        Workload("proj_d1024_r128", 1024, 128, 32000, 8, 2048, "bf16"),
        Workload("proj_d1024_r256", 1024, 256, 32000, 8, 2048, "bf16"),
        Workload("proj_d1024_r512", 1024, 512, 32000, 8, 2048, "bf16"),
        Workload("vq_d1024_r128", 1024, 128, 32000, 16, 2048, "bf16",
                 G=4, R=2, K=256, code_sigma=_SIGMA_D1024_R128),
        Workload("vq_d2048_r128", 2048, 128, 32000, 8, 2048, "bf16",
                 G=8, R=2, K=256, signal_rank=500,
                 code_sigma=_SIGMA_D2048_R128),
        Workload("vq_d2048_r256", 2048, 256, 32000, 8, 2048, "bf16",
                 G=8, R=2, K=256, signal_rank=500,
                 code_sigma=_SIGMA_D2048_R256),
    ]
}


@dataclasses.dataclass(frozen=True)
class SpelWorkload:
    name: str
    d: int
    r: int
    batch: int
    lr: float = 2e-3
    beta: float = 0.9
    grad_std: float = 1e-3


SPEL_WORKLOADS = {
    w.name: w for w in [
        SpelWorkload("spel_d1024_r256", 1024, 256, 3),
        SpelWorkload("spel_d2048_r256", 2048, 256, 3),
    ]
}


# ----------------------------------------------------------------------------
# storage helpers (no method arithmetic: only rounding to the storage format)
# ----------------------------------------------------------------------------
def bf16_bits(x) -> np.ndarray:
    """Round to bfloat16 (nearest, ties to even) and return uint16 bit patterns."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(f)
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def widen(t) -> np.ndarray:
    """Exact float64 value of a stored tensor (uint16 means bf16 bits)."""
    t = np.asarray(t)
    if t.dtype == np.uint16:
        return bf16_to_f64(t)
    return t.astype(np.float64)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits(x)
    return np.ascontiguousarray(x, dtype=np.float32)


def _rngs(seed: int) -> dict:
    kids = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    return {n: np.random.Generator(np.random.PCG64(k)) for n, k in zip(_STREAMS, kids)}


def _orthonormal_cols(rng, d: int, r: int) -> np.ndarray:
    q, rr = np.linalg.qr(rng.standard_normal((d, r)))
    s = np.sign(np.diag(rr))
    s[s == 0] = 1.0
    return q * s


def _draw_tids(rng, n: int, V: int, law: str) -> np.ndarray:
    if law == "uniform":
        return rng.integers(0, V, size=n, dtype=np.int64).astype(np.int32)
    w = np.arange(1, V + 1, dtype=np.float64) ** -1.1
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng.random(n)
    t = np.searchsorted(cdf, u, side="right")
    return np.minimum(t, V - 1).astype(np.int32)


def make_boundary(w: Workload | str, seed: int = 0, n_tokens: int | None = None) -> dict:
    """All inputs of one boundary crossing, in storage dtype.

    Returns a dict with X (N x d), tids (N,), A (d x r), P (r x d), E (V x r),
    P_next (r x d), E_next (V x r) and, for VQ workloads, C (R x G x K x gd).
    ``n_tokens`` overrides B*T (same recipe, other size).
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    n = w.N if n_tokens is None else int(n_tokens)
    g = _rngs(seed)
    d, r, V = w.d, w.r, w.V
    tids = _draw_tids(g["tids"], n, V, w.tids_law)
    E = 0.02 * g["E"].standard_normal((V, r))
    P = _orthonormal_cols(g["P"], d, r).T.copy()
    A = _orthonormal_cols(g["A"], d, r)
    E_next = 0.02 * g["E_next"].standard_normal((V, r))
    P_next = _orthonormal_cols(g["P_next"], d, r).T.copy()

    st = lambda x: _store(x, w.dtype)
    E_s, P_s, A_s, En_s, Pn_s = st(E), st(P), st(A), st(E_next), st(P_next)

    # activation = stored anchor rows of the sending stage + signal + noise
    anchor = widen(E_s)[tids] @ widen(P_s)
    if w.tiny_recipe:
        S = g["S"].standard_normal((n, r))
        W = g["W"].standard_normal((r, d)) / 8.0
        X = anchor + S @ W + 0.01 * g["noise"].standard_normal((n, d))
    else:
        k = w.signal_rank
        S = g["S"].standard_normal((n, k))
        W = g["W"].standard_normal((k, d))
        sig = S @ W
        rms = np.sqrt(np.mean(sig * sig)) if sig.size else 1.0
        X = anchor + sig / rms + 0.05 * g["noise"].standard_normal((n, d))
    out = dict(X=st(X), tids=tids, A=A_s, P=P_s, E=E_s, P_next=Pn_s, E_next=En_s,
               A_f64=A, P_f64=P, P_next_f64=P_next)
    if w.vq:
        C = np.empty((w.R, w.G, w.K, w.gd))
        for rho in range(w.R):
            C[rho] = w.code_sigma[rho] * g["C"].standard_normal((w.G, w.K, w.gd))
        out["C"] = st(C)
    return out


def make_boundary_grad(w: Workload | str, seed: int = 0, n_tokens: int | None = None,
                       scale: float = 0.01) -> np.ndarray:
    """Gradient arriving at the boundary in the backward pass, dL/dX_hat
    (N x d, storage dtype): scale * N(0, 1), from its own seeded stream
    (independent of make_boundary's tensors for the same seed)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    n = w.N if n_tokens is None else int(n_tokens)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7, 1]).spawn(1)[0]))
    return _store(scale * rng.standard_normal((n, w.d)), w.dtype)


def make_grad_codebooks(w: Workload | str, seed: int = 0, scale: float = 0.01) -> np.ndarray:
    """Codebooks for the MCVQ of backward gradients (R x G x K x gd, storage
    dtype), from their own seeded stream.  The boundary gradient of
    ``make_boundary_grad`` has N(0, scale) entries and A has orthonormal
    columns, so gZ = dL/dX_hat A has N(0, scale) entries too: round 0 codes
    are N(0, scale), and later rounds shrink by the ratio the forward books
    of the workload use between their rounds (code_sigma)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7, 2]).spawn(1)[0]))
    C = np.empty((w.R, w.G, w.K, w.gd))
    for rho in range(w.R):
        ratio = w.code_sigma[rho] / w.code_sigma[0] if w.code_sigma else 1.0
        C[rho] = scale * ratio * rng.standard_normal((w.G, w.K, w.gd))
    return _store(C, w.dtype)


def make_first_boundary(w: Workload | str, seed: int = 0, n_tokens: int | None = None,
                        emb_std: float = 1.0) -> dict:
    """Inputs of the first boundary, where the anchor is the full token
    embedding (V x d) rather than a low-rank factor.

    Same shapes, token law, projector and codebooks as ``make_boundary`` for
    the same seed; E_emb ~ emb_std * N(0, 1) from its own seeded stream, and
    X = E_emb[tids] + signal (unit RMS, rank ``signal_rank``) + 0.05 noise:
    right after the first stage the residual stream still carries the
    embedding at full strength.  Returns X, tids, A, E_emb (and C with VQ).
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    base = make_boundary(w, seed=seed, n_tokens=n_tokens)
    n = base["X"].shape[0]
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 11, 1]).spawn(1)[0]))
    st = lambda x: _store(x, w.dtype)
    E_emb = st(emb_std * rng.standard_normal((w.V, w.d)))
    k = min(w.signal_rank, w.d)
    sig = rng.standard_normal((n, k)) @ rng.standard_normal((k, w.d))
    rms = np.sqrt(np.mean(sig * sig)) if sig.size else 1.0
    X = widen(E_emb)[base["tids"]] + sig / rms + 0.05 * rng.standard_normal((n, w.d))
    out = dict(X=st(X), tids=base["tids"], A=base["A"], E_emb=E_emb)
    if w.vq:
        out["C"] = base["C"]
    return out


def make_spel(w: SpelWorkload | str, seed: int = 0) -> dict:
    """Initial projectors (batch x d x r, on St(d,r)) and zero momentum, fp32."""
    if isinstance(w, str):
        w = SPEL_WORKLOADS[w]
    g = _rngs(seed)
    A = np.stack([_orthonormal_cols(g["A"], w.d, w.r) for _ in range(w.batch)])
    return dict(A=A.astype(np.float32), m=np.zeros_like(A, dtype=np.float32))


def spel_gradients(w: SpelWorkload | str, seed: int = 0):
    """Endless stream of fresh Euclidean gradients, N(0, grad_std), fp32."""
    if isinstance(w, str):
        w = SPEL_WORKLOADS[w]
    rng = _rngs(seed)["G"]
    while True:
        yield (w.grad_std * rng.standard_normal((w.batch, w.d, w.r))).astype(np.float32)


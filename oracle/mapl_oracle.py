"""Plain fp64 CPU oracle of the MAPL boundary codec and of the SPEL step.

TEST INFRASTRUCTURE ONLY.  This module is the independent reference that the
CUDA library is checked against.  Only the test-suite, the package smoke check
and the benchmark's CPU-baseline leg may import it; the library itself never
does, and it shares no code with the CUDA path (no kernels, headers, helpers,
tables or constants).  Inputs come from the shared seeded generator.

Source: *Learned Subspace Compression for Communication-Efficient Pipeline
Parallelism* (MAPL).  Every function names the passage it writes out:

* anchor            -- §3.2, eq. (3): E_small[ids] P
* compress          -- §3.2, eq. (1): Z = (X - E_small[ids] P) A
* reconstruct       -- §3.2, eq. (2): X_hat = Z A^T + E_small_next[ids] P_next
* compress_embed    -- Fig. 2 caption: at the first boundary the anchor is the
                       original token embedding, Z = (X - E_emb[ids]) A
* reconstruct_embed -- its receiver side, X_hat = Z A^T + E_emb[ids]
* grad_A_embed      -- Euclidean gradient of A for that first-boundary codec
* grad_compress     -- §3.2 (backward pass): the boundary gradient dL/dX_hat
                       routed through the same projector, gZ = dL/dX_hat A
* grad_decompress   -- §3.2 (backward pass): dL/dX = gZ A^T
* grad_A            -- Euclidean gradient of A that §3.3 feeds to SPEL, for the
                       composed codec X_hat = (X - E[ids] P) A A^T + E'[ids] P'
* stream_subset     -- §3.5 / App. F streaming codebook synchronisation: the
                       random subset of codes refreshed at a micro-batch
* apply_code_update -- §3.5 / App. F: the shared codebook after a refresh
* rvq_encode/decode -- §3.5 "Composing with vector quantization" and App. E.4:
                       G groups, R rounds of residual quantisation, K codes
* tangent_project   -- §3.3, eq. (4): g - A sym(A^T g), sym(M) = (M + M^T)/2
* momentum          -- §3.3, eq. (5): beta m + (1 - beta) g_R
* polar_express     -- §3.3, eqs. (6)-(7): odd matrix polynomial iterations
* spel_step         -- §3.3, Algorithm 1 step 4 (eqs. (4)-(7) in order)

Readings where the pages leave a step open (each also listed in the design
notes):

* Codebook layout: per round and per group, C[rho][g] is K x gd with gd = r/G
  (§3.5 prints one r x K codebook per stage; read column-wise it is G stacked
  gd x K sub-codebooks; separate codebooks per round).
* Nearest code: squared Euclidean distance, brute force over all K codes;
  exact ties go to the lowest index.  Group g's residual only ever involves
  group g's columns, so groups are independent.
* Near-tie flag: the gap between the best and second-best distance is below
  ``rel_tie * ||v||^2`` where v is the vector being quantised (the group's
  residual in that round).
* PolarExpress: the pages give iteration counts, not coefficients.  The
  polynomial is an input: a list of (a, b, c) with Y <- Y (a I + b S + c S^2),
  S = Y^T Y, applied in order.  The LMO input is scaled by its Frobenius norm
  (plus 1e-7) first; the retraction input is not scaled.
* Momentum is not re-projected onto the new tangent space (Algorithm 1 does
  not do so).
* The learning rate alpha multiplies the LMO direction d (eq. (7)).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "anchor", "compress", "compress_folded", "reconstruct", "compress_embed",
    "reconstruct_embed", "grad_A_embed", "grad_compress",
    "grad_decompress", "grad_A", "grad_A_given", "stream_subset", "apply_code_update",
    "splitmix64", "rvq_encode",
    "rvq_encode_given", "rvq_decode", "tangent_project", "sym", "momentum",
    "polar_express", "spel_step", "payload_bytes_per_token",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# boundary codec, §3.2
# ---------------------------------------------------------------------------
def anchor(E, P, tids) -> np.ndarray:
    """Factorised anchor of eq. (3): row n is E_small[tids[n]] @ P (N x d)."""
    E, P = _f64(E), _f64(P)
    tids = np.asarray(tids, dtype=np.int64)
    return E[tids] @ P


def compress(X, tids, A, E, P) -> np.ndarray:
    """Sender side, eq. (1): Z = (X - E_small[tids] P) A, N x r.

    Written literally: the anchor is formed in full (N x d) and subtracted
    before the projection.
    """
    X, A = _f64(X), _f64(A)
    return (X - anchor(E, P, tids)) @ A


def compress_folded(X, tids, A, E, P) -> np.ndarray:
    """The same Z with the anchor folded through M = P A (r x r):
    Z = X A - E_small[tids] (P A).  An algebraic identity of eq. (1), kept
    only so the tests can check that both groupings agree."""
    X, A, E, P = _f64(X), _f64(A), _f64(E), _f64(P)
    M = P @ A
    return X @ A - E[np.asarray(tids, dtype=np.int64)] @ M


def reconstruct(Zhat, tids, A, E_next, P_next) -> np.ndarray:
    """Receiver side, eq. (2): X_hat = Z A^T + E_small_{p+1}[tids] P_{p+1}."""
    Zhat, A = _f64(Zhat), _f64(A)
    return Zhat @ A.T + anchor(E_next, P_next, tids)


# ---------------------------------------------------------------------------
# first boundary, Fig. 2: the anchor is the full token embedding
# ---------------------------------------------------------------------------
def compress_embed(X, tids, A, E_emb) -> np.ndarray:
    """Sender side at the first boundary: Z = (X - E_emb[tids]) A, with the
    V x d embedding table itself as the anchor (no low-rank factor)."""
    X, A, E_emb = _f64(X), _f64(A), _f64(E_emb)
    return (X - E_emb[np.asarray(tids, dtype=np.int64)]) @ A


def reconstruct_embed(Zhat, tids, A, E_emb) -> np.ndarray:
    """Receiver side at the first boundary: X_hat = Z A^T + E_emb[tids]."""
    Zhat, A, E_emb = _f64(Zhat), _f64(A), _f64(E_emb)
    return Zhat @ A.T + E_emb[np.asarray(tids, dtype=np.int64)]


def grad_A_embed(X, tids, E_emb, gZ, gXhat, Z) -> np.ndarray:
    """dL/dA for X_hat = (X - E_emb[tids]) A A^T + E_emb[tids], given the
    gradient gZ of Z and Z itself: X_res^T gZ + gX_hat^T Z with
    X_res = X - E_emb[tids]."""
    Xres = _f64(X) - _f64(E_emb)[np.asarray(tids, dtype=np.int64)]
    return Xres.T @ _f64(gZ) + _f64(gXhat).T @ _f64(Z)


# ---------------------------------------------------------------------------
# backward pass, §3.2 ("we symmetrically route the gradient through the same
# orthogonal projector")
# ---------------------------------------------------------------------------
def grad_compress(gXhat, A) -> np.ndarray:
    """Receiver side of the backward pass: gZ = dL/dX_hat A (N x r).  Since
    X_hat = Z A^T + (anchor, independent of Z), dL/dZ = dL/dX_hat A."""
    return _f64(gXhat) @ _f64(A)


def grad_decompress(gZ, A) -> np.ndarray:
    """Sender side: dL/dX = gZ A^T (N x d).  Z = (X - anchor) A, so
    dL/dX = dL/dZ A^T."""
    return _f64(gZ) @ _f64(A).T


def grad_A_given(X, tids, E, P, gZ, gXhat, Z) -> np.ndarray:
    """dL/dA = X_res^T gZ + gX_hat^T Z with X_res = X - E[tids] P, for given
    gZ (the gradient of Z) and Z (d x r): the two places A appears in
    X_hat = X_res A A^T + E'[tids] P'."""
    Xres = _f64(X) - anchor(E, P, tids)
    return Xres.T @ _f64(gZ) + _f64(gXhat).T @ _f64(Z)


def grad_A(X, tids, A, E, P, gXhat) -> np.ndarray:
    """Euclidean gradient of L = <dL/dX_hat, X_hat(A)> with respect to A for
    X_hat = (X - E[tids] P) A A^T + E'[tids] P' (the anchor' term does not
    involve A): X_res^T (gX_hat A) + gX_hat^T (X_res A)."""
    Xres = _f64(X) - anchor(E, P, tids)
    A, g = _f64(A), _f64(gXhat)
    return Xres.T @ (g @ A) + g.T @ (Xres @ A)


# ---------------------------------------------------------------------------
# multi-codebook residual vector quantisation, §3.5
# ---------------------------------------------------------------------------
def _nearest(v, Cg):
    """Brute-force nearest code for each row of v (n x gd) among the rows of
    Cg (K x gd).  Returns (index, best distance, second-best distance)."""
    n = v.shape[0]
    K = Cg.shape[0]
    idx = np.empty(n, dtype=np.int64)
    d1 = np.empty(n)
    d2 = np.full(n, np.inf)
    step = max(1, 4_000_000 // max(1, K * Cg.shape[1]))
    for s in range(0, n, step):
        diff = v[s:s + step, None, :] - Cg[None, :, :]
        D = np.einsum("nkj,nkj->nk", diff, diff)          # squared distances
        k = np.argmin(D, axis=1)                          # first index on ties
        idx[s:s + step] = k
        rows = np.arange(D.shape[0])
        d1[s:s + step] = D[rows, k]
        if K > 1:
            D[rows, k] = np.inf
            d2[s:s + step] = D.min(axis=1)
    return idx, d1, d2


def rvq_encode(Z, C, rel_tie: float = 1e-6):
    """Residual VQ of Z (N x r) with codebooks C (R x G x K x gd).

    For each round rho and group g the group's current residual v is replaced
    by v - C[rho][g][k*], k* = argmin_k ||v - C[rho][g][k]||^2.

    Returns dict(idx (N,R,G) int64, flag (N,R,G) bool near-tie flags,
    gap (N,R,G) second-best minus best distance, vnorm2 (N,R,G) ||v||^2,
    residual (N x r) what is left after the last round).
    """
    return rvq_encode_given(Z, C, None, rel_tie)


def rvq_encode_given(Z, C, idx_given=None, rel_tie: float = 1e-6):
    """Like ``rvq_encode`` but, when ``idx_given`` (N,R,G) is passed, the
    residual carried into round rho+1 uses idx_given[:, rho] instead of the
    oracle's own choice.  Each round's argmin, gap and flag are still the
    oracle's own, computed from that residual.  This lets a test check every
    round of another implementation even after a legitimate near-tie
    disagreement in an earlier round."""
    Z, C = _f64(Z), _f64(C)
    R, G, K, gd = C.shape
    N = Z.shape[0]
    if Z.shape[1] != G * gd:
        raise ValueError("Z width must be G * gd")
    u = Z.copy()
    idx = np.zeros((N, R, G), dtype=np.int64)
    gap = np.zeros((N, R, G))
    vn = np.zeros((N, R, G))
    for rho in range(R):
        for g in range(G):
            cols = slice(g * gd, (g + 1) * gd)
            v = u[:, cols]
            k, d1, d2 = _nearest(v, C[rho, g])
            idx[:, rho, g] = k
            gap[:, rho, g] = d2 - d1
            vn[:, rho, g] = np.einsum("nj,nj->n", v, v)
            take = k if idx_given is None else np.asarray(idx_given)[:, rho, g].astype(np.int64)
            u[:, cols] = v - C[rho, g][take]
    flag = gap < rel_tie * vn
    return dict(idx=idx, flag=flag, gap=gap, vnorm2=vn, residual=u)


def rvq_decode(idx, C) -> np.ndarray:
    """Z_hat[n, g-block] = sum over rounds of C[rho][g][idx[n, rho, g]]."""
    C = _f64(C)
    idx = np.asarray(idx, dtype=np.int64)
    R, G, K, gd = C.shape
    N = idx.shape[0]
    Zh = np.zeros((N, G * gd))
    for rho in range(R):
        for g in range(G):
            Zh[:, g * gd:(g + 1) * gd] += C[rho, g][idx[:, rho, g]]
    return Zh


def payload_bytes_per_token(r: int, dtype_bytes: int = 2, G: int = 0, R: int = 0,
                            K: int = 0) -> float:
    """Bytes crossing the boundary per token (token id excluded).

    Without VQ the payload is Z: r numbers of ``dtype_bytes`` (§3.2: the
    compression ratio is exactly r/d of the d-wide activation).  With VQ it
    is R*G indices of ceil(log2 K) bits.
    """
    if G:
        return R * G * int(np.ceil(np.log2(max(K, 2)))) / 8.0
    return float(dtype_bytes * r)


# ---------------------------------------------------------------------------
# streaming codebook synchronisation, §3.5 and App. F
# ---------------------------------------------------------------------------
_M64 = (1 << 64) - 1


def splitmix64(state: int):
    """One step of splitmix64 (Steele, Lea and Flood 2014, with the constants
    of Vigna's reference implementation): returns (output, new state)."""
    state = (state + 0x9E3779B97F4A7C15) & _M64
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31), state


def stream_subset(total: int, per_batch: int, seed: int, step: int) -> np.ndarray:
    """Codes refreshed at micro-batch `step`.  Reading of App. F ("the codebook
    is partitioned into random subsets"): epoch e = step // n_sub (n_sub =
    ceil(total / per_batch)) shuffles the flat code ids 0..total-1 with
    Fisher-Yates (for i from total-1 down to 1, swap i with j = u_i mod
    (i + 1)), the u_i drawn from splitmix64 seeded with
    seed XOR (0xD1B54A32D192ED03 * (e + 1)); the step takes block
    step % n_sub of per_batch consecutive entries."""
    n_sub = -(-total // per_batch)
    epoch, blk = divmod(step, n_sub)
    perm = list(range(total))
    state = (seed ^ ((0xD1B54A32D192ED03 * (epoch + 1)) & _M64)) & _M64
    for i in range(total - 1, 0, -1):
        u, state = splitmix64(state)
        j = u % (i + 1)
        perm[i], perm[j] = perm[j], perm[i]
    return np.asarray(perm[blk * per_batch:(blk + 1) * per_batch], dtype=np.int64)


def apply_code_update(C, ids, codes) -> np.ndarray:
    """The shared codebook after a refresh: flat code ids[i] (over R x G x K)
    take the values codes[i] (gd entries); every other code is unchanged."""
    C = _f64(C).copy()
    R, G, K, gd = C.shape
    flat = C.reshape(R * G * K, gd)
    flat[np.asarray(ids, dtype=np.int64)] = _f64(codes)
    return flat.reshape(R, G, K, gd)


# ---------------------------------------------------------------------------
# SPEL projector update, §3.3 eqs. (4)-(7)# ---------------------------------------------------------------------------
# SPEL projector update, §3.3 eqs. (4)-(7)
# ---------------------------------------------------------------------------
def sym(M) -> np.ndarray:
    """sym(M) = (M + M^T) / 2 (§3.3)."""
    M = _f64(M)
    return 0.5 * (M + M.T)


def tangent_project(A, g) -> np.ndarray:
    """eq. (4): g_R = g - A sym(A^T g)."""
    A, g = _f64(A), _f64(g)
    return g - A @ sym(A.T @ g)


def momentum(m, gR, beta: float) -> np.ndarray:
    """eq. (5): m <- beta m + (1 - beta) g_R."""
    return beta * _f64(m) + (1.0 - beta) * _f64(gR)


def polar_express(Y, coeffs) -> np.ndarray:
    """Odd matrix polynomial iterations Y <- Y (a I + b S + c S^2), S = Y^T Y,
    one (a, b, c) per iteration, in the given order (eqs. (6)-(7))."""
    Y = _f64(Y).copy()
    I = np.eye(Y.shape[1])
    for a, b, c in coeffs:
        S = Y.T @ Y
        Y = Y @ (a * I + b * S + c * (S @ S))
    return Y


def spel_step(A, g, m, lr: float, beta: float, coeffs_lmo, coeffs_retr):
    """One SPEL update of one projector (Algorithm 1, step 4).

    Returns (A_new, m_new, d) with d the LMO direction of eq. (6).
    """
    gR = tangent_project(A, g)
    m_new = momentum(m, gR, beta)
    nrm = np.linalg.norm(m_new)
    d = polar_express(m_new / (nrm + 1e-7), coeffs_lmo)
    A_new = polar_express(_f64(A) - lr * d, coeffs_retr)
    return A_new, m_new, d

"""Pins of the fp64 oracle to facts the MAPL paper and mathematics fix.

Each pin takes the oracle module ``o`` so that the mutation tests can run the
same pins against an oracle with a planted mistake and show that some pin
fails.  Every pin states the fact it relies on; none re-types the oracle's own
formula.
"""
from __future__ import annotations

import numpy as np
from scipy.spatial import cKDTree

from pipeline_activation_compression_gb300 import synth


def _orth(rng, d, r):
    q, _ = np.linalg.qr(rng.standard_normal((d, r)))
    return q


# ---------------------------------------------------------------- §3.2 codec
def pin_exact_reconstruction(o):
    """§3.2: A^T is the exact inverse of A on col(A).  If X - anchor lies in
    span(A) (X = E[t] P + S A^T) and the receiver uses the same anchor, the
    codec returns X, and Z equals the coordinates S."""
    rng = np.random.default_rng(1)
    d, r, V, n = 48, 12, 37, 64
    A = _orth(rng, d, r)
    P = _orth(rng, d, r).T
    E = rng.standard_normal((V, r))
    S = rng.standard_normal((n, r))
    t = rng.integers(0, V, n)
    X = np.stack([E[t[i]] @ P for i in range(n)]) + S @ A.T
    Z = o.compress(X, t, A, E, P)
    assert np.max(np.abs(Z - S)) < 1e-12
    Xh = o.reconstruct(Z, t, A, E, P)
    assert np.linalg.norm(Xh - X) / np.linalg.norm(X) < 1e-12


def pin_anchor_one_hot(o):
    """eq. (3): with one-hot anchor rows E[v] = e_{j(v)}, the anchor of token v
    is row j(v) of P, the receiver adds row j(v) of P_next, and Z of a zero
    activation is minus that row projected."""
    rng = np.random.default_rng(2)
    d, r, V = 20, 5, 9
    P = rng.standard_normal((r, d))
    Pn = rng.standard_normal((r, d))
    A = _orth(rng, d, r)
    E = np.zeros((V, r))
    j = (np.arange(V) * 3) % r
    E[np.arange(V), j] = 1.0
    t = np.array([0, 4, 8, 1, 1, 7])
    an = o.anchor(E, P, t)
    assert np.array_equal(an, P[j[t]])
    Xh = o.reconstruct(np.zeros((len(t), r)), t, A, E, Pn)
    assert np.array_equal(Xh, Pn[j[t]])
    Z = o.compress(np.zeros((len(t), d)), t, A, E, P)
    assert np.max(np.abs(Z + P[j[t]] @ A)) < 1e-12


def pin_isometry(o):
    """§3.2: projection and reconstruction are isometric on col(A):
    ||Z A^T||_F = ||Z||_F for any Z (zero anchor at the receiver), and
    compressing Z A^T returns Z."""
    rng = np.random.default_rng(3)
    d, r, n = 40, 7, 30
    A = _orth(rng, d, r)
    Z = rng.standard_normal((n, r))
    E0 = np.zeros((3, r))
    P0 = np.zeros((r, d))
    t = np.zeros(n, dtype=np.int64)
    Xh = o.reconstruct(Z, t, A, E0, P0)
    assert abs(np.linalg.norm(Xh) - np.linalg.norm(Z)) < 1e-12 * np.linalg.norm(Z)
    assert np.max(np.abs(o.compress(Xh, t, A, E0, P0) - Z)) < 1e-12


def pin_projection_against_lstsq(o):
    """With a zero anchor, Z holds the least-squares coordinates of X in the
    orthonormal basis A (numpy.linalg.lstsq, a library routine), because
    A^T A = I makes the normal equations read Z = X A."""
    rng = np.random.default_rng(4)
    d, r, n = 33, 6, 17
    A = _orth(rng, d, r)
    X = rng.standard_normal((n, d))
    t = np.zeros(n, dtype=np.int64)
    Z = o.compress(X, t, A, np.zeros((1, r)), np.zeros((r, d)))
    ref = np.linalg.lstsq(A, X.T, rcond=None)[0].T
    assert np.max(np.abs(Z - ref)) < 1e-12


def pin_fold(o):
    """Folding the anchor through M = P A is an algebraic identity of eq. (1)."""
    rng = np.random.default_rng(5)
    d, r, V, n = 64, 16, 50, 40
    X = rng.standard_normal((n, d))
    A = _orth(rng, d, r)
    P = rng.standard_normal((r, d))
    E = rng.standard_normal((V, r))
    t = rng.integers(0, V, n)
    a = o.compress(X, t, A, E, P)
    b = o.compress_folded(X, t, A, E, P)
    assert np.max(np.abs(a - b)) < 1e-12 * max(1.0, np.max(np.abs(a)))


def pin_payload(o):
    """Table 1 and Fig. 1: at d = 1024 the uncompressed bf16 boundary is 2048
    B/token; MAPL at r = 256 sends 512 B (4x); r = 64...512 gives 128...1024
    B; MAPL+VQ (K = 256, R = 2, group size 2 at r = 256) sends 256 B (8x)."""
    assert o.payload_bytes_per_token(r=1024) == 2048
    assert o.payload_bytes_per_token(r=256) == 512
    assert [o.payload_bytes_per_token(r=x) for x in (64, 128, 256, 512)] == [128, 256, 512, 1024]
    assert o.payload_bytes_per_token(r=256, G=128, R=2, K=256) == 256
    # compression ratio r/d (§3.2)
    assert o.payload_bytes_per_token(r=128) / o.payload_bytes_per_token(r=1024) == 128 / 1024


# ------------------------------------------------------------------ §3.5 RVQ
def pin_rvq_nearest_kdtree(o):
    """R = 1, G = 1 is textbook nearest-neighbour search: agree with a
    KD-tree query (scipy, a library routine)."""
    rng = np.random.default_rng(6)
    n, K, gd = 300, 40, 5
    C = rng.standard_normal((1, 1, K, gd))
    Z = rng.standard_normal((n, gd))
    res = o.rvq_encode(Z, C)
    dist, ref = cKDTree(C[0, 0]).query(Z, k=2)
    assert np.array_equal(res["idx"][:, 0, 0], ref[:, 0])
    assert np.allclose(res["gap"][:, 0, 0], dist[:, 1] ** 2 - dist[:, 0] ** 2, atol=1e-10)
    assert np.allclose(Z - C[0, 0][ref[:, 0]], res["residual"], atol=0)


def pin_rvq_sort_ranking(o):
    """Multi-group, multi-round encode equals an independent ranking that
    sorts the expanded distances ||c||^2 - 2 v.c (+ ||v||^2) with a stable sort
    (first index on ties), group by group, round by round."""
    rng = np.random.default_rng(7)
    n, R, G, K, gd = 200, 3, 4, 16, 3
    C = rng.standard_normal((R, G, K, gd))
    Z = rng.standard_normal((n, G * gd)) * 2
    res = o.rvq_encode(Z, C)
    u = Z.copy()
    for rho in range(R):
        for g in range(G):
            v = u[:, g * gd:(g + 1) * gd]
            D = (C[rho, g] ** 2).sum(1)[None, :] - 2 * v @ C[rho, g].T
            k = np.argsort(D, axis=1, kind="stable")[:, 0]
            assert np.array_equal(res["idx"][:, rho, g], k)
            u[:, g * gd:(g + 1) * gd] = v - C[rho, g][k]
    assert np.max(np.abs(u - res["residual"])) < 1e-12


def pin_rvq_special_cases(o):
    """K = 1 always picks code 0; a codebook holding v exactly picks it with
    zero distance and leaves a zero residual; duplicated codes resolve to the
    lowest index and are flagged as ties."""
    rng = np.random.default_rng(8)
    Z = rng.standard_normal((10, 6))
    C1 = rng.standard_normal((2, 2, 1, 3))
    r1 = o.rvq_encode(Z, C1)
    assert np.all(r1["idx"] == 0)
    C = rng.standard_normal((1, 2, 8, 3)) * 5
    C[0, 1, 5] = Z[3, 3:6]
    r2 = o.rvq_encode(Z, C)
    assert r2["idx"][3, 0, 1] == 5
    assert np.all(r2["residual"][3, 3:6] == 0)
    Cd = rng.standard_normal((1, 1, 6, 6))
    Cd[0, 0, 4] = Cd[0, 0, 2]
    near = Cd[0, 0, 2] + 1e-3 * rng.standard_normal((5, 6))
    r3 = o.rvq_encode(near, Cd)
    assert np.all(r3["idx"][:, 0, 0] == 2)
    assert np.all(r3["flag"][:, 0, 0]) and np.all(r3["gap"][:, 0, 0] == 0)


def pin_rvq_progressive(o):
    """§3.5: each round quantises the residual of the previous one, so the
    residual norm never grows when every codebook holds the zero vector, and
    decode(encode(Z)) + residual reproduces Z."""
    rng = np.random.default_rng(9)
    n, R, G, K, gd = 150, 4, 2, 12, 4
    C = rng.standard_normal((R, G, K, gd)) * np.array([1.0, 0.5, 0.25, 0.125])[:, None, None, None]
    C[:, :, 0, :] = 0.0
    Z = rng.standard_normal((n, G * gd))
    prev = np.linalg.norm(Z, axis=1)
    for rr in range(1, R + 1):
        res = o.rvq_encode(Z, C[:rr])
        cur = np.linalg.norm(res["residual"], axis=1)
        assert np.all(cur <= prev + 1e-12)
        prev = cur
        Zh = o.rvq_decode(res["idx"], C[:rr])
        assert np.max(np.abs(Zh + res["residual"] - Z)) < 1e-12
    # a second round whose codebook holds the exact round-1 residual zeroes it
    C2 = rng.standard_normal((2, 1, 5, gd))
    Z1 = rng.standard_normal((1, gd))
    k0 = o.rvq_encode(Z1, C2[:1])["idx"][0, 0, 0]
    C2[1, 0, 3] = Z1[0] - C2[0, 0, k0]
    res = o.rvq_encode(Z1, C2)
    assert res["idx"][0, 1, 0] == 3 and np.all(res["residual"] == 0)


def pin_rvq_given(o):
    """Conditioning on the oracle's own choices reproduces the plain encode."""
    rng = np.random.default_rng(10)
    C = rng.standard_normal((2, 3, 10, 2))
    Z = rng.standard_normal((40, 6))
    a = o.rvq_encode(Z, C)
    b = o.rvq_encode_given(Z, C, a["idx"])
    for k in ("idx", "flag", "gap", "residual"):
        assert np.array_equal(a[k], b[k])


def pin_rvq_given_diverged(o):
    """§3.5 residual rounds, conditioned on another encoder's round-0 choice.

    Hand-built one-dimensional case (G = 1, gd = 1, R = 2), values exact in
    binary.  z = 0; round-0 codes {0, 1}: the nearest is code 0, but the other
    encoder took code 1, so the residual carried into round 1 is 0 - 1 = -1.
    Round-1 codes {-1, 0, 5}: from -1 the nearest is code 0 (distance 0, next
    best code 1 at distance 1), whereas from the unconditioned residual 0 it
    would be code 1.  A second group (z = 2, codes {2, 7} then {0, 3}) is
    given its own nearest choices and must be unaffected.
    """
    Z = np.array([[0.0, 2.0]])
    C = np.zeros((2, 2, 3, 1))
    C[0, 0, :, 0] = [0.0, 1.0, 9.0]
    C[1, 0, :, 0] = [-1.0, 0.0, 5.0]
    C[0, 1, :, 0] = [2.0, 7.0, 8.0]
    C[1, 1, :, 0] = [0.0, 3.0, 4.0]
    given = np.array([[[1, 0], [0, 0]]])
    res = o.rvq_encode_given(Z, C, given)
    # round 0 is still the oracle's own decision from z
    assert res["idx"][0, 0, 0] == 0 and res["gap"][0, 0, 0] == 1.0
    assert res["vnorm2"][0, 0, 0] == 0.0
    # round 1 starts from the residual the given choice left: -1
    assert res["idx"][0, 1, 0] == 0
    assert res["gap"][0, 1, 0] == 1.0
    assert res["vnorm2"][0, 1, 0] == 1.0
    assert res["residual"][0, 0] == 0.0
    # untouched group: z = 2 -> code 0 (exact), residual 0 -> code 0 (exact)
    assert res["idx"][0, 0, 1] == 0 and res["idx"][0, 1, 1] == 0
    assert res["gap"][0, 0, 1] == 25.0 and res["gap"][0, 1, 1] == 9.0
    assert res["residual"][0, 1] == 0.0
    # without conditioning the same input follows its own choice instead
    own = o.rvq_encode(Z, C)
    assert own["idx"][0, 1, 0] == 1 and own["residual"][0, 0] == 0.0


def pin_rvq_tie_flag_norm(o):
    """The near-tie flag compares the best-to-second gap with rel_tie times the
    squared norm of the vector quantised in that round (the group's own
    residual), not its norm and not the whole token's.

    Group 0 holds v = (3, 4), ||v||^2 = 25; group 1 holds (30, 40), whose
    norm would dominate a whole-token reading.  Code 0 of each book is v
    itself and code 1 is v + (delta, 0), so the gap is delta^2: 0.9e-6 * 25
    must be flagged and 1.1e-6 * 25 must not be.
    """
    for frac, want in ((0.9, True), (1.1, False)):
        delta = np.sqrt(frac * 1e-6 * 25.0)
        Z = np.array([[3.0, 4.0, 30.0, 40.0]])
        C = np.zeros((1, 2, 2, 2))
        C[0, 0, 0] = [3.0, 4.0]
        C[0, 0, 1] = [3.0 + delta, 4.0]
        C[0, 1, 0] = [30.0, 40.0]
        C[0, 1, 1] = [-30.0, -40.0]
        res = o.rvq_encode(Z, C)
        assert res["vnorm2"][0, 0, 0] == 25.0
        assert res["idx"][0, 0, 0] == 0
        assert abs(res["gap"][0, 0, 0] - delta ** 2) < 1e-12
        assert bool(res["flag"][0, 0, 0]) is want
        assert not res["flag"][0, 0, 1]


# ----------------------------------------------------------------- §3.3 SPEL
def pin_tangent(o):
    """eq. (4) maps onto the tangent space of St(d,r) at A, {V : sym(A^T V) = 0};
    it leaves tangent vectors unchanged and sends normal vectors A S (S
    symmetric) to zero."""
    rng = np.random.default_rng(11)
    d, r = 30, 6
    A = _orth(rng, d, r)
    g = rng.standard_normal((d, r))
    gR = o.tangent_project(A, g)
    S = A.T @ gR
    assert np.max(np.abs(S + S.T)) < 1e-12
    W = rng.standard_normal((r, r))
    H = rng.standard_normal((d, r))
    tang = A @ (W - W.T) + (np.eye(d) - A @ A.T) @ H
    assert np.max(np.abs(o.tangent_project(A, tang) - tang)) < 1e-12
    Ssym = W + W.T
    assert np.max(np.abs(o.tangent_project(A, A @ Ssym))) < 1e-12
    Ms = rng.standard_normal((4, 4))
    assert np.array_equal(o.sym(Ms), o.sym(Ms).T)
    assert np.allclose(o.sym(Ms) + (Ms - Ms.T) / 2, Ms)


def pin_momentum(o):
    """eq. (5) with a constant input: m_t = (1 - beta^t) g_R from m_0 = 0."""
    rng = np.random.default_rng(12)
    gR = rng.standard_normal((5, 3))
    m = np.zeros_like(gR)
    beta = 0.9
    for t in range(1, 31):
        m = o.momentum(m, gR, beta)
        assert np.max(np.abs(m - (1 - beta ** t) * gR)) < 1e-12


def pin_polar_diagonal(o):
    """An odd matrix polynomial acts on singular values only: for
    Y = U diag(s) V^T, PolarExpress(Y) = U diag(p_n(...p_1(s))) V^T."""
    from pipeline_activation_compression_gb300.polar import default_coeffs
    rng = np.random.default_rng(13)
    d, r = 25, 6
    U = _orth(rng, d, r)
    Vt = _orth(rng, r, r).T
    s = np.array([1.0, 0.7, 0.3, 0.05, 0.01, 0.002])
    co = default_coeffs(5, 0).astype(np.float64)
    Y = U @ np.diag(s) @ Vt
    out = o.polar_express(Y, co)
    t = s.copy()
    for a, b, c in co:
        t = a * t + b * t ** 3 + c * t ** 5
    # the first polynomials amplify fp64 rounding by about 8x per step
    assert np.max(np.abs(out - U @ np.diag(t) @ Vt)) < 1e-10


def pin_polar_limit(o):
    """Enough iterations converge to the polar factor U V^T of an SVD
    (numpy.linalg.svd, a library routine); the result lies on St(d, r)."""
    from pipeline_activation_compression_gb300.polar import default_coeffs
    rng = np.random.default_rng(14)
    Y = rng.standard_normal((40, 8))
    Y /= np.linalg.norm(Y)
    co = default_coeffs(12, 0).astype(np.float64)
    out = o.polar_express(Y, co)
    U, _, Vt = np.linalg.svd(Y, full_matrices=False)
    assert np.max(np.abs(out - U @ Vt)) < 1e-9
    assert np.max(np.abs(out.T @ out - np.eye(8))) < 1e-9


def pin_spel_descends(o):
    """SPEL is a descent method on St(d, r): for f(A) = -tr(A^T B) (gradient
    -B) small steps decrease f, every iterate stays on the manifold, and the
    iterates approach the maximiser polar(B)."""
    from pipeline_activation_compression_gb300.polar import default_coeffs
    rng = np.random.default_rng(15)
    d, r = 24, 4
    B = rng.standard_normal((d, r))
    A = _orth(rng, d, r)
    m = np.zeros_like(A)
    co = default_coeffs(5, 5).astype(np.float64)
    f0 = -np.trace(A.T @ B)
    f = f0
    for _ in range(60):
        A, m, _ = o.spel_step(A, -B, m, 0.05, 0.9, co[:5], co[5:])
        assert np.max(np.abs(A.T @ A - np.eye(r))) < 1e-10
        f = -np.trace(A.T @ B)
    U, _, Vt = np.linalg.svd(B, full_matrices=False)
    fstar = -np.trace((U @ Vt).T @ B)
    assert f < f0 and (f - fstar) < 0.05 * (f0 - fstar)


def pin_spel_momentum_tangent(o):
    """Algorithm 1 feeds the momentum with the tangent projection g_R (eq. (4)
    before eq. (5)): from m = 0 the first momentum is (1 - beta) g_R, which
    lies in the tangent space at A (sym(A^T m) = 0) even for a gradient with
    a large normal component."""
    from pipeline_activation_compression_gb300.polar import default_coeffs
    rng = np.random.default_rng(17)
    d, r = 20, 5
    A = _orth(rng, d, r)
    g = rng.standard_normal((d, r)) + A @ np.diag(np.arange(1.0, r + 1))
    co = default_coeffs(5, 5).astype(np.float64)
    _, m, _ = o.spel_step(A, g, np.zeros_like(A), 1e-3, 0.9, co[:5], co[5:])
    S = A.T @ m
    assert np.max(np.abs(S + S.T)) < 1e-12
    assert np.linalg.norm(m) > 0.01


def pin_spel_drift(o, steps=200):
    """Repeated steps with random gradients keep ||A^T A - I||_max tiny."""
    from pipeline_activation_compression_gb300.polar import default_coeffs
    rng = np.random.default_rng(16)
    d, r = 64, 16
    A = _orth(rng, d, r)
    m = np.zeros_like(A)
    co = default_coeffs(5, 5).astype(np.float64)
    for _ in range(steps):
        A, m, _ = o.spel_step(A, 1e-3 * rng.standard_normal((d, r)), m, 2e-3, 0.9, co[:5], co[5:])
    assert np.max(np.abs(A.T @ A - np.eye(r))) < 1e-10


# ------------------------------------------------------------ §3.2 backward
def _codec_loss(o, X, t, A, E, P, E2, P2, W):
    """L = <W, X_hat> for the composed codec, a scalar function of X and A."""
    Xh = o.reconstruct(o.compress(X, t, A, E, P), t, A, E2, P2)
    return float(np.sum(W * Xh))


def pin_grad_finite_differences(o):
    """The backward pass is the derivative of the forward codec: central
    differences of L = <W, X_hat(X, A)> (quadratic in A, linear in X, so
    the central difference is exact up to rounding) must equal
    dL/dX = grad_decompress(grad_compress(W)) and dL/dA = grad_A; and
    grad_A_given with gZ = W A, Z = compress(...) must agree with grad_A."""
    rng = np.random.default_rng(31)
    d, r, V, n = 7, 3, 5, 6
    A = _orth(rng, d, r)
    P, P2 = _orth(rng, d, r).T, _orth(rng, d, r).T
    E, E2 = rng.standard_normal((V, r)), rng.standard_normal((V, r))
    X, W = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    t = rng.integers(0, V, n)
    h = 1e-4
    gX = np.zeros_like(X)
    for i in range(n):
        for j in range(d):
            Xp, Xm = X.copy(), X.copy()
            Xp[i, j] += h
            Xm[i, j] -= h
            gX[i, j] = (_codec_loss(o, Xp, t, A, E, P, E2, P2, W) -
                        _codec_loss(o, Xm, t, A, E, P, E2, P2, W)) / (2 * h)
    got = o.grad_decompress(o.grad_compress(W, A), A)
    assert np.max(np.abs(got - gX)) < 1e-8 * max(1.0, np.max(np.abs(gX)))
    gA = np.zeros_like(A)
    for i in range(d):
        for j in range(r):
            Ap, Am = A.copy(), A.copy()
            Ap[i, j] += h
            Am[i, j] -= h
            gA[i, j] = (_codec_loss(o, X, t, Ap, E, P, E2, P2, W) -
                        _codec_loss(o, X, t, Am, E, P, E2, P2, W)) / (2 * h)
    got = o.grad_A(X, t, A, E, P, W)
    assert np.max(np.abs(got - gA)) < 1e-7 * max(1.0, np.max(np.abs(gA)))
    given = o.grad_A_given(X, t, E, P, W @ A, W, o.compress(X, t, A, E, P))
    assert np.max(np.abs(given - gA)) < 1e-7 * max(1.0, np.max(np.abs(gA)))


# ------------------------------------------- Fig. 2 first-boundary anchor
def pin_embed_exact_reconstruction(o):
    """Fig. 2 (first boundary): an activation that is its token's embedding
    plus a component S A^T inside span(A) is sent as exactly S and rebuilt
    exactly; a component orthogonal to span(A) is dropped, so X_hat is the
    orthogonal projection of X - E_emb[t] onto span(A) plus E_emb[t]."""
    rng = np.random.default_rng(41)
    d, r, V, n = 24, 6, 9, 11
    A = _orth(rng, d, r)
    E = rng.standard_normal((V, d))
    t = rng.integers(0, V, n)
    S = rng.standard_normal((n, r))
    X = E[t] + S @ A.T
    Z = o.compress_embed(X, t, A, E)
    assert np.max(np.abs(Z - S)) < 1e-12
    assert np.max(np.abs(o.reconstruct_embed(Z, t, A, E) - X)) < 1e-12
    # off-subspace part: lstsq projection of the residual onto span(A)
    Y = rng.standard_normal((n, d))
    coef = np.linalg.lstsq(A, (Y - E[t]).T, rcond=None)[0]
    Xh = o.reconstruct_embed(o.compress_embed(Y, t, A, E), t, A, E)
    assert np.max(np.abs(Xh - (E[t] + (A @ coef).T))) < 1e-12


def pin_embed_one_hot(o):
    """A one-hot embedding row: token v's anchor is e_j, so token v's Z row is
    X A minus row j of A; tokens are looked up by id, not by position."""
    d, r, V = 8, 3, 4
    rng = np.random.default_rng(43)
    A = _orth(rng, d, r)
    E = np.zeros((V, d))
    for v in range(V):
        E[v, (3 * v + 1) % d] = 1.0
    t = np.array([2, 0, 3, 3, 1])
    X = rng.standard_normal((len(t), d))
    Z = o.compress_embed(X, t, A, E)
    for i, v in enumerate(t):
        expect = X[i] @ A - A[(3 * v + 1) % d]
        assert np.max(np.abs(Z[i] - expect)) < 1e-14
    Xh = o.reconstruct_embed(np.zeros((len(t), r)), t, A, E)
    for i, v in enumerate(t):
        assert Xh[i, (3 * v + 1) % d] == 1.0 and np.count_nonzero(Xh[i]) == 1


def pin_embed_grad_finite_differences(o):
    """grad_A_embed is the derivative in A of <W, X_hat(A)> for the
    first-boundary codec X_hat = (X - E_emb[t]) A A^T + E_emb[t]; the loss is
    quadratic in A, so central differences are exact up to rounding."""
    rng = np.random.default_rng(47)
    d, r, V, n = 7, 3, 5, 6
    A = _orth(rng, d, r)
    E = rng.standard_normal((V, d))
    X, W = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    t = rng.integers(0, V, n)

    def loss(Am):
        return float(np.sum(W * o.reconstruct_embed(o.compress_embed(X, t, Am, E), t, Am, E)))

    h = 1e-4
    gA = np.zeros_like(A)
    for i in range(d):
        for j in range(r):
            Ap, Am = A.copy(), A.copy()
            Ap[i, j] += h
            Am[i, j] -= h
            gA[i, j] = (loss(Ap) - loss(Am)) / (2 * h)
    got = o.grad_A_embed(X, t, E, W @ A, W, o.compress_embed(X, t, A, E))
    assert np.max(np.abs(got - gA)) < 1e-7 * max(1.0, np.max(np.abs(gA)))


# ------------------------------------------------- §3.5 codebook streaming
def pin_splitmix64_reference(o):
    """Published first outputs of splitmix64 from state 0 (Vigna's reference
    implementation): 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4,
    0x06c45d188009454f."""
    state, outs = 0, []
    for _ in range(3):
        u, state = o.splitmix64(state)
        outs.append(u)
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def pin_stream_partition(o):
    """App. F: the codebook is partitioned into random subsets.  Over one
    epoch the subsets are disjoint and cover every code; the next epoch is a
    different permutation; the subset is a function of (seed, step) only."""
    total, per = 97, 20
    n_sub = -(-total // per)
    for epoch in range(2):
        ids = [o.stream_subset(total, per, 5, epoch * n_sub + b) for b in range(n_sub)]
        assert [len(x) for x in ids] == [20, 20, 20, 20, 17]
        allids = np.concatenate(ids)
        assert np.array_equal(np.sort(allids), np.arange(total))
    e0 = np.concatenate([o.stream_subset(total, per, 5, b) for b in range(n_sub)])
    e1 = np.concatenate([o.stream_subset(total, per, 5, n_sub + b) for b in range(n_sub)])
    assert not np.array_equal(e0, e1)
    assert np.array_equal(o.stream_subset(total, per, 5, 3), o.stream_subset(total, per, 5, 3))
    assert not np.array_equal(o.stream_subset(total, per, 5, 0), o.stream_subset(total, per, 6, 0))
    # a uniform shuffle of 10 ids leaves some id in place with probability
    # about 1 - 1/e; a single-cycle shuffle (Sattolo) never does
    fixed = [np.any(o.stream_subset(10, 10, sd, 0) == np.arange(10)) for sd in range(20)]
    assert 6 <= sum(fixed) <= 19


def pin_code_update_epoch(o):
    """After a full epoch of refreshes from a live codebook C1, the shared
    codebook equals C1 exactly; after part of it, exactly the refreshed
    codes have moved."""
    rng = np.random.default_rng(41)
    R, G, K, gd = 2, 3, 8, 4
    C0 = rng.standard_normal((R, G, K, gd))
    C1 = rng.standard_normal((R, G, K, gd))
    total, per = R * G * K, 10
    flat1 = C1.reshape(-1, gd)
    C = C0
    moved = set()
    for step in range(-(-total // per)):
        ids = o.stream_subset(total, per, 9, step)
        C = o.apply_code_update(C, ids, flat1[ids])
        moved |= set(ids.tolist())
        if step == 1:
            diff = np.nonzero(np.any(C.reshape(-1, gd) != C0.reshape(-1, gd), axis=1))[0]
            assert set(diff.tolist()) == moved
    assert np.array_equal(C, C1)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


# -------------------------------------------------------------- generator
def check_generator(name="tiny_d64_r16", n_tokens=None):
    w = synth.WORKLOADS[name]
    b = synth.make_boundary(w, n_tokens=n_tokens)
    A, P = b["A_f64"], b["P_f64"]
    assert np.max(np.abs(A.T @ A - np.eye(w.r))) < 1e-12      # St(d,r) definition
    assert np.max(np.abs(P @ P.T - np.eye(w.r))) < 1e-12      # orthonormal rows
    return w, b

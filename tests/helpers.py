"""Shared test utilities: storage-dtype tensors to/from the GPU, error
measures, and the certified comparison of VQ indices with the oracle."""
from __future__ import annotations

import numpy as np

import oracle
from pipeline_activation_compression_gb300 import synth


def to_dev(a, device="cuda"):
    """numpy array in storage dtype (uint16 = bf16 bits) -> CUDA tensor."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def to_host(t) -> np.ndarray:
    """CUDA tensor -> numpy in storage dtype (bf16 -> uint16 bits)."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def rel_frob(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def gpu_residuals(Z32, C, idx):
    """Residual the GPU quantises in each round: fp32 Z minus the chosen
    codes, subtracted in fp32 exactly as the kernel does (IEEE round to
    nearest).  Returns float64 array (N, R, G, gd)."""
    Z32 = np.asarray(Z32, dtype=np.float32)
    Cf = synth.widen(C).astype(np.float32)
    R, G, K, gd = Cf.shape
    N = Z32.shape[0]
    out = np.zeros((N, R, G, gd))
    for g in range(G):
        v = Z32[:, g * gd:(g + 1) * gd].copy()
        for rho in range(R):
            out[:, rho, g] = v
            v = (v - Cf[rho, g][idx[:, rho, g]]).astype(np.float32)
    return out


def check_vq_indices(idx_gpu, Z32_gpu, Z_oracle, C, rel_tie=1e-6):
    """Compare GPU VQ indices with the oracle.

    1. Internal exactness: every GPU index is the exact (fp64) nearest code
       of the residual the GPU itself carried (from its own fp32 Z).
    2. Oracle parity: the oracle re-runs each round from the residual left by
       the GPU's earlier choices; wherever the GPU index differs from the
       oracle's, the disagreement must be a near tie certified by the size of
       the GPU's residual error delta = ||v_gpu - v_oracle||:
         D(k_gpu) - D(k_oracle) <= 2 delta (||v - c_gpu|| + ||v - c_oracle||) + 2 delta^2.
    3. Every mismatch must also carry the oracle's own near-tie flag
       (gap < rel_tie * ||v||^2): indices are bit-exact elsewhere.
    Returns a dict of counts (mismatches, of which inside the literal
    rel_tie * ||v||^2 flag, and the largest certified-band ratio); the
    counts are printed as a diagnostic.
    """
    idx_gpu = np.asarray(idx_gpu).astype(np.int64)
    Cd = synth.widen(C)
    R, G, K, gd = Cd.shape
    V = gpu_residuals(Z32_gpu, C, idx_gpu)
    # 1. the GPU's own decision is exact for its own residual
    for rho in range(R):
        for g in range(G):
            v = V[:, rho, g]
            D = ((v[:, None, :] - Cd[rho, g][None, :, :]) ** 2).sum(-1)
            ref = np.argmin(D, axis=1)
            bad = np.nonzero(ref != idx_gpu[:, rho, g])[0]
            if bad.size:
                n = bad[0]
                raise AssertionError(
                    f"GPU index not the nearest code of its own residual at n={n}, rho={rho}, "
                    f"g={g}: gpu {idx_gpu[n, rho, g]} (D={D[n, idx_gpu[n, rho, g]]:.9g}) vs "
                    f"{ref[n]} (D={D[n, ref[n]]:.9g})")
    # 2. oracle parity with certified near ties
    res = oracle.rvq_encode_given(Z_oracle, Cd, idx_gpu, rel_tie=rel_tie)
    mism = np.argwhere(res["idx"] != idx_gpu)
    u = np.asarray(Z_oracle, dtype=np.float64).copy()
    worst = 0.0
    in_flag = 0
    # oracle residual with GPU choices, per round
    Vo = np.zeros_like(V)
    for g in range(G):
        v = u[:, g * gd:(g + 1) * gd].copy()
        for rho in range(R):
            Vo[:, rho, g] = v
            v = v - Cd[rho, g][idx_gpu[:, rho, g]]
    for n, rho, g in mism:
        vo = Vo[n, rho, g]
        delta = np.linalg.norm(V[n, rho, g] - vo)
        cg = Cd[rho, g][idx_gpu[n, rho, g]]
        co = Cd[rho, g][res["idx"][n, rho, g]]
        gap = np.sum((vo - cg) ** 2) - np.sum((vo - co) ** 2)
        band = 2 * delta * (np.linalg.norm(vo - cg) + np.linalg.norm(vo - co)) + 2 * delta ** 2
        band += 1e-12 * (1 + np.sum(vo ** 2))
        worst = max(worst, gap / band if band > 0 else np.inf)
        if res["flag"][n, rho, g]:
            in_flag += 1
        assert gap <= band, (
            f"index mismatch outside the certified near-tie band at n={n} rho={rho} g={g}: "
            f"gap {gap:.3g} > band {band:.3g} (delta {delta:.3g})")
    total = idx_gpu.size
    rep = dict(total=int(total), mismatches=int(len(mism)), literal_flagged=int(in_flag),
               unflagged=int(len(mism) - in_flag), worst_band_ratio=float(worst))
    print(f"VQ parity: {rep}")
    # bit-exact except where the oracle itself flags a near tie
    assert rep["unflagged"] == 0, f"{rep['unflagged']} unflagged index mismatches of {total}"
    return rep

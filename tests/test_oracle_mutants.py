"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant rewrites one line of the oracle's source (a dropped term, a wrong
sign, a transposed or swapped operand, a wrong index) and loads the result as
a separate module; the real oracle is never modified.  All on the CPU.
"""
import inspect
import types

import pytest

import oracle.mapl_oracle as real
from tests import pins

MUTANTS = {
    "anchor_sign": ("return (X - anchor(E, P, tids)) @ A", "return (X + anchor(E, P, tids)) @ A"),
    "anchor_dropped": ("return (X - anchor(E, P, tids)) @ A", "return X @ A"),
    "anchor_index_shift": ("return E[tids] @ P", "return E[(tids + 1) % E.shape[0]] @ P"),
    "recon_no_anchor": ("return Zhat @ A.T + anchor(E_next, P_next, tids)", "return Zhat @ A.T"),
    "recon_sign": ("return Zhat @ A.T + anchor(E_next, P_next, tids)", "return Zhat @ A.T - anchor(E_next, P_next, tids)"),
    "fold_wrong_M": ("M = P @ A\n", "M = P @ A * 0.5\n"),
    "rvq_argmax": ("k = np.argmin(D, axis=1)", "k = np.argmax(D, axis=1)"),
    "rvq_last_tie": ("k = np.argmin(D, axis=1)", "k = D.shape[1] - 1 - np.argmin(D[:, ::-1], axis=1)"),
    "rvq_residual_sign": ("u[:, cols] = v - C[rho, g][take]", "u[:, cols] = v + C[rho, g][take]"),
    "rvq_no_residual": ("u[:, cols] = v - C[rho, g][take]", "u[:, cols] = v"),
    "rvq_given_ignored": ("take = k if idx_given is None else np.asarray(idx_given)[:, rho, g].astype(np.int64)", "take = k"),
    "rvq_flag_sqrt_norm": ("flag = gap < rel_tie * vn", "flag = gap < rel_tie * np.sqrt(vn)"),
    "rvq_flag_whole_token_norm": ('vn[:, rho, g] = np.einsum("nj,nj->n", v, v)', 'vn[:, rho, g] = np.einsum("nj,nj->n", u, u)'),
    "rvq_wrong_round_book":("k, d1, d2 = _nearest(v, C[rho, g])", "k, d1, d2 = _nearest(v, C[0, g])"),
    "decode_one_round": ("for rho in range(R):\n        for g in range(G):\n            Zh", "for rho in range(1):\n        for g in range(G):\n            Zh"),
    "tangent_no_sym": ("return g - A @ sym(A.T @ g)", "return g - A @ (A.T @ g)"),
    "tangent_sign": ("return g - A @ sym(A.T @ g)", "return g + A @ sym(A.T @ g)"),
    "sym_half_dropped": ("return 0.5 * (M + M.T)", "return (M + M.T)"),
    "momentum_swapped": ("return beta * _f64(m) + (1.0 - beta) * _f64(gR)", "return (1.0 - beta) * _f64(m) + beta * _f64(gR)"),
    "polar_coeff_order": ("Y = Y @ (a * I + b * S + c * (S @ S))", "Y = Y @ (a * I + c * S + b * (S @ S))"),
    "polar_no_square": ("Y = Y @ (a * I + b * S + c * (S @ S))", "Y = Y @ (a * I + b * S + c * S)"),
    "spel_step_sign": ("A_new = polar_express(_f64(A) - lr * d, coeffs_retr)", "A_new = polar_express(_f64(A) + lr * d, coeffs_retr)"),
    "spel_no_retraction": ("A_new = polar_express(_f64(A) - lr * d, coeffs_retr)", "A_new = _f64(A) - lr * d"),
    "spel_raw_gradient": ("m_new = momentum(m, gR, beta)", "m_new = momentum(m, g, beta)"),
    "embed_anchor_sign": ("return (X - E_emb[np.asarray(tids, dtype=np.int64)]) @ A", "return (X + E_emb[np.asarray(tids, dtype=np.int64)]) @ A"),
    "embed_anchor_projected_twice": ("return (X - E_emb[np.asarray(tids, dtype=np.int64)]) @ A", "return X @ A - (E_emb[np.asarray(tids, dtype=np.int64)] @ A) @ (A.T @ A) * 0.5"),
    "embed_recon_no_anchor": ("return Zhat @ A.T + E_emb[np.asarray(tids, dtype=np.int64)]", "return Zhat @ A.T"),
    "embed_recon_positional": ("return Zhat @ A.T + E_emb[np.asarray(tids, dtype=np.int64)]", "return Zhat @ A.T + E_emb[np.arange(Zhat.shape[0]) % E_emb.shape[0]]"),
    "embed_gradA_raw_X": ("    Xres = _f64(X) - _f64(E_emb)[np.asarray(tids, dtype=np.int64)]\n    return Xres.T", "    Xres = _f64(X)\n    return Xres.T"),
    "embed_gradA_term_dropped": ("    return Xres.T @ _f64(gZ) + _f64(gXhat).T @ _f64(Z)\n\n\n# ----", "    return Xres.T @ _f64(gZ)\n\n\n# ----"),
    "gradA_term_dropped": ("return Xres.T @ (g @ A) + g.T @ (Xres @ A)", "return Xres.T @ (g @ A)"),
    "gradA_no_anchor": ("    Xres = _f64(X) - anchor(E, P, tids)\n    A, g = _f64(A), _f64(gXhat)", "    Xres = _f64(X)\n    A, g = _f64(A), _f64(gXhat)"),
    "gradA_given_raw_X": ("    Xres = _f64(X) - anchor(E, P, tids)\n    return Xres.T @ _f64(gZ)", "    Xres = _f64(X) - anchor(E, P, tids)\n    return _f64(X).T @ _f64(gZ)"),
    "grad_decompress_no_T": ("return _f64(gZ) @ _f64(A).T", "return _f64(gZ) @ _f64(A).T * 2.0"),
    "splitmix_shift": ("z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64", "z = ((z ^ (z >> 26)) * 0x94D049BB133111EB) & _M64"),
    "subset_same_epoch": ("state = (seed ^ ((0xD1B54A32D192ED03 * (epoch + 1)) & _M64)) & _M64", "state = seed"),
    "subset_off_by_one": ("        j = u % (i + 1)", "        j = u % i"),
    "code_update_dropped": ("    flat[np.asarray(ids, dtype=np.int64)] = _f64(codes)", "    pass"),
}


def _mutant(old, new):
    src = inspect.getsource(real)
    assert src.count(old) == 1, old
    src = src.replace(old, new, 1)
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    mod = _mutant(*MUTANTS[name])
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(mod)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutant {name}"

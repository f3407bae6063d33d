"""First-boundary anchor (MAPL, Fig. 2: after the first stage the anchor is
the original token embedding) on the GPU vs the fp64 oracle, via the C ABI.

    compress    Z     = (X - E_emb[tids]) A
    decompress  X_hat = Z_hat A^T + E_emb[tids]
    grad_A      dA    = (X - E_emb[tids])^T gZ + gX_hat^T Z

Tolerances as in the main parity tests: 1e-5 relative Frobenius error for
fp32 results (the fp32 Z, dA), 2e-2 for bf16 outputs (Z payload, X_hat); VQ
indices equal the oracle's except at certified near ties.
"""
import numpy as np
import pytest

import oracle
import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import synth
from tests.helpers import check_vq_indices, rel_frob, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_F32 = 1e-5
W = synth.widen


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


def _plan(w, b):
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    A = to_dev(b["A"])
    # P_send / P_recv are not used by an embedding-anchor plan; any valid
    # r x d operand will do
    Pz = torch.zeros(w.r, w.d, dtype=torch.bfloat16, device="cuda")
    plan = mapl.mapl_plan_create(cfg, A, Pz, Pz, to_dev(b["C"]) if w.vq else None)
    E = to_dev(b["E_emb"])
    mapl.mapl_plan_set_embedding_anchor(plan, E)
    return plan, E


def _run(plan, w, b, tids=None):
    X = to_dev(b["X"])
    t = torch.from_numpy(b["tids"] if tids is None else tids).cuda()
    N = X.shape[0]
    payload = torch.empty(plan.payload_shape(N), dtype=plan.payload_dtype(), device="cuda")
    mapl.mapl_compress(plan, X, t, None, payload)
    Z32 = torch.empty(N, w.r, dtype=torch.float32, device="cuda")
    mapl.mapl_compress_z32(plan, X, t, None, Z32)
    Xh = torch.empty(N, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_decompress(plan, payload, t, None, Xh)
    mapl.mapl_check(plan)
    torch.cuda.synchronize()
    return to_host(payload), Z32.cpu().numpy(), to_host(Xh)


def _check(w, b, payload, Z32, Xh, A=None):
    A = W(b["A"]) if A is None else A
    Zo = oracle.compress_embed(W(b["X"]), b["tids"], A, W(b["E_emb"]))
    assert rel_frob(Z32, Zo) <= TOL_F32, rel_frob(Z32, Zo)
    if w.vq:
        check_vq_indices(payload, Z32, Zo, b["C"])
        Zh = oracle.rvq_decode(payload, W(b["C"]))
    else:
        assert rel_frob(W(payload), Zo) <= TOL_BF16
        Zh = W(payload)
    Xo = oracle.reconstruct_embed(Zh, b["tids"], A, W(b["E_emb"]))
    assert rel_frob(W(Xh), Xo) <= TOL_BF16, rel_frob(W(Xh), Xo)


@pytest.mark.parametrize("name,n", [("proj_d1024_r128", 1000), ("vq_d1024_r128", 777),
                                    ("proj_d1024_r64", 300), ("vq_d2048_r128", 259)])
def test_embed_parity(name, n):
    w = synth.WORKLOADS[name]
    b = synth.make_first_boundary(w, seed=5, n_tokens=n)
    plan, _ = _plan(w, b)
    _check(w, b, *_run(plan, w, b))


@pytest.mark.parametrize("n", [1, 127, 128, 129, 4099])
def test_embed_ragged(n):
    w = synth.WORKLOADS["vq_d1024_r128"]
    b = synth.make_first_boundary(w, seed=6, n_tokens=n)
    plan, _ = _plan(w, b)
    _check(w, b, *_run(plan, w, b))


def test_embed_exact_subspace_signal():
    """X = E_emb[t] + S A^T (bf16-exact pieces): Z is S to fp32 rounding and
    X_hat rebuilds X (bf16 rounding of exact values)."""
    w = synth.WORKLOADS["proj_d1024_r128"]
    b = synth.make_first_boundary(w, seed=7, n_tokens=517)
    S = np.random.default_rng(8).standard_normal((517, w.r))
    X = W(b["E_emb"])[b["tids"]] + S @ W(b["A"]).T
    b = dict(b, X=synth._store(X, "bf16"))
    plan, _ = _plan(w, b)
    payload, Z32, Xh = _run(plan, w, b)
    _check(w, b, payload, Z32, Xh)
    assert rel_frob(Z32, S) <= 3e-2   # X itself was rounded to bf16


def test_embed_after_update_A():
    """mapl_plan_update_A recomputes the E_emb A table."""
    w = synth.WORKLOADS["vq_d1024_r128"]
    b = synth.make_first_boundary(w, seed=9, n_tokens=1500)
    plan, _ = _plan(w, b)
    _run(plan, w, b)
    b2 = synth.make_boundary(w, seed=10, n_tokens=8)
    mapl.mapl_plan_update_A(plan, to_dev(b2["A"]))
    b = dict(b, A=b2["A"])
    _check(w, b, *_run(plan, w, b))


def test_embed_grad_A():
    w = synth.WORKLOADS["proj_d1024_r128"]
    n = 999
    b = synth.make_first_boundary(w, seed=11, n_tokens=n)
    gxh = synth.make_boundary_grad(w, seed=11, n_tokens=n)
    plan, _ = _plan(w, b)
    X, t, gXh = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda(), to_dev(gxh)
    Z = torch.empty(n, w.r, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_compress(plan, X, t, None, Z)
    gZ = torch.empty(n, w.r, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_grad_compress(plan, gXh, gZ)
    dA = torch.empty(w.d, w.r, dtype=torch.float32, device="cuda")
    mapl.mapl_grad_A(plan, X, t, None, gZ, gXh, Z, dA)
    mapl.mapl_check(plan)
    torch.cuda.synchronize()
    dA_or = oracle.grad_A_embed(W(b["X"]), b["tids"], W(b["E_emb"]), W(to_host(gZ)), W(gxh),
                                W(to_host(Z)))
    assert rel_frob(dA.cpu().numpy(), dA_or) <= TOL_F32


def test_embed_bad_token_flagged():
    w = synth.WORKLOADS["proj_d1024_r128"]
    b = synth.make_first_boundary(w, seed=12, n_tokens=200)
    plan, _ = _plan(w, b)
    t = b["tids"].copy()
    t[17] = w.V + 3
    X = to_dev(b["X"])
    tt = torch.from_numpy(t).cuda()
    Xh = torch.empty(200, w.d, dtype=torch.bfloat16, device="cuda")
    Z = torch.empty(200, w.r, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_decompress(plan, Z.zero_(), tt, None, Xh)
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_check(plan)
    assert ei.value.name == "MAPL_ERR_BAD_TOKEN"
    mapl.mapl_compress(plan, X, tt, None, Z)
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_check(plan)
    assert ei.value.name == "MAPL_ERR_BAD_TOKEN"


def test_embed_unsupported():
    w = synth.WORKLOADS["proj_d1024_r256"]   # 3r = 768 table columns
    b = synth.make_first_boundary(w, seed=13, n_tokens=8)
    with pytest.raises(mapl.MaplError) as ei:
        _plan(w, b)
    assert ei.value.name == "MAPL_ERR_UNSUPPORTED"

"""Backward pass through the codec (MAPL §3.2: the boundary gradient is routed
through the same projector A) on the GPU vs the fp64 oracle, via the C ABI.

gZ = dL/dX_hat A and dL/dX = gZ A^T are bf16 outputs (relative Frobenius
error <= 2e-2); each kernel is checked in isolation on the GPU's own input
(dL/dX from the GPU's gZ widened).  dA = X_res^T gZ + dL/dX_hat^T Z is an
fp32 output (<= 1e-5), computed by the oracle from the same bf16 gZ and Z.
"""
import numpy as np
import pytest

import oracle
import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import synth
from tests.helpers import rel_frob, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_F32 = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


def _plan(w, b):
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    return mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(b["C"]) if w.vq else None)


def _backward(w, n, seed=3):
    b = synth.make_boundary(w, seed=seed, n_tokens=n)
    gxh = synth.make_boundary_grad(w, seed=seed, n_tokens=n)
    plan = _plan(w, b)
    X, t, E = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda(), to_dev(b["E"])
    gXh = to_dev(gxh)
    gZ = torch.empty(n, w.r, dtype=torch.bfloat16, device="cuda")
    gX = torch.empty(n, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_grad_compress(plan, gXh, gZ)
    mapl.mapl_grad_decompress(plan, gZ, gX)
    # Z as the receiver has it without VQ: the bf16 payload of the same plan
    # shape (a no-VQ plan gives the bf16 Z)
    cfg0 = mapl.make_config(w.d, w.r, w.V, dtype=mapl.MAPL_BF16)
    plan0 = mapl.mapl_plan_create(cfg0, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]))
    Z = torch.empty(n, w.r, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_compress(plan0, X, t, E, Z)
    dA = torch.empty(w.d, w.r, dtype=torch.float32, device="cuda")
    mapl.mapl_grad_A(plan, X, t, E, gZ, gXh, Z, dA)
    mapl.mapl_check(plan)
    torch.cuda.synchronize()
    return b, gxh, to_host(gZ), to_host(gX), to_host(Z), dA.cpu().numpy()


@pytest.mark.parametrize("name,n", [("proj_d1024_r128", 1000), ("vq_d1024_r128", 777),
                                    ("proj_d1024_r256", 513), ("vq_d2048_r128", 300),
                                    ("proj_d1024_r512", 300), ("proj_d1024_r64", 129)])
def test_backward_parity(name, n):
    w = synth.WORKLOADS[name]
    b, gxh, gZ, gX, Z, dA = _backward(w, n)
    W = synth.widen
    gZ_or = oracle.grad_compress(W(gxh), W(b["A"]))
    assert rel_frob(W(gZ), gZ_or) <= TOL_BF16
    gX_or = oracle.grad_decompress(W(gZ), W(b["A"]))
    assert rel_frob(W(gX), gX_or) <= TOL_BF16
    dA_or = oracle.grad_A_given(W(b["X"]), b["tids"], W(b["E"]), W(b["P"]), W(gZ), W(gxh), W(Z))
    assert rel_frob(dA, dA_or) <= TOL_F32, rel_frob(dA, dA_or)


@pytest.mark.parametrize("n", [1, 127, 128, 129])
def test_backward_ragged(n):
    w = synth.WORKLOADS["proj_d1024_r128"]
    b, gxh, gZ, gX, Z, dA = _backward(w, n, seed=4)
    W = synth.widen
    assert rel_frob(W(gZ), oracle.grad_compress(W(gxh), W(b["A"]))) <= TOL_BF16
    assert rel_frob(W(gX), oracle.grad_decompress(W(gZ), W(b["A"]))) <= TOL_BF16
    dA_or = oracle.grad_A_given(W(b["X"]), b["tids"], W(b["E"]), W(b["P"]), W(gZ), W(gxh), W(Z))
    assert rel_frob(dA, dA_or) <= TOL_F32


def test_backward_full_size():
    """32768 tokens at d=1024, r=128 (the forward workload's size): dA in full,
    gZ and dL/dX on sampled rows."""
    w = synth.WORKLOADS["vq_d1024_r128"]
    b, gxh, gZ, gX, Z, dA = _backward(w, w.N, seed=5)
    W = synth.widen
    rows = np.sort(np.random.default_rng(9).choice(w.N, size=1024, replace=False))
    assert rel_frob(W(gZ)[rows], oracle.grad_compress(W(gxh)[rows], W(b["A"]))) <= TOL_BF16
    assert rel_frob(W(gX)[rows], oracle.grad_decompress(W(gZ)[rows], W(b["A"]))) <= TOL_BF16
    dA_or = oracle.grad_A_given(W(b["X"]), b["tids"], W(b["E"]), W(b["P"]), W(gZ), W(gxh), W(Z))
    assert rel_frob(dA, dA_or) <= TOL_F32
    assert np.isfinite(dA).all()


@pytest.mark.parametrize("name,n", [("vq_d1024_r128", 3001), ("proj_d1024_r256", 1000)])
def test_grad_A_same_bits_every_call_and_bad_ids(name, n):
    """Two calls give the same bits (the split sums are added in a fixed
    order), and token ids outside [0, V) set MAPL_ERR_BAD_TOKEN and contribute
    no anchor term: the oracle's result with those tokens' anchor rows zero."""
    w = synth.WORKLOADS[name]
    b = synth.make_boundary(w, seed=8, n_tokens=n)
    gxh = synth.make_boundary_grad(w, seed=8, n_tokens=n)
    plan = _plan(w, b)
    tids = b["tids"].copy()
    bad = np.array([0, 5, n // 2, n - 1])
    tids[bad] = np.array([-1, w.V, w.V + 7, -(2 ** 31)], dtype=tids.dtype)
    X, t, E = to_dev(b["X"]), torch.from_numpy(tids).cuda(), to_dev(b["E"])
    gXh, Z = to_dev(gxh), to_dev(b["X"][:, : w.r])
    gZ = torch.empty(n, w.r, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_grad_compress(plan, gXh, gZ)
    ws = torch.empty(mapl.mapl_grad_workspace_size(plan, n), dtype=torch.uint8, device="cuda")
    dA1 = torch.empty(w.d, w.r, dtype=torch.float32, device="cuda")
    dA2 = torch.empty_like(dA1)
    mapl.mapl_grad_A(plan, X, t, E, gZ, gXh, Z, dA1, ws)
    mapl.mapl_grad_A(plan, X, t, E, gZ, gXh, Z, dA2, ws)
    torch.cuda.synchronize()
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_check(plan)
    assert ei.value.name == "MAPL_ERR_BAD_TOKEN"
    assert torch.equal(dA1, dA2)
    Wd = synth.widen
    E0 = np.vstack([Wd(b["E"]), np.zeros((1, w.r))])   # row V: the zero anchor
    t0 = np.where((tids < 0) | (tids >= w.V), w.V, tids)
    dA_or = oracle.grad_A_given(Wd(b["X"]), t0, E0, Wd(b["P"]), Wd(to_host(gZ)), Wd(gxh),
                                Wd(b["X"][:, : w.r]))
    assert rel_frob(dA1.cpu().numpy(), dA_or) <= TOL_F32

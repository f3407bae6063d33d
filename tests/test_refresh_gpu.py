"""Projector broadcast fused into the SPEL step (MAPL §3.3: the updated A_p
goes to the next stage after every optimizer step), on the GPU via the C ABI.

mapl_spel_step_refresh must leave A and m bit-identical to mapl_spel_step and
each refreshed plan in the state mapl_plan_update_A(bf16(A)) gives: the
codec's outputs from the two plans are compared bit for bit, and against the
fp64 oracle on the new projector.
"""
import numpy as np
import pytest

import oracle
import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import polar, synth
from tests.helpers import check_vq_indices, rel_frob, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


def _ws(d, r, batch):
    n = mapl.mapl_spel_workspace_size(d, r, batch)
    return torch.empty(n // 4 + 64, dtype=torch.float32, device="cuda")


def _codec(plan, w, b, X, t, E, En):
    N = X.shape[0]
    pay = torch.empty(plan.payload_shape(N), dtype=plan.payload_dtype(), device="cuda")
    mapl.mapl_compress(plan, X, t, E, pay)
    Z32 = torch.empty(N, w.r, dtype=torch.float32, device="cuda")
    mapl.mapl_compress_z32(plan, X, t, E, Z32)
    Xh = torch.empty(N, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_decompress(plan, pay, t, En, Xh)
    mapl.mapl_check(plan)
    torch.cuda.synchronize()
    return to_host(pay), Z32.cpu().numpy(), to_host(Xh)


@pytest.mark.parametrize("name,n_retr", [("vq_d1024_r128", 5), ("proj_d1024_r256", 7),
                                         ("proj_d1024_r128", 0)])
def test_refresh_matches_update_A(name, n_retr):
    w = synth.WORKLOADS[name]
    n = 700
    batch = 3
    b = synth.make_boundary(w, seed=21, n_tokens=n)
    sw = synth.SpelWorkload("refresh", w.d, w.r, batch)
    s = synth.make_spel(sw, seed=2)
    G = next(synth.spel_gradients(sw, seed=2))
    co = polar.default_coeffs(5, max(n_retr, 1))[: 5 + n_retr]
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    C = to_dev(b["C"]) if w.vq else None
    mk = lambda: mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]), C)
    plans = [mk(), None, mk()]
    A1 = torch.from_numpy(s["A"]).cuda()
    m1 = torch.zeros_like(A1)
    A2, m2 = A1.clone(), m1.clone()
    Gd = torch.from_numpy(G).cuda()
    mapl.mapl_spel_step_refresh(A1, Gd, m1, sw.lr, sw.beta, co, 5, n_retr, plans, _ws(w.d, w.r, batch))
    mapl.mapl_spel_step(A2, Gd, m2, sw.lr, sw.beta, co, 5, n_retr, _ws(w.d, w.r, batch))
    torch.cuda.synchronize()
    assert torch.equal(A1, A2) and torch.equal(m1, m2)
    X, t = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda()
    E, En = to_dev(b["E"]), to_dev(b["E_next"])
    for i in (0, 2):
        Ab = A2[i].to(torch.bfloat16).contiguous()
        ref = mk()
        mapl.mapl_plan_update_A(ref, Ab)
        got = _codec(plans[i], w, b, X, t, E, En)
        want = _codec(ref, w, b, X, t, E, En)
        for g, h in zip(got, want):
            assert np.array_equal(g, h)
        # and the oracle on the new projector
        Anew = synth.widen(to_host(Ab))
        Zo = oracle.compress(synth.widen(b["X"]), b["tids"], Anew, synth.widen(b["E"]),
                             synth.widen(b["P"]))
        assert rel_frob(got[1], Zo) <= 1e-5
        if w.vq:
            check_vq_indices(got[0], got[1], Zo, b["C"])


def test_refresh_embedding_plan():
    """An embedding-anchor plan refreshed by the step recomputes E_emb A."""
    w = synth.WORKLOADS["proj_d1024_r128"]
    b = synth.make_first_boundary(w, seed=23, n_tokens=300)
    sw = synth.SpelWorkload("refresh", w.d, w.r, 1)
    s = synth.make_spel(sw, seed=3)
    G = next(synth.spel_gradients(sw, seed=3))
    co = polar.default_coeffs(5, 5)
    cfg = mapl.make_config(w.d, w.r, w.V, dtype=mapl.MAPL_BF16)
    Pz = torch.zeros(w.r, w.d, dtype=torch.bfloat16, device="cuda")
    plan = mapl.mapl_plan_create(cfg, to_dev(b["A"]), Pz, Pz)
    mapl.mapl_plan_set_embedding_anchor(plan, to_dev(b["E_emb"]))
    A = torch.from_numpy(s["A"]).cuda()
    m = torch.zeros_like(A)
    mapl.mapl_spel_step_refresh(A, torch.from_numpy(G).cuda(), m, sw.lr, sw.beta, co, 5, 5,
                                [plan], _ws(w.d, w.r, 1))
    X, t = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda()
    Z32 = torch.empty(300, w.r, dtype=torch.float32, device="cuda")
    mapl.mapl_compress_z32(plan, X, t, None, Z32)
    mapl.mapl_check(plan)
    Anew = synth.widen(to_host(A[0].to(torch.bfloat16).contiguous()))
    Zo = oracle.compress_embed(synth.widen(b["X"]), b["tids"], Anew, synth.widen(b["E_emb"]))
    assert rel_frob(Z32.cpu().numpy(), Zo) <= 1e-5


def test_refresh_rejects_mismatched_plan():
    w = synth.WORKLOADS["proj_d1024_r128"]
    b = synth.make_boundary(w, seed=24, n_tokens=8)
    cfg = mapl.make_config(w.d, w.r, w.V, dtype=mapl.MAPL_BF16)
    plan = mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]))
    sw = synth.SpelWorkload("refresh", 1024, 256, 1)
    s = synth.make_spel(sw)
    A = torch.from_numpy(s["A"]).cuda()
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_spel_step_refresh(A, torch.zeros_like(A), torch.zeros_like(A), 1e-3, 0.9,
                                    polar.default_coeffs(5, 5), 5, 5, [plan], _ws(1024, 256, 1))
    assert ei.value.name == "MAPL_ERR_INVALID_ARG"
    sw2 = synth.SpelWorkload("refresh", 1024, 128, 2)
    A2 = torch.from_numpy(synth.make_spel(sw2)["A"]).cuda()
    before = A2.clone()
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_spel_step_refresh(A2, torch.zeros_like(A2), torch.zeros_like(A2), 1e-3, 0.9,
                                    polar.default_coeffs(5, 5), 5, 5, [plan, plan],
                                    _ws(1024, 128, 2))
    assert ei.value.name == "MAPL_ERR_INVALID_ARG"
    torch.cuda.synchronize()
    assert torch.equal(A2, before)   # rejected before anything ran

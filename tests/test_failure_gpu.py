"""Failure detection without a GPU fault: the codec kernels' bounded wait.

Every wait inside the kernels gives up after a budget, records the timeout in
the plan's error word and lets the kernel exit, so the context stays usable.
mapl_selftest_bounded_wait runs that same wait on a barrier that nothing
completes (no copy or MMA in flight); the test checks the budget is honoured,
that mapl_check reports MAPL_ERR_TIMEOUT once, and that the codec then runs
and matches the oracle on the same plan and context.
"""
import numpy as np
import pytest

import oracle
import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import synth
from tests.helpers import rel_frob, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


def _plan(w, b):
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    return mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(b["C"]) if w.vq else None)


@pytest.mark.parametrize("budget_ns", [20_000, 2_000_000, 50_000_000])
def test_bounded_wait_reports_timeout(budget_ns):
    w = synth.WORKLOADS["proj_d1024_r128"]
    b = synth.make_boundary(w, seed=31, n_tokens=300)
    plan = _plan(w, b)
    waited = mapl.mapl_selftest_bounded_wait(plan, budget_ns)
    assert budget_ns <= waited < budget_ns + 100_000_000
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_check(plan)
    assert ei.value.name == "MAPL_ERR_TIMEOUT"
    mapl.mapl_check(plan)   # the word was cleared: reported once

    # the same plan and context still run the codec correctly
    X, t = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda()
    Z = torch.empty(300, w.r, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_compress(plan, X, t, to_dev(b["E"]), Z)
    Xh = torch.empty(300, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_decompress(plan, Z, t, to_dev(b["E_next"]), Xh)
    mapl.mapl_check(plan)
    W = synth.widen
    Zo = oracle.compress(W(b["X"]), b["tids"], W(b["A"]), W(b["E"]), W(b["P"]))
    assert rel_frob(W(to_host(Z)), Zo) <= 2e-2
    Xo = oracle.reconstruct(W(to_host(Z)), b["tids"], W(b["A"]), W(b["E_next"]), W(b["P_next"]))
    assert rel_frob(W(to_host(Xh)), Xo) <= 2e-2


def test_bounded_wait_argument_checks():
    w = synth.WORKLOADS["proj_d1024_r64"]
    b = synth.make_boundary(w, seed=32, n_tokens=8)
    plan = _plan(w, b)
    for bad in (0, 999, 3_000_000_000):
        with pytest.raises(mapl.MaplError) as ei:
            mapl.mapl_selftest_bounded_wait(plan, bad)
        assert ei.value.name == "MAPL_ERR_INVALID_ARG"
    mapl.mapl_check(plan)

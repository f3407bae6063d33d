"""Largest inputs: more than 2^31 activation elements in one call.

Rows are independent through the whole codec, so a batch made of 64 copies of
a 32768-token micro-batch (plus a ragged tail) must reproduce, bit for bit,
the payload and X_hat of the micro-batch itself in every copy; the
micro-batch is checked against the oracle by the main parity tests.  This
exercises 64-bit offsets, tile counts past 2^14 and the ragged last tile at
N * d > 2^31.
"""
import numpy as np
import pytest

import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import synth
from tests.helpers import to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("name", ["vq_d1024_r128", "proj_d1024_r128"])
def test_copies_reproduce_the_micro_batch(name):
    w = synth.WORKLOADS[name]
    n0 = 32768
    b = synth.make_boundary(w, seed=41, n_tokens=n0)
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    plan = mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(b["C"]) if w.vq else None)
    E, En = to_dev(b["E"]), to_dev(b["E_next"])
    X0, t0 = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda()
    reps, tail = 64, 77
    N = reps * n0 + tail
    assert N * w.d > 2 ** 31
    X = torch.cat([X0.repeat(reps, 1), X0[:tail]])
    t = torch.cat([t0.repeat(reps), t0[:tail]])
    pay0 = torch.empty(plan.payload_shape(n0), dtype=plan.payload_dtype(), device="cuda")
    Xh0 = torch.empty(n0, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_compress(plan, X0, t0, E, pay0)
    mapl.mapl_decompress(plan, pay0, t0, En, Xh0)
    pay = torch.empty(plan.payload_shape(N), dtype=plan.payload_dtype(), device="cuda")
    mapl.mapl_compress(plan, X, t, E, pay)
    del X
    Xh = torch.empty(N, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_decompress(plan, pay, t, En, Xh)
    mapl.mapl_check(plan)
    torch.cuda.synchronize()
    for k in (0, 1, reps // 2, reps - 1):
        sl = slice(k * n0, (k + 1) * n0)
        assert torch.equal(pay[sl], pay0), f"payload copy {k}"
        assert torch.equal(Xh[sl], Xh0), f"X_hat copy {k}"
    assert torch.equal(pay[reps * n0:], pay0[:tail])
    assert torch.equal(Xh[reps * n0:], Xh0[:tail])

"""Several plans used at once: on different streams of one thread, and from
several host threads.  Calls on distinct plans share nothing, so every
result must equal, bit for bit, the same call made alone."""
import threading

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


def _setup(wname, seed, N):
    w = synth.WORKLOADS[wname]
    b = synth.make_boundary(w, seed=seed, n_tokens=N)
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    plan = mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(b["C"]) if w.vq else None)
    io = dict(X=to_dev(b["X"]), t=torch.from_numpy(b["tids"]).cuda(), E=to_dev(b["E"]),
              En=to_dev(b["E_next"]))
    return w, plan, io


def _codec(w, plan, io, stream=None):
    N = io["X"].shape[0]
    pay = torch.empty(plan.payload_shape(N), dtype=plan.payload_dtype(), device="cuda")
    xh = torch.empty(N, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_compress(plan, io["X"], io["t"], io["E"], pay, stream)
    mapl.mapl_decompress(plan, pay, io["t"], io["En"], xh, stream)
    return pay, xh


CASES = [("vq_d1024_r128", 1, 5000), ("proj_d1024_r128", 2, 3000), ("vq_d2048_r128", 3, 2000),
         ("proj_d1024_r64", 4, 4097)]


def test_streams_of_one_thread():
    setups = [_setup(*c) for c in CASES]
    alone = []
    for w, plan, io in setups:
        alone.append(_codec(w, plan, io))
        mapl.mapl_check(plan)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in setups]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = []
    for rep in range(3):
        outs = [_codec(w, plan, io, s) for (w, plan, io), s in zip(setups, streams)]
    torch.cuda.synchronize()
    for (w, plan, io), (p0, x0), (p1, x1) in zip(setups, alone, outs):
        mapl.mapl_check(plan)
        assert torch.equal(p0, p1)
        assert torch.equal(x0.view(torch.int16), x1.view(torch.int16))


def test_host_threads():
    setups = [_setup(*c) for c in CASES]
    alone = [_codec(w, plan, io) for w, plan, io in setups]
    torch.cuda.synchronize()
    results = [None] * len(setups)
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            w, plan, io = setups[i]
            with torch.cuda.stream(s):
                for _ in range(3):
                    results[i] = _codec(w, plan, io, s)
            s.synchronize()
            mapl.mapl_check(plan, s)
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(setups))]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    for (p0, x0), (p1, x1) in zip(alone, results):
        assert torch.equal(p0, p1)
        assert torch.equal(x0.view(torch.int16), x1.view(torch.int16))

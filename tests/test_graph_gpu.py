"""mapl_compress / mapl_decompress captured in a CUDA graph and replayed give
the same bits as the eager calls (the calls enqueue only kernels on the given
stream, so stream capture records them as they are)."""
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


@pytest.mark.parametrize("wname", ["vq_d1024_r128", "proj_d1024_r128"])
def test_graph_replay_matches_eager(wname):
    w = synth.WORKLOADS[wname]
    N = 1000
    b = synth.make_boundary(w, seed=21, n_tokens=N)
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    plan = mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(b["C"]) if w.vq else None)
    X, t = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda()
    E, En = to_dev(b["E"]), to_dev(b["E_next"])
    pay_e = torch.empty(plan.payload_shape(N), dtype=plan.payload_dtype(), device="cuda")
    xh_e = torch.empty(N, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_compress(plan, X, t, E, pay_e)
    mapl.mapl_decompress(plan, pay_e, t, En, xh_e)
    torch.cuda.synchronize()
    pay_g = torch.zeros_like(pay_e)
    xh_g = torch.zeros_like(xh_e)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mapl.mapl_compress(plan, X, t, E, pay_g)
        mapl.mapl_decompress(plan, pay_g, t, En, xh_g)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    mapl.mapl_check(plan)
    assert torch.equal(pay_g, pay_e)
    assert torch.equal(xh_g.view(torch.int16), xh_e.view(torch.int16))

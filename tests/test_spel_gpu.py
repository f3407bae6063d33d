"""SPEL projector update on the GPU vs the fp64 oracle (needs a GB300)."""
import numpy as np
import pytest

import oracle
import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import polar, synth
from tests.helpers import rel_frob

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


def workspace(d, r, batch):
    n = mapl.mapl_spel_workspace_size(d, r, batch)
    return torch.empty(n // 4 + 64, dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("d,r,batch,n_lmo,n_retr", [
    (256, 64, 2, 5, 5), (1024, 256, 3, 5, 5), (2048, 256, 3, 5, 7), (96, 20, 1, 3, 2),
    (384, 128, 2, 2, 1), (2176, 128, 1, 1, 1), (640, 256, 1, 0, 2)])
def test_one_step_parity(d, r, batch, n_lmo, n_retr):
    w = synth.SpelWorkload(f"t{d}", d, r, batch)
    s = synth.make_spel(w)
    G = next(synth.spel_gradients(w))
    rng = np.random.default_rng(3)
    m0 = (1e-3 * rng.standard_normal(s["A"].shape)).astype(np.float32)
    co = polar.default_coeffs(n_lmo, n_retr)
    A_d = torch.from_numpy(s["A"]).cuda()
    G_d = torch.from_numpy(G).cuda()
    m_d = torch.from_numpy(m0).cuda()
    mapl.mapl_spel_step(A_d, G_d, m_d, w.lr, w.beta, co, n_lmo, n_retr, workspace(d, r, batch))
    torch.cuda.synchronize()
    A_g, m_g = A_d.cpu().numpy(), m_d.cpu().numpy()
    cod = co.astype(np.float64)
    for i in range(batch):
        A_o, m_o, _ = oracle.spel_step(s["A"][i], G[i], m0[i], w.lr, w.beta, cod[:n_lmo], cod[n_lmo:])
        assert rel_frob(m_g[i], m_o) <= 1e-5
        assert rel_frob(A_g[i], A_o) <= 1e-5
        assert np.max(np.abs(A_g[i].T.astype(np.float64) @ A_g[i] - np.eye(r))) <= 1e-3


@pytest.mark.parametrize("name", ["spel_d1024_r256", "spel_d2048_r256"])
def test_drift_1000_steps(name):
    w = synth.SPEL_WORKLOADS[name]
    s = synth.make_spel(w)
    co = polar.default_coeffs(5, 5)
    A_d = torch.from_numpy(s["A"]).cuda()
    m_d = torch.zeros_like(A_d)
    ws = workspace(w.d, w.r, w.batch)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    G_d = torch.empty_like(A_d)
    for _ in range(1000):
        G_d.normal_(0.0, w.grad_std, generator=gen)
        mapl.mapl_spel_step(A_d, G_d, m_d, w.lr, w.beta, co, 5, 5, ws)
    torch.cuda.synchronize()
    A = A_d.double()
    eye = torch.eye(w.r, dtype=torch.float64, device="cuda")
    drift = max(float((A[i].T @ A[i] - eye).abs().max()) for i in range(w.batch))
    print(name, "max |A^T A - I| after 1000 steps:", drift)
    assert drift <= 1e-3
    assert torch.isfinite(A).all()

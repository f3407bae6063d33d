"""mapl_spel_step_static: the SPEL step for callers that cannot allocate.

Some callers cannot hand the library freshly allocated device memory when the
projector update runs (a framework whose caching allocator already reserved
its device memory, a latency-bound loop that cannot absorb cudaMalloc's
implicit synchronisation, a plugin with a fixed tensor-only signature).  The
static entry point runs the same update on a fixed scratch array inside the
library instead of a caller workspace.  These tests call it through the C ABI
and check it against the workspace entry point, on two calls in a row.
"""
import numpy as np
import pytest

import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import polar, synth
from tests.helpers import rel_frob

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-5   # the SPEL parity tolerance of the other GPU tests


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("d,r,batch", [(1024, 256, 3), (256, 64, 2)])
def test_static_matches_workspace_entry_two_calls(d, r, batch):
    w = synth.SpelWorkload(f"noalloc{d}", d, r, batch)
    s = synth.make_spel(w)
    grads = synth.spel_gradients(w, seed=5)
    co = polar.default_coeffs(5, 5)
    A_ref = torch.from_numpy(s["A"]).cuda()
    m_ref = torch.zeros_like(A_ref)
    A_sta = A_ref.clone()
    m_sta = m_ref.clone()
    ws = torch.empty(mapl.mapl_spel_workspace_size(d, r, batch) // 4 + 64, dtype=torch.float32,
                     device="cuda")
    for call in range(2):
        G = torch.from_numpy(next(grads)).cuda()
        mapl.mapl_spel_step(A_ref, G, m_ref, w.lr, w.beta, co, 5, 5, ws)
        mapl.mapl_spel_step_static(A_sta, G, m_sta, w.lr, w.beta, co, 5, 5)
        torch.cuda.synchronize()
        a_ref, a_sta = A_ref.cpu().numpy(), A_sta.cpu().numpy()
        assert np.isfinite(a_sta).all()
        assert rel_frob(a_sta, a_ref) <= TOL, f"call {call}: A"
        assert rel_frob(m_sta.cpu().numpy(), m_ref.cpu().numpy()) <= TOL, f"call {call}: m"


def test_static_rejects_sizes_beyond_its_scratch():
    d, r, batch = 2048, 256, 3
    assert mapl.mapl_spel_workspace_size(d, r, batch) > 16 << 20
    A = torch.zeros(batch, d, r, dtype=torch.float32, device="cuda")
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_spel_step_static(A, A.clone(), A.clone(), 1e-3, 0.9, polar.default_coeffs(5, 5),
                                   5, 5)
    assert ei.value.name == "MAPL_ERR_UNSUPPORTED"
    assert "scratch" in str(ei.value)

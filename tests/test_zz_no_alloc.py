"""mapl_spel_step_static: the SPEL step for callers that cannot allocate.

Some callers cannot hand the library freshly allocated device memory when the
projector update runs (a framework whose caching allocator already reserved
its device memory, a latency-bound loop that cannot absorb cudaMalloc's
implicit synchronisation, a plugin with a fixed tensor-only signature).  The
static entry point runs the same update on a fixed scratch array inside the
library instead of a caller workspace.  These tests call it through the C ABI
and check it bit for bit against the workspace entry point, on two calls in a
row, after calls of another shape and on a side stream, and check that it
reserves no device memory.
"""
import pytest

import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import polar, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


class _Pair:
    """One projector batch stepped by both entry points side by side."""

    def __init__(self, d, r, batch, seed):
        self.w = synth.SpelWorkload(f"noalloc{d}", d, r, batch)
        s = synth.make_spel(self.w)
        self.grads = synth.spel_gradients(self.w, seed=seed)
        self.co = polar.default_coeffs(5, 5)
        self.A_ref = torch.from_numpy(s["A"]).cuda()
        self.m_ref = torch.zeros_like(self.A_ref)
        self.A_sta = self.A_ref.clone()
        self.m_sta = self.m_ref.clone()
        self.ws = torch.empty(mapl.mapl_spel_workspace_size(d, r, batch) // 4 + 64,
                              dtype=torch.float32, device="cuda")

    def step(self, stream=None):
        G = torch.from_numpy(next(self.grads)).cuda()
        w = self.w
        mapl.mapl_spel_step(self.A_ref, G, self.m_ref, w.lr, w.beta, self.co, 5, 5, self.ws,
                            stream=stream)
        mapl.mapl_spel_step_static(self.A_sta, G, self.m_sta, w.lr, w.beta, self.co, 5, 5,
                                   stream=stream)

    def check(self, what):
        torch.cuda.synchronize()
        assert torch.isfinite(self.A_sta).all(), what
        # the same kernels on the same inputs: identical bits, so a stale
        # read of the shared scratch cannot hide under a tolerance
        assert torch.equal(self.A_sta, self.A_ref), f"{what}: A"
        assert torch.equal(self.m_sta, self.m_ref), f"{what}: m"


@pytest.mark.parametrize("d,r,batch", [(1024, 256, 3), (256, 64, 2)])
def test_static_matches_workspace_entry_two_calls(d, r, batch):
    p = _Pair(d, r, batch, seed=5)
    for call in range(2):
        p.step()
        p.check(f"call {call}")


def test_static_after_other_shapes_and_streams():
    """A large call, then a small one that leaves different contents in the
    shared array, then the large shape again on another stream: every result
    is bit-identical to the workspace entry point's."""
    big, small = _Pair(1024, 256, 3, seed=11), _Pair(256, 64, 2, seed=12)
    big.step()
    big.check("large")
    small.step()
    small.check("small")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        big.step(stream=s)
    big.check("large on a side stream")


def test_static_allocates_nothing():
    """After a first call, further calls leave the device's free memory and
    the framework allocator's reservation unchanged."""
    p = _Pair(1024, 256, 3, seed=13)
    G = torch.from_numpy(next(p.grads)).cuda()
    w = p.w
    mapl.mapl_spel_step_static(p.A_sta, G, p.m_sta, w.lr, w.beta, p.co, 5, 5)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    res0 = torch.cuda.memory_reserved()
    for _ in range(5):
        mapl.mapl_spel_step_static(p.A_sta, G, p.m_sta, w.lr, w.beta, p.co, 5, 5)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_reserved() == res0
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"


def test_static_rejects_sizes_beyond_its_scratch():
    d, r, batch = 2048, 256, 3
    assert mapl.mapl_spel_workspace_size(d, r, batch) > 16 << 20
    A = torch.zeros(batch, d, r, dtype=torch.float32, device="cuda")
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_spel_step_static(A, A.clone(), A.clone(), 1e-3, 0.9, polar.default_coeffs(5, 5),
                                   5, 5)
    assert ei.value.name == "MAPL_ERR_UNSUPPORTED"
    assert "scratch" in str(ei.value)

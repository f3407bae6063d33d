"""Streaming codebook synchronisation on the GPU (MAPL §3.5, App. F): codes
applied to a plan with mapl_plan_update_codes behave exactly like a plan
created from the updated codebook (the oracle's apply_code_update), after
part of an epoch and after a full one."""
import numpy as np
import pytest

import oracle
import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import synth
from tests.helpers import to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


def _plan(w, b, C):
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    return mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(C))


def _codec(plan, w, b, n):
    X, t = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda()
    pay = torch.empty(plan.payload_shape(n), dtype=torch.uint8, device="cuda")
    xh = torch.empty(n, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_compress(plan, X, t, to_dev(b["E"]), pay)
    mapl.mapl_decompress(plan, pay, t, to_dev(b["E_next"]), xh)
    mapl.mapl_check(plan)
    torch.cuda.synchronize()
    return pay.cpu().numpy(), xh.cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("wname,steps", [("vq_d1024_r128", 2), ("vq_d1024_r128", None),
                                         ("vq_d2048_r128", 3)])
def test_streamed_plan_equals_fresh_plan(wname, steps):
    w = synth.WORKLOADS[wname]
    n = 600
    b = synth.make_boundary(w, seed=2, n_tokens=n)
    C0 = b["C"]
    # the sender's live codebook drifted: C1 = C0 + small noise, stored bf16
    rng = np.random.default_rng(17)
    C1 = synth.bf16_bits(synth.widen(C0) + 0.05 * rng.standard_normal(C0.shape))
    total = w.R * w.G * w.K
    per = total // 5
    n_sub = -(-total // per)
    steps = n_sub if steps is None else steps
    plan = _plan(w, b, C0)
    flat1 = C1.reshape(total, w.gd)
    mixed = synth.widen(C0)
    for step in range(steps):
        ids = mapl.mapl_stream_subset(total, per, 99, step)
        mapl.mapl_plan_update_codes(plan, torch.from_numpy(ids).cuda(), to_dev(flat1[ids]))
        mixed = oracle.apply_code_update(mixed, ids, synth.widen(flat1[ids]))
    fresh = _plan(w, b, synth.bf16_bits(mixed))
    got, want = _codec(plan, w, b, n), _codec(fresh, w, b, n)
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1], want[1])
    if steps == n_sub:
        assert np.array_equal(synth.bf16_bits(mixed), C1)


def test_update_codes_rejects_bad_ids():
    w = synth.WORKLOADS["vq_d1024_r128"]
    b = synth.make_boundary(w, seed=3, n_tokens=128)
    plan = _plan(w, b, b["C"])
    ids = torch.tensor([0, w.R * w.G * w.K], dtype=torch.int32, device="cuda")
    codes = to_dev(b["C"].reshape(-1, w.gd)[:2])
    mapl.mapl_plan_update_codes(plan, ids, codes)
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_check(plan)
    assert ei.value.name == "MAPL_ERR_INVALID_ARG"


@pytest.mark.parametrize("wname", ["vq_d1024_r128", "vq_d2048_r256"])
def test_whole_table_update_equals_fresh_plan(wname):
    """Every code replaced in one call (more codes than one block of the
    update takes, so the multi-block form with the last-block maxima runs),
    then the same payload and X_hat as a plan created from the new table."""
    w = synth.WORKLOADS[wname]
    n = 384
    b = synth.make_boundary(w, seed=5, n_tokens=n)
    total = w.R * w.G * w.K
    assert total > 512
    rng = np.random.default_rng(23)
    C1 = synth.bf16_bits(synth.widen(b["C"]) * 0.9 + 0.05 * rng.standard_normal(b["C"].shape))
    plan = _plan(w, b, b["C"])
    ids = np.arange(total, dtype=np.int32)[::-1].copy()   # every code, in reverse order
    flat1 = C1.reshape(total, w.gd)
    mapl.mapl_plan_update_codes(plan, torch.from_numpy(ids).cuda(), to_dev(flat1[ids]))
    fresh = _plan(w, b, C1)
    got, want = _codec(plan, w, b, n), _codec(fresh, w, b, n)
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1], want[1])

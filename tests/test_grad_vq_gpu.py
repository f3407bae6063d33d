"""MCVQ of backward gradients (MAPL §3.5: the multi-codebook quantiser
compresses forward activations and backward gradients) on the GPU vs the
fp64 oracle, via the C ABI.

The plan gets gradient codebooks of its own (mapl_plan_set_grad_codebooks);
mapl_grad_compress_vq quantises gZ = dL/dX_hat A (no anchor term) with them
and mapl_grad_decompress_vq returns dL/dX = gZ_hat A^T.  Indices are checked
like the forward ones (check_vq_indices: each index is the exact nearest code
of the GPU's own fp32 residual, and equal to the oracle's except on the
oracle's own flagged near ties), the GPU's fp32 gZ taken from mapl_compress_z32
with an all-zero anchor table (the anchor term then adds exact zeros after
the same X A accumulation); dL/dX is compared with the oracle's decode of the
GPU's indices at the bf16 tolerance.
"""
import numpy as np
import pytest

import oracle
import pipeline_activation_compression_gb300 as mapl
from pipeline_activation_compression_gb300 import synth
from tests.helpers import check_vq_indices, rel_frob, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


def _plan(w, b):
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    return mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(b["C"]))


@pytest.mark.parametrize("name,n", [("vq_d1024_r128", 1000), ("vq_d1024_r128", 129),
                                    ("vq_d2048_r128", 777), ("vq_d2048_r256", 500)])
def test_grad_vq_parity(name, n):
    w = synth.WORKLOADS[name]
    b = synth.make_boundary(w, seed=21, n_tokens=n)
    gxh = synth.make_boundary_grad(w, seed=21, n_tokens=n)
    Cg = synth.make_grad_codebooks(w, seed=21)
    plan = _plan(w, b)
    mapl.mapl_plan_set_grad_codebooks(plan, to_dev(Cg))
    gXh = to_dev(gxh)
    payload = torch.randint(0, 256, plan.payload_shape(n), dtype=torch.uint8, device="cuda")
    mapl.mapl_grad_compress_vq(plan, gXh, payload)
    gX = torch.full((n, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    mapl.mapl_grad_decompress_vq(plan, payload, gX)
    # the kernel's fp32 gZ: the same accumulation with a zero anchor
    Z32 = torch.full((n, w.r), float("nan"), dtype=torch.float32, device="cuda")
    zt = torch.zeros(n, dtype=torch.int32, device="cuda")
    zE = torch.zeros(w.V, w.r, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_compress_z32(plan, gXh, zt, zE, Z32)
    mapl.mapl_check(plan)
    torch.cuda.synchronize()
    Wd = synth.widen
    gZ_or = oracle.grad_compress(Wd(gxh), Wd(b["A"]))
    Z32h = Z32.cpu().numpy()
    assert rel_frob(Z32h, gZ_or) <= 1e-5
    idx = to_host(payload)
    check_vq_indices(idx, Z32h, gZ_or, Cg)
    gX_or = oracle.grad_decompress(oracle.rvq_decode(idx, Wd(Cg)), Wd(b["A"]))
    assert rel_frob(Wd(to_host(gX)), gX_or) <= TOL_BF16
    # the forward codebooks are untouched: the forward path still matches
    Zf = torch.empty(n, w.r, dtype=torch.float32, device="cuda")
    X, t, E = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda(), to_dev(b["E"])
    pf = torch.empty(plan.payload_shape(n), dtype=torch.uint8, device="cuda")
    mapl.mapl_compress(plan, X, t, E, pf)
    mapl.mapl_compress_z32(plan, X, t, E, Zf)
    mapl.mapl_check(plan)
    Zo = oracle.compress(Wd(b["X"]), b["tids"], Wd(b["A"]), Wd(b["E"]), Wd(b["P"]))
    check_vq_indices(to_host(pf), Zf.cpu().numpy(), Zo, b["C"])


def test_grad_vq_needs_codebooks_and_a_vq_plan():
    w = synth.WORKLOADS["vq_d1024_r128"]
    b = synth.make_boundary(w, seed=22, n_tokens=64)
    plan = _plan(w, b)
    gXh = to_dev(synth.make_boundary_grad(w, seed=22, n_tokens=64))
    payload = torch.empty(plan.payload_shape(64), dtype=torch.uint8, device="cuda")
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_grad_compress_vq(plan, gXh, payload)
    assert ei.value.name == "MAPL_ERR_INVALID_ARG"
    w0 = synth.WORKLOADS["proj_d1024_r128"]
    b0 = synth.make_boundary(w0, seed=22, n_tokens=64)
    cfg0 = mapl.make_config(w0.d, w0.r, w0.V, dtype=mapl.MAPL_BF16)
    plan0 = mapl.mapl_plan_create(cfg0, to_dev(b0["A"]), to_dev(b0["P"]), to_dev(b0["P_next"]))
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_plan_set_grad_codebooks(plan0, to_dev(synth.make_grad_codebooks(w)))
    assert ei.value.name == "MAPL_ERR_UNSUPPORTED"

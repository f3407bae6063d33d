"""Host-buffer forms of the codec calls (mapl_compress_host /
mapl_decompress_host) against the device forms, through the C ABI.

The host forms only stage data through a device workspace, so their outputs
must equal the device forms' bit for bit; a workspace one byte short and a
device tensor passed where host memory is expected must be refused.
"""
import numpy as np
import pytest

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


@pytest.mark.parametrize("wname,N", [("vq_d1024_r128", 1000), ("proj_d1024_r128", 777)])
@pytest.mark.parametrize("pin", [True, False])
def test_host_forms_equal_device_forms(wname, N, pin):
    w = synth.WORKLOADS[wname]
    b = synth.make_boundary(w, seed=11, n_tokens=N)
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    plan = mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(b["C"]) if w.vq else None)
    E, En = to_dev(b["E"]), to_dev(b["E_next"])
    # device forms
    X, t = to_dev(b["X"]), torch.from_numpy(b["tids"]).cuda()
    pay_d = torch.empty(plan.payload_shape(N), dtype=plan.payload_dtype(), device="cuda")
    xh_d = torch.empty(N, w.d, dtype=torch.bfloat16, device="cuda")
    mapl.mapl_compress(plan, X, t, E, pay_d)
    mapl.mapl_decompress(plan, pay_d, t, En, xh_d)
    # host forms
    ws = torch.empty(mapl.mapl_host_workspace_size(plan, N), dtype=torch.uint8, device="cuda")
    X_host = X.cpu()
    t_host = t.cpu()
    if pin:
        X_host, t_host = X_host.pin_memory(), t_host.pin_memory()
    pay_h = torch.empty(plan.payload_shape(N), dtype=plan.payload_dtype(), pin_memory=pin)
    xh_h = torch.empty(N, w.d, dtype=torch.bfloat16, pin_memory=pin)
    mapl.mapl_compress_host(plan, X_host, t_host, E, pay_h, ws)
    mapl.mapl_decompress_host(plan, pay_h, t_host, En, xh_h, ws)
    mapl.mapl_check(plan)
    torch.cuda.synchronize()
    assert torch.equal(pay_h, pay_d.cpu())
    assert torch.equal(xh_h.view(torch.int16), xh_d.cpu().view(torch.int16))


def test_host_forms_refuse_bad_arguments():
    w = synth.WORKLOADS["vq_d1024_r128"]
    N = 256
    b = synth.make_boundary(w, seed=12, n_tokens=N)
    cfg = mapl.make_config(w.d, w.r, w.V, w.G, w.R, w.K, mapl.MAPL_BF16)
    plan = mapl.mapl_plan_create(cfg, to_dev(b["A"]), to_dev(b["P"]), to_dev(b["P_next"]),
                                 to_dev(b["C"]))
    need = mapl.mapl_host_workspace_size(plan, N)
    X_host = to_dev(b["X"]).cpu().pin_memory()
    t_host = torch.from_numpy(b["tids"]).pin_memory()
    pay_h = torch.empty(plan.payload_shape(N), dtype=torch.uint8, pin_memory=True)
    short = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_compress_host(plan, X_host, t_host, to_dev(b["E"]), pay_h, short)
    assert ei.value.name == "MAPL_ERR_INVALID_ARG"
    with pytest.raises(ValueError):
        mapl.mapl_compress_host(plan, X_host.cuda(), t_host, to_dev(b["E"]), pay_h,
                                torch.empty(need, dtype=torch.uint8, device="cuda"))

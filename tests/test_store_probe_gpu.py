"""The write-rate probe (mapl_store_probe) writes zeros over exactly the bytes
it is given, by each of its store paths, and rejects misaligned requests."""
import pytest

import pipeline_activation_compression_gb300 as mapl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mapl.build()
    mapl.load_library()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("n16", [1, 7, 2048, 2048 * 152 + 3, (64 << 20) // 16 + 5])
def test_store_probe_zeroes_exactly_its_range(mode, n16):
    buf = torch.full((n16 * 4 + 8,), -1, dtype=torch.int32, device="cuda")
    dst = buf[4:4 + n16 * 4]   # 16-byte aligned view, guards on both sides
    mapl.mapl_store_probe(dst, mode)
    torch.cuda.synchronize()
    assert int((dst != 0).sum()) == 0
    assert int((buf[:4] != -1).sum()) == 0 and int((buf[-4:] != -1).sum()) == 0


def test_store_probe_rejects_bad_arguments():
    lib = mapl.load_library()
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    assert lib.mapl_store_probe(p + 4, 32, 0, None) == 1     # misaligned
    assert lib.mapl_store_probe(p, 24, 0, None) == 1         # not a multiple of 16
    assert lib.mapl_store_probe(p, 32, 3, None) == 1         # no such mode
    assert lib.mapl_store_probe(None, 32, 0, None) == 1
    assert lib.mapl_store_probe(p, 0, 2, None) == 0          # nothing to write

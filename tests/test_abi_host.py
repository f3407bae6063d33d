"""The C-ABI library loads, exports every declared entry point, and rejects
bad arguments on the host (no GPU work is issued by these calls)."""
import os
import re

import pytest

import pipeline_activation_compression_gb300 as mapl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mapl.build()
    return mapl.load_library()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(mapl_[A-Za-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert mapl.mapl_version() >= 100


def test_payload_bytes_host():
    c = mapl.make_config(1024, 128, 32000, 4, 2, 256, mapl.MAPL_BF16)
    assert mapl.mapl_payload_bytes(c) == 8                      # R*G uint8 indices
    c = mapl.make_config(1024, 256, 32000, dtype=mapl.MAPL_BF16)
    assert mapl.mapl_payload_bytes(c) == 512                    # 2r bytes of bf16 Z
    c = mapl.make_config(64, 16, 512, 1, 2, 16, mapl.MAPL_F32)
    assert mapl.mapl_payload_bytes(c) == 2


@pytest.mark.parametrize("cfg,status", [
    (dict(d=1000, r=128, V=10), "MAPL_ERR_INVALID_ARG"),          # d % 64
    (dict(d=1024, r=100, V=10), "MAPL_ERR_INVALID_ARG"),          # r % 16
    (dict(d=1024, r=1024, V=10), "MAPL_ERR_INVALID_ARG"),         # r > 512
    (dict(d=1024, r=128, V=0), "MAPL_ERR_INVALID_ARG"),           # V
    (dict(d=1024, r=128, V=10, G=3, R=2, K=256), "MAPL_ERR_INVALID_ARG"),   # G does not divide r
    (dict(d=1024, r=128, V=10, G=4, R=2, K=300), "MAPL_ERR_INVALID_ARG"),   # K > 256 (uint8 ids)
    (dict(d=1024, r=128, V=10, G=4, R=9, K=256), "MAPL_ERR_INVALID_ARG"),   # R > 8
    (dict(d=1024, r=96, V=10), "MAPL_ERR_UNSUPPORTED"),           # bf16 tensor path: r % 64
    (dict(d=1024, r=128, V=10, G=64, R=2, K=256), "MAPL_ERR_UNSUPPORTED"),  # group width 2
    (dict(d=1024, r=512, V=10, G=8, R=2, K=256), "MAPL_ERR_UNSUPPORTED"),   # r + K > 512
])
def test_config_validation_host(lib, cfg, status):
    c = mapl.make_config(cfg["d"], cfg["r"], cfg["V"], cfg.get("G", 0), cfg.get("R", 0),
                         cfg.get("K", 0), mapl.MAPL_BF16)
    with pytest.raises(mapl.MaplError) as ei:
        mapl.mapl_payload_bytes(c)
    assert ei.value.name == status


def test_spel_workspace_host(lib):
    b = mapl.mapl_spel_workspace_size(1024, 256, 3)
    assert b >= 3 * 2 * 1024 * 256 * 4
    with pytest.raises(mapl.MaplError):
        mapl.mapl_spel_workspace_size(1024, 2048, 3)   # r > d


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(mapl, "_LIB", None)
    monkeypatch.setattr(mapl, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        mapl.load_library()

"""MAPL boundary codec on GB300: thin Python binding of ``libmapl.so``.

Functions carry the names of the C ABI in ``include/mapl.h`` and only marshal
arguments: torch tensors become device pointers, the current torch stream
becomes the CUDA stream.  Every step of the codec runs in the library's CUDA
kernels; there is no other implementation behind these calls.  Importing the
package does not need a GPU; calling into the library needs the built
``libmapl.so`` (``build()``) and fails loudly without it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "MaplError", "MaplConfig", "Plan", "load_library", "library_path", "build",
    "mapl_plan_create", "mapl_plan_update_A", "mapl_plan_set_embedding_anchor",
    "mapl_payload_bytes", "mapl_compress",
    "mapl_compress_z32", "mapl_decompress", "mapl_check", "mapl_plan_destroy",
    "mapl_host_workspace_size", "mapl_compress_host", "mapl_decompress_host",
    "mapl_grad_compress", "mapl_grad_decompress", "mapl_grad_workspace_size", "mapl_grad_A",
    "mapl_plan_set_grad_codebooks", "mapl_grad_compress_vq", "mapl_grad_decompress_vq",
    "mapl_stream_subset", "mapl_plan_update_codes", "mapl_selftest_bounded_wait",
    "mapl_store_probe",
    "mapl_spel_workspace_size", "mapl_spel_step", "mapl_spel_step_refresh",
    "mapl_spel_step_static", "mapl_last_error",
    "mapl_version",
    "MAPL_F32", "MAPL_BF16", "STATUS",
]

MAPL_F32, MAPL_BF16 = 0, 1
STATUS = {0: "MAPL_OK", 1: "MAPL_ERR_INVALID_ARG", 2: "MAPL_ERR_UNSUPPORTED",
          3: "MAPL_ERR_CUDA", 4: "MAPL_ERR_BAD_TOKEN", 5: "MAPL_ERR_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


class MaplError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{self.name}: {message}")


class MaplConfig(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int64), ("r", ctypes.c_int64), ("V", ctypes.c_int64),
                ("G", ctypes.c_int32), ("R", ctypes.c_int32), ("K", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


def library_path() -> str:
    return os.path.join(_HERE, "libmapl.so")


def build(force: bool = False, verbose: bool = False) -> str:
    from . import _build
    return _build.build(force=force, verbose=verbose)


def load_library():
    """Load libmapl.so (built in-tree); raise if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: call pipeline_activation_compression_gb300.build()")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "mapl_plan_create": [ctypes.POINTER(P), ctypes.POINTER(MaplConfig), P, P, P, P, P],
        "mapl_plan_update_A": [P, P, P],
        "mapl_plan_set_embedding_anchor": [P, P, P],
        "mapl_payload_bytes": [ctypes.POINTER(MaplConfig), ctypes.POINTER(I64)],
        "mapl_compress": [P, P, P, I64, P, P, P],
        "mapl_compress_z32": [P, P, P, I64, P, P, P],
        "mapl_decompress": [P, P, P, I64, P, P, P],
        "mapl_check": [P, P],
        "mapl_selftest_bounded_wait": [P, I64, ctypes.POINTER(I64), P],
        "mapl_store_probe": [P, SZ, I32, P],
        "mapl_host_workspace_size": [P, I64, ctypes.POINTER(SZ)],
        "mapl_grad_compress": [P, P, I64, P, P],
        "mapl_grad_decompress": [P, P, I64, P, P],
        "mapl_grad_workspace_size": [P, I64, ctypes.POINTER(SZ)],
        "mapl_plan_set_grad_codebooks": [P, P, P],
        "mapl_grad_compress_vq": [P, P, I64, P, P],
        "mapl_grad_decompress_vq": [P, P, I64, P, P],
        "mapl_grad_A": [P, P, P, P, P, P, P, I64, P, P, SZ, P],
        "mapl_stream_subset": [I64, I64, ctypes.c_uint64, I64, P, ctypes.POINTER(I32)],
        "mapl_plan_update_codes": [P, P, I32, P, P],
        "mapl_compress_host": [P, P, P, I64, P, P, P, SZ, P],
        "mapl_decompress_host": [P, P, P, I64, P, P, P, SZ, P],
        "mapl_spel_workspace_size": [I64, I64, I32, ctypes.POINTER(SZ)],
        "mapl_spel_step": [P, P, P, I64, I64, I32, ctypes.c_float, ctypes.c_float, P, I32, I32,
                           P, SZ, P],
        "mapl_spel_step_static": [P, P, P, I64, I64, I32, ctypes.c_float, ctypes.c_float, P,
                                  I32, I32, P],
        "mapl_spel_step_refresh": [P, P, P, I64, I64, I32, ctypes.c_float, ctypes.c_float, P,
                                   I32, I32, P, P, SZ, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.mapl_plan_destroy.argtypes = [P]
    lib.mapl_plan_destroy.restype = None
    lib.mapl_last_error.argtypes = []
    lib.mapl_last_error.restype = ctypes.c_char_p
    lib.mapl_version.argtypes = []
    lib.mapl_version.restype = ctypes.c_int32
    _LIB = lib
    return lib


def mapl_last_error() -> str:
    return load_library().mapl_last_error().decode()


def mapl_version() -> int:
    return int(load_library().mapl_version())


def _check(status: int):
    if status != 0:
        raise MaplError(status, mapl_last_error())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t, dtype=None, what="tensor"):
    """Device pointer of a contiguous CUDA tensor (checked dtype)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must have dtype {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _tdtype(dt: int):
    import torch
    return torch.bfloat16 if dt == MAPL_BF16 else torch.float32


class Plan:
    """Owning handle of a ``mapl_plan``; destroyed with the object."""

    def __init__(self, handle, cfg: MaplConfig):
        self.handle = handle
        self.cfg = cfg

    @property
    def vq(self) -> bool:
        return self.cfg.G > 0

    def payload_shape(self, N: int):
        return (N, self.cfg.R, self.cfg.G) if self.vq else (N, self.cfg.r)

    def payload_dtype(self):
        import torch
        return torch.uint8 if self.vq else _tdtype(self.cfg.dtype)

    def destroy(self):
        if self.handle is not None and _LIB is not None:
            _LIB.mapl_plan_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def make_config(d, r, V, G=0, R=0, K=0, dtype=MAPL_BF16) -> MaplConfig:
    return MaplConfig(d, r, V, G, R, K, dtype, 0)


def mapl_payload_bytes(cfg: MaplConfig) -> int:
    out = ctypes.c_int64(0)
    _check(load_library().mapl_payload_bytes(ctypes.byref(cfg), ctypes.byref(out)))
    return int(out.value)


def mapl_plan_create(cfg: MaplConfig, A, P_send, P_recv, codebooks=None, stream=None) -> Plan:
    lib = load_library()
    dt = _tdtype(cfg.dtype)
    h = ctypes.c_void_p()
    _check(lib.mapl_plan_create(ctypes.byref(h), ctypes.byref(cfg), _ptr(A, dt, "A"),
                                _ptr(P_send, dt, "P_send"), _ptr(P_recv, dt, "P_recv"),
                                _ptr(codebooks, dt, "codebooks"), _stream(stream)))
    return Plan(h, cfg)


def mapl_plan_update_A(plan: Plan, A, stream=None):
    _check(load_library().mapl_plan_update_A(plan.handle, _ptr(A, _tdtype(plan.cfg.dtype), "A"),
                                             _stream(stream)))


def mapl_plan_set_embedding_anchor(plan: Plan, E_emb, stream=None):
    """First-boundary anchor: the plan keeps a reference to E_emb (V x d bf16)."""
    _check(load_library().mapl_plan_set_embedding_anchor(
        plan.handle, _ptr(E_emb, _tdtype(plan.cfg.dtype), "E_emb"), _stream(stream)))
    plan.E_emb = E_emb


def mapl_compress(plan: Plan, X, tids, E_send, payload, stream=None):
    import torch
    dt = _tdtype(plan.cfg.dtype)
    _check(load_library().mapl_compress(
        plan.handle, _ptr(X, dt, "X"), _ptr(tids, torch.int32, "tids"), int(X.shape[0]),
        _ptr(E_send, dt, "E_send"), _ptr(payload, plan.payload_dtype(), "payload"),
        _stream(stream)))
    return payload


def mapl_compress_z32(plan: Plan, X, tids, E_send, Z, stream=None):
    import torch
    dt = _tdtype(plan.cfg.dtype)
    _check(load_library().mapl_compress_z32(
        plan.handle, _ptr(X, dt, "X"), _ptr(tids, torch.int32, "tids"), int(X.shape[0]),
        _ptr(E_send, dt, "E_send"), _ptr(Z, torch.float32, "Z"), _stream(stream)))
    return Z


def mapl_decompress(plan: Plan, payload, tids, E_recv, X_hat, stream=None):
    import torch
    dt = _tdtype(plan.cfg.dtype)
    _check(load_library().mapl_decompress(
        plan.handle, _ptr(payload, plan.payload_dtype(), "payload"),
        _ptr(tids, torch.int32, "tids"), int(tids.shape[0]), _ptr(E_recv, dt, "E_recv"),
        _ptr(X_hat, dt, "X_hat"), _stream(stream)))
    return X_hat


def _host_ptr(t, dtype, what):
    """Address of a contiguous CPU tensor (pinned for asynchronous copies)."""
    if t.is_cuda:
        raise ValueError(f"{what} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must have dtype {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def mapl_host_workspace_size(plan: Plan, N: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().mapl_host_workspace_size(plan.handle, int(N), ctypes.byref(out)))
    return int(out.value)


def mapl_compress_host(plan: Plan, X, tids, E_send, payload, workspace, stream=None):
    """X, tids, payload: host tensors; E_send, workspace: device tensors."""
    import torch
    dt = _tdtype(plan.cfg.dtype)
    _check(load_library().mapl_compress_host(
        plan.handle, _host_ptr(X, dt, "X"), _host_ptr(tids, torch.int32, "tids"),
        int(X.shape[0]), _ptr(E_send, dt, "E_send"),
        _host_ptr(payload, plan.payload_dtype(), "payload"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return payload


def mapl_decompress_host(plan: Plan, payload, tids, E_recv, X_hat, workspace, stream=None):
    """payload, tids, X_hat: host tensors; E_recv, workspace: device tensors."""
    import torch
    dt = _tdtype(plan.cfg.dtype)
    _check(load_library().mapl_decompress_host(
        plan.handle, _host_ptr(payload, plan.payload_dtype(), "payload"),
        _host_ptr(tids, torch.int32, "tids"), int(tids.shape[0]), _ptr(E_recv, dt, "E_recv"),
        _host_ptr(X_hat, dt, "X_hat"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return X_hat


def mapl_grad_compress(plan: Plan, gX_hat, gZ, stream=None):
    """gZ = gX_hat A (receiver side of the backward pass); bf16 device tensors."""
    import torch
    _check(load_library().mapl_grad_compress(
        plan.handle, _ptr(gX_hat, torch.bfloat16, "gX_hat"), int(gX_hat.shape[0]),
        _ptr(gZ, torch.bfloat16, "gZ"), _stream(stream)))
    return gZ


def mapl_grad_decompress(plan: Plan, gZ, gX, stream=None):
    """gX = gZ A^T (sender side of the backward pass); bf16 device tensors."""
    import torch
    _check(load_library().mapl_grad_decompress(
        plan.handle, _ptr(gZ, torch.bfloat16, "gZ"), int(gZ.shape[0]),
        _ptr(gX, torch.bfloat16, "gX"), _stream(stream)))
    return gX


def mapl_plan_set_grad_codebooks(plan: Plan, codebooks, stream=None):
    """Gradient codebooks (R x G x K x gd bf16 device tensor) for the MCVQ of
    backward gradients."""
    import torch
    _check(load_library().mapl_plan_set_grad_codebooks(
        plan.handle, _ptr(codebooks, torch.bfloat16, "codebooks"), _stream(stream)))


def mapl_grad_compress_vq(plan: Plan, gX_hat, payload, stream=None):
    """payload (N x R*G uint8) = the gradient codebooks' RVQ of gZ = gX_hat A."""
    import torch
    _check(load_library().mapl_grad_compress_vq(
        plan.handle, _ptr(gX_hat, torch.bfloat16, "gX_hat"), int(gX_hat.shape[0]),
        _ptr(payload, torch.uint8, "payload"), _stream(stream)))
    return payload


def mapl_grad_decompress_vq(plan: Plan, payload, gX, stream=None):
    """gX (N x d bf16) = gZ_hat A^T, gZ_hat decoded from the payload with the
    gradient codebooks."""
    import torch
    _check(load_library().mapl_grad_decompress_vq(
        plan.handle, _ptr(payload, torch.uint8, "payload"), int(payload.shape[0]),
        _ptr(gX, torch.bfloat16, "gX"), _stream(stream)))
    return gX


def mapl_grad_workspace_size(plan: Plan, N: int) -> int:
    """Bytes of device workspace mapl_grad_A needs for N tokens."""
    n = ctypes.c_size_t(0)
    _check(load_library().mapl_grad_workspace_size(plan.handle, int(N), ctypes.byref(n)))
    return int(n.value)


def mapl_grad_A(plan: Plan, X, tids, E_send, gZ, gX_hat, Z, dA, workspace=None, stream=None):
    """dA = (X - E_send[tids] P_send)^T gZ + gX_hat^T Z, fp32 d x r.  The
    workspace (a device tensor of at least mapl_grad_workspace_size bytes) is
    the caller's; without one a tensor of that size is made for the call."""
    import torch
    N = int(X.shape[0])
    if workspace is None:
        workspace = torch.empty(mapl_grad_workspace_size(plan, N), dtype=torch.uint8,
                                device=X.device)
    _check(load_library().mapl_grad_A(
        plan.handle, _ptr(X, torch.bfloat16, "X"), _ptr(tids, torch.int32, "tids"),
        _ptr(E_send, torch.bfloat16, "E_send"), _ptr(gZ, torch.bfloat16, "gZ"),
        _ptr(gX_hat, torch.bfloat16, "gX_hat"), _ptr(Z, torch.bfloat16, "Z"),
        N, _ptr(dA, torch.float32, "dA"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return dA


def mapl_stream_subset(total: int, per_batch: int, seed: int, step: int) -> np.ndarray:
    """Code ids (flat over R x G x K) to refresh at micro-batch `step`; host only."""
    ids = np.empty(int(per_batch), dtype=np.int32)
    n = ctypes.c_int32(0)
    _check(load_library().mapl_stream_subset(int(total), int(per_batch), ctypes.c_uint64(seed),
                                             int(step), ids.ctypes.data_as(ctypes.c_void_p),
                                             ctypes.byref(n)))
    return ids[:n.value].copy()


def mapl_plan_update_codes(plan: Plan, ids, codes, stream=None):
    """Codes ids[i] (device int32) take the values codes[i] (device, count x gd)."""
    import torch
    _check(load_library().mapl_plan_update_codes(
        plan.handle, _ptr(ids, torch.int32, "ids"), int(ids.numel()),
        _ptr(codes, _tdtype(plan.cfg.dtype), "codes"), _stream(stream)))


def mapl_check(plan: Plan, stream=None):
    """Synchronise and raise MaplError if a kernel flagged a data error."""
    _check(load_library().mapl_check(plan.handle, _stream(stream)))


def mapl_store_probe(dst, mode: int = 0, stream=None) -> None:
    """Write zeros over the device tensor `dst` (no reads) by store path
    `mode` (0: 16-byte stores, 1: streaming stores, 2: bulk async copies):
    the write-rate probe."""
    _check(load_library().mapl_store_probe(_ptr(dst), dst.numel() * dst.element_size(),
                                           int(mode), _stream(stream)))


def mapl_selftest_bounded_wait(plan: Plan, budget_ns: int, stream=None) -> int:
    """Run the kernels' bounded wait on a barrier nothing completes; returns
    the nanoseconds waited.  The plan's next mapl_check reports the timeout."""
    out = ctypes.c_int64(0)
    _check(load_library().mapl_selftest_bounded_wait(plan.handle, int(budget_ns),
                                                     ctypes.byref(out), _stream(stream)))
    return int(out.value)


def mapl_plan_destroy(plan: Plan):
    plan.destroy()


def mapl_spel_workspace_size(d: int, r: int, batch: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().mapl_spel_workspace_size(int(d), int(r), int(batch), ctypes.byref(out)))
    return int(out.value)


def mapl_spel_step(A, G, m, lr: float, beta: float, coeffs, n_lmo: int, n_retr: int,
                   workspace, stream=None):
    """In-place SPEL update of A (batch x d x r) and m; coeffs: (n_lmo+n_retr) x 3."""
    import torch
    co = np.ascontiguousarray(np.asarray(coeffs, dtype=np.float32).reshape(-1))
    if co.size != 3 * (n_lmo + n_retr):
        raise ValueError("coeffs must hold (n_lmo + n_retr) rows of (a, b, c)")
    b, d, r = A.shape
    _check(load_library().mapl_spel_step(
        _ptr(A, torch.float32, "A"), _ptr(G, torch.float32, "G"), _ptr(m, torch.float32, "m"),
        d, r, b, float(lr), float(beta), co.ctypes.data_as(ctypes.c_void_p), int(n_lmo),
        int(n_retr), _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def mapl_spel_step_refresh(A, G, m, lr: float, beta: float, coeffs, n_lmo: int, n_retr: int,
                           plans, workspace, stream=None):
    """mapl_spel_step, then plans[b] (a Plan or None per boundary) refreshed
    from bf16(A[b]) by the same launches (see include/mapl.h)."""
    import torch
    co = np.ascontiguousarray(np.asarray(coeffs, dtype=np.float32).reshape(-1))
    if co.size != 3 * (n_lmo + n_retr):
        raise ValueError("coeffs must hold (n_lmo + n_retr) rows of (a, b, c)")
    b, d, r = A.shape
    if len(plans) != b:
        raise ValueError("plans must hold one entry (Plan or None) per boundary")
    handles = (ctypes.c_void_p * b)(*[None if p is None else p.handle for p in plans])
    _check(load_library().mapl_spel_step_refresh(
        _ptr(A, torch.float32, "A"), _ptr(G, torch.float32, "G"), _ptr(m, torch.float32, "m"),
        d, r, b, float(lr), float(beta), co.ctypes.data_as(ctypes.c_void_p), int(n_lmo),
        int(n_retr), ctypes.cast(handles, ctypes.c_void_p), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def mapl_spel_step_static(A, G, m, lr: float, beta: float, coeffs, n_lmo: int, n_retr: int,
                          stream=None):
    """SPEL update without a workspace argument, for callers that cannot
    allocate: the library's fixed 16 MiB device scratch is used instead (see
    include/mapl.h).  Calls that overlap on the GPU race on that scratch."""
    import torch
    co = np.ascontiguousarray(np.asarray(coeffs, dtype=np.float32).reshape(-1))
    if co.size != 3 * (n_lmo + n_retr):
        raise ValueError("coeffs must hold (n_lmo + n_retr) rows of (a, b, c)")
    b, d, r = A.shape
    _check(load_library().mapl_spel_step_static(
        _ptr(A, torch.float32, "A"), _ptr(G, torch.float32, "G"), _ptr(m, torch.float32, "m"),
        d, r, b, float(lr), float(beta), co.ctypes.data_as(ctypes.c_void_p), int(n_lmo),
        int(n_retr), _stream(stream)))

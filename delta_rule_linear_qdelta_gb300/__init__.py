"""GB300-native (sm_103a) Q-Delta / QED chunked forward and decode step.

A thin ctypes binding of the C ABI in include/qdelta.h: it checks tensor
metadata, allocates outputs with torch when the caller does not pass them, and
calls the library on the current CUDA stream.  Every step of the computation
runs in the library's CUDA kernels; there is no CPU path.  If the shared
library is missing this module raises instead of computing anything.

Functions keep the C names: qdelta_fwd, qed_fwd (with its ablation arms, the C
qed_fwd_variant), qdelta_step, qed_step, qdelta_fwd_static_scratch,
qdelta_workspace_bytes, qed_workspace_bytes, qd_device_status, qd_last_error.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqdelta_gb300.so")

QD_OK, QD_ERR_ARG, QD_ERR_UNSUPPORTED, QD_ERR_CUDA, QD_ERR_TIMEOUT, QD_ERR_WORKSPACE = range(6)
QD_F32, QD_BF16 = 0, 1
STATUS_NAMES = {0: "QD_OK", 1: "QD_ERR_ARG", 2: "QD_ERR_UNSUPPORTED", 3: "QD_ERR_CUDA",
                4: "QD_ERR_TIMEOUT", 5: "QD_ERR_WORKSPACE"}
EXPORTS = ("qdelta_fwd", "qdelta_fwd_prologue", "qdelta_workspace_bytes", "qed_fwd", "qed_fwd_variant",
           "qed_workspace_bytes", "qdelta_step", "qdelta_step_prologue", "qed_step", "qdelta_fwd_static_scratch",
           "qdelta_bwd", "qdelta_bwd_workspace_bytes", "qdelta_bwd_prologue", "qdelta_bwd_prologue_workspace_bytes",
           "eda_fwd", "eda_workspace_bytes", "qd_device_status",
           "qd_selftest_bounded_wait",
           "qd_last_error",
           "qd_last_launch_count")
QED_VARIANTS = {"full": 0, "nogate": 1, "nogate_noproj": 2, "rand": 3}


class QDError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the CUDA library (no GPU needed to load).  Raises if it is not built."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: call delta_rule_linear_qdelta_gb300.build.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.qdelta_fwd.argtypes = [P] * 9 + [I] * 7 + [P, Z, P]
    lib.qdelta_fwd_prologue.argtypes = [P] * 9 + [I] * 7 + [P, Z, P]
    lib.qdelta_step_prologue.argtypes = [P] * 8 + [I] * 5 + [P]
    lib.qdelta_fwd_static_scratch.argtypes = [P] * 9 + [I] * 7 + [P]
    lib.qed_fwd.argtypes = [P] * 10 + [I] * 7 + [P, Z, P]
    lib.qdelta_step.argtypes = [P] * 8 + [I] * 5 + [P]
    lib.qed_fwd_variant.argtypes = [P] * 10 + [I] * 8 + [P, P, Z, P]
    lib.qed_step.argtypes = [P] * 9 + [I] * 6 + [P, P]
    lib.qdelta_workspace_bytes.argtypes = [I] * 7
    lib.qed_workspace_bytes.argtypes = [I] * 7
    lib.qdelta_bwd.argtypes = [P] * 16 + [I] * 7 + [P, Z, P]
    lib.qdelta_bwd_workspace_bytes.argtypes = [I] * 7
    lib.qdelta_bwd_prologue.argtypes = [P] * 16 + [I] * 7 + [P, Z, P]
    lib.qdelta_bwd_prologue.restype = I
    lib.qdelta_bwd_prologue_workspace_bytes.argtypes = [I] * 7
    lib.qdelta_bwd_prologue_workspace_bytes.restype = Z
    lib.eda_fwd.argtypes = [P] * 8 + [I] * 7 + [P, Z, P]
    lib.eda_workspace_bytes.argtypes = [I] * 7
    lib.eda_fwd.restype = I
    lib.eda_workspace_bytes.restype = Z
    lib.qd_device_status.argtypes = [P]
    lib.qd_selftest_bounded_wait.argtypes = [ctypes.c_uint, P]
    lib.qd_selftest_bounded_wait.restype = I
    for f in (lib.qdelta_fwd, lib.qed_fwd, lib.qdelta_step, lib.qdelta_fwd_static_scratch, lib.qd_device_status,
              lib.qd_last_launch_count, lib.qed_fwd_variant, lib.qed_step, lib.qdelta_fwd_prologue,
              lib.qdelta_step_prologue, lib.qdelta_bwd):
        f.restype = I
    lib.qdelta_workspace_bytes.restype = Z
    lib.qed_workspace_bytes.restype = Z
    lib.qdelta_bwd_workspace_bytes.restype = Z
    lib.qd_last_error.restype = ctypes.c_char_p
    lib.qd_last_error.argtypes = []
    lib.qd_last_launch_count.argtypes = []
    if path == LIB_PATH:
        _lib = lib
    return lib


def qd_last_error() -> str:
    return load_library().qd_last_error().decode()


def last_launch_count() -> int:
    """Kernels launched by the last successful compute call on this thread."""
    return load_library().qd_last_launch_count()


def _check(status: int, fn: str):
    if status != QD_OK:
        raise QDError(status, fn, qd_last_error())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return QD_BF16
    if t.dtype == torch.float32:
        return QD_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor | None, name: str, dtype, shape, optional: bool = False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _same_device(device, *tensors):
    for t in tensors:
        if t is not None and t.device != device:
            raise ValueError(f"tensor on {t.device}, expected every argument on {device}")


def _call(device, fn, *args):
    """Runs one C call with `device` current: the library takes the SM count, the
    TMA descriptors and the static scratch address from the current device."""
    with torch.cuda.device(device):
        return fn(*args)


def _stream(stream, device):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def qdelta_workspace_bytes(B, T, H, dk, dv, chunk=64, dtype=QD_BF16) -> int:
    return load_library().qdelta_workspace_bytes(B, T, H, dk, dv, chunk, dtype)


def qed_workspace_bytes(B, T, H, dk, dv, chunk=64, dtype=QD_BF16) -> int:
    return load_library().qed_workspace_bytes(B, T, H, dk, dv, chunk, dtype)


def _workspace(nbytes, workspace, device):
    if nbytes == 0:
        return workspace, 0 if workspace is None else workspace.numel() * workspace.element_size()
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def qdelta_fwd(q, k, v, alpha, beta, lam, S0=None, *, o=None, S_final=None, return_final=True,
               chunk=64, workspace=None, stream=None, prologue=False):
    """Chunked Q-Delta forward.  q, k [B,T,H,dk]; v [B,T,H,dv]; alpha, beta, lam [B,T,H]
    (alpha None = 1, lam None = 0); S0 [B,H,dv,dk] fp32 or None.  Returns (o, S_final).
    prologue=True: q, k are projections and alpha, beta, lam logits; the feature map
    SiLU(x)/|SiLU(x)| and the gates (exp(-softplus), sigmoid, sigmoid) are applied
    inside (the C qdelta_fwd_prologue)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    _need(q, "q", dt, (B, T, H, dk))
    _need(k, "k", dt, (B, T, H, dk))
    _need(v, "v", dt, (B, T, H, dv))
    _need(beta, "beta", dt, (B, T, H))
    _need(alpha, "alpha", dt, (B, T, H), optional=True)
    _need(lam, "lam", dt, (B, T, H), optional=True)
    _need(S0, "S0", torch.float32, (B, H, dv, dk), optional=True)
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=dt, device=q.device)
    _need(o, "o", dt, (B, T, H, dv))
    if S_final is None and return_final:
        S_final = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    _need(S_final, "S_final", torch.float32, (B, H, dv, dk), optional=True)
    code = _dtype_code(q)
    workspace, wsb = _workspace(qdelta_workspace_bytes(B, T, H, dk, dv, chunk, code), workspace, q.device)
    _same_device(q.device, k, v, alpha, beta, lam, S0, o, S_final, workspace)
    fn = load_library().qdelta_fwd_prologue if prologue else load_library().qdelta_fwd
    st = _call(q.device, fn, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(lam), _ptr(S0), _ptr(o),
               _ptr(S_final), B, T, H, dk, dv, chunk, code, _ptr(workspace), wsb, _stream(stream, q.device))
    _check(st, "qdelta_fwd_prologue" if prologue else "qdelta_fwd")
    return o, S_final


def qdelta_bwd_workspace_bytes(B, T, H, dk, dv, chunk=64, dtype=QD_BF16) -> int:
    return load_library().qdelta_bwd_workspace_bytes(B, T, H, dk, dv, chunk, dtype)


def qdelta_bwd(q, k, v, alpha, beta, lam, S0, dO, dS_final=None, *, want_dS0=True, chunk=64, workspace=None,
               stream=None, prologue=False):
    """Backward of qdelta_fwd: gradients of sum(dO * o) + sum(dS_final * S_final)
    (the C qdelta_bwd).  Inputs as for qdelta_fwd, dO [B,T,H,dv] in the inputs' dtype,
    dS_final [B,H,dv,dk] fp32 or None.  Returns a dict dq, dk, dv, dalpha (None when
    alpha is None), dbeta, dlam (None when lam is None), dS0 (fp32; None unless
    want_dS0), the token and gate gradients in the inputs' dtype.  prologue=True: the
    backward of qdelta_fwd(..., prologue=True), i.e. q, k are projections and alpha, beta,
    lam logits, and the gradients are theirs (the C qdelta_bwd_prologue)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    _need(q, "q", dt, (B, T, H, dk))
    _need(k, "k", dt, (B, T, H, dk))
    _need(v, "v", dt, (B, T, H, dv))
    _need(beta, "beta", dt, (B, T, H))
    _need(alpha, "alpha", dt, (B, T, H), optional=True)
    _need(lam, "lam", dt, (B, T, H), optional=True)
    _need(S0, "S0", torch.float32, (B, H, dv, dk), optional=True)
    _need(dO, "dO", dt, (B, T, H, dv))
    _need(dS_final, "dS_final", torch.float32, (B, H, dv, dk), optional=True)
    g = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
         "dalpha": None if alpha is None else torch.empty_like(alpha), "dbeta": torch.empty_like(beta),
         "dlam": None if lam is None else torch.empty_like(lam),
         "dS0": torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device) if want_dS0 else None}
    code = _dtype_code(q)
    lib = load_library()
    nbytes = (lib.qdelta_bwd_prologue_workspace_bytes if prologue else lib.qdelta_bwd_workspace_bytes)(
        B, T, H, dk, dv, chunk, code)
    workspace, wsb = _workspace(nbytes, workspace, q.device)
    _same_device(q.device, k, v, alpha, beta, lam, S0, dO, dS_final, workspace)
    st = _call(q.device, lib.qdelta_bwd_prologue if prologue else lib.qdelta_bwd, _ptr(q), _ptr(k), _ptr(v),
               _ptr(alpha), _ptr(beta), _ptr(lam), _ptr(S0), _ptr(dO), _ptr(dS_final), _ptr(g["dq"]),
               _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dalpha"]), _ptr(g["dbeta"]), _ptr(g["dlam"]), _ptr(g["dS0"]),
               B, T, H, dk, dv, chunk, code, _ptr(workspace), wsb, _stream(stream, q.device))
    _check(st, "qdelta_bwd_prologue" if prologue else "qdelta_bwd")
    return g


def eda_workspace_bytes(B, T, H, dk, dv, chunk=64, dtype=QD_BF16) -> int:
    return load_library().eda_workspace_bytes(B, T, H, dk, dv, chunk, dtype)


def eda_fwd(q, k, v, e, beta=None, S0=None, *, o=None, S_final=None, return_final=True, chunk=64, workspace=None,
            stream=None):
    """EDA forward (the C eda_fwd): erase along e, then the Delta write along k with
    strength beta (None = 1), o_t read after both.  q, k, e [B,T,H,dk]; v [B,T,H,dv];
    beta [B,T,H] or None; S0 [B,H,dv,dk] fp32 or None.  bf16 at dk = dv = 128 runs on the
    tensor cores and needs eda_workspace_bytes() of workspace (allocated here when None).
    Returns (o, S_final)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    for t, name, shape in ((q, "q", (B, T, H, dk)), (k, "k", (B, T, H, dk)), (e, "e", (B, T, H, dk)),
                           (v, "v", (B, T, H, dv))):
        _need(t, name, dt, shape)
    _need(beta, "beta", dt, (B, T, H), optional=True)
    _need(S0, "S0", torch.float32, (B, H, dv, dk), optional=True)
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=dt, device=q.device)
    _need(o, "o", dt, (B, T, H, dv))
    if S_final is None and return_final:
        S_final = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    _need(S_final, "S_final", torch.float32, (B, H, dv, dk), optional=True)
    code = _dtype_code(q)
    workspace, wsb = _workspace(eda_workspace_bytes(B, T, H, dk, dv, chunk, code), workspace, q.device)
    _same_device(q.device, k, v, e, beta, S0, o, S_final, workspace)
    st = _call(q.device, load_library().eda_fwd, _ptr(q), _ptr(k), _ptr(v), _ptr(e), _ptr(beta), _ptr(S0),
               _ptr(o), _ptr(S_final), B, T, H, dk, dv, chunk, code, _ptr(workspace), wsb,
               _stream(stream, q.device))
    _check(st, "eda_fwd")
    return o, S_final


def qdelta_fwd_static_scratch(q, k, v, alpha, beta, lam, S0=None, *, o=None, S_final=None, return_final=True,
                              chunk=64, stream=None):
    """qdelta_fwd without a workspace argument: for callers that cannot allocate
    device memory at call time, any scratch comes from a fixed 24 MiB array inside
    the library (sizes needing more raise QDError with QD_ERR_WORKSPACE).  Calls
    whose work overlaps on the GPU share that array and race."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    _need(q, "q", dt, (B, T, H, dk))
    _need(k, "k", dt, (B, T, H, dk))
    _need(v, "v", dt, (B, T, H, dv))
    _need(beta, "beta", dt, (B, T, H))
    _need(alpha, "alpha", dt, (B, T, H), optional=True)
    _need(lam, "lam", dt, (B, T, H), optional=True)
    _need(S0, "S0", torch.float32, (B, H, dv, dk), optional=True)
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=dt, device=q.device)
    _need(o, "o", dt, (B, T, H, dv))
    if S_final is None and return_final:
        S_final = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    _need(S_final, "S_final", torch.float32, (B, H, dv, dk), optional=True)
    _same_device(q.device, k, v, alpha, beta, lam, S0, o, S_final)
    st = _call(q.device, load_library().qdelta_fwd_static_scratch, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
               _ptr(beta), _ptr(lam), _ptr(S0), _ptr(o), _ptr(S_final), B, T, H, dk, dv, chunk, _dtype_code(q),
               _stream(stream, q.device))
    _check(st, "qdelta_fwd_static_scratch")
    return o, S_final


def qed_fwd(q, k, v, g, b, w, lam_h, S0=None, *, o=None, S_final=None, return_final=True, chunk=64,
            workspace=None, stream=None, variant="full", z=None):
    """Chunked QED forward.  q, k, g, b [B,T,H,dk]; v, w [B,T,H,dv]; lam_h [H] fp32;
    S0 [B,H,dv,dk] fp32 (QED's K x V state transposed) or None.  variant: the ablation
    arm (full, nogate, nogate_noproj, rand; rand needs z [H,dk] fp32).  Returns (o, S_final)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    for name, t, shp in (("q", q, (B, T, H, dk)), ("k", k, (B, T, H, dk)), ("v", v, (B, T, H, dv)),
                         ("g", g, (B, T, H, dk)), ("b", b, (B, T, H, dk)), ("w", w, (B, T, H, dv))):
        _need(t, name, dt, shp)
    _need(lam_h, "lam_h", torch.float32, (H,))
    _need(S0, "S0", torch.float32, (B, H, dv, dk), optional=True)
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=dt, device=q.device)
    _need(o, "o", dt, (B, T, H, dv))
    if S_final is None and return_final:
        S_final = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    _need(S_final, "S_final", torch.float32, (B, H, dv, dk), optional=True)
    vid = QED_VARIANTS[variant]
    _need(z, "z", torch.float32, (H, dk), optional=vid != QED_VARIANTS["rand"])
    code = _dtype_code(q)
    workspace, wsb = _workspace(qed_workspace_bytes(B, T, H, dk, dv, chunk, code), workspace, q.device)
    _same_device(q.device, k, v, g, b, w, lam_h, S0, o, S_final, z, workspace)
    st = _call(q.device, load_library().qed_fwd_variant, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(w),
               _ptr(lam_h), _ptr(S0), _ptr(o), _ptr(S_final), B, T, H, dk, dv, chunk, code, vid, _ptr(z),
               _ptr(workspace), wsb, _stream(stream, q.device))
    _check(st, "qed_fwd_variant")
    return o, S_final


def qed_step(S, q, k, v, g, b, w, lam_h, *, o=None, stream=None, variant="full", z=None):
    """One QED decode step, S [N,H,dv,dk] fp32 (QED's state transposed) updated in place;
    q, k, g, b [N,H,dk]; v, w [N,H,dv]; lam_h [H] fp32; variant / z as in qed_fwd.
    Returns o [N,H,dv]."""
    N, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    _need(S, "S", torch.float32, (N, H, dv, dk))
    for name, t, shp in (("q", q, (N, H, dk)), ("k", k, (N, H, dk)), ("g", g, (N, H, dk)), ("b", b, (N, H, dk)),
                         ("v", v, (N, H, dv)), ("w", w, (N, H, dv))):
        _need(t, name, dt, shp)
    _need(lam_h, "lam_h", torch.float32, (H,))
    vid = QED_VARIANTS[variant]
    _need(z, "z", torch.float32, (H, dk), optional=vid != QED_VARIANTS["rand"])
    if o is None:
        o = torch.empty((N, H, dv), dtype=dt, device=q.device)
    _need(o, "o", dt, (N, H, dv))
    _same_device(q.device, S, k, v, g, b, w, lam_h, o, z)
    st = _call(q.device, load_library().qed_step, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(w),
               _ptr(lam_h), _ptr(o), N, H, dk, dv, _dtype_code(q), vid, _ptr(z), _stream(stream, q.device))
    _check(st, "qed_step")
    return o


def qdelta_step(S, q, k, v, alpha, beta, lam, *, o=None, stream=None, prologue=False):
    """One decode step, S [N,H,dv,dk] fp32 updated in place; tokens [N,H,d]; gates [N,H]
    (alpha None = 1, lam None = 0).  Returns o [N,H,dv].  prologue=True as in qdelta_fwd."""
    N, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    _need(S, "S", torch.float32, (N, H, dv, dk))
    _need(q, "q", dt, (N, H, dk))
    _need(k, "k", dt, (N, H, dk))
    _need(v, "v", dt, (N, H, dv))
    _need(beta, "beta", dt, (N, H))
    _need(alpha, "alpha", dt, (N, H), optional=True)
    _need(lam, "lam", dt, (N, H), optional=True)
    if o is None:
        o = torch.empty((N, H, dv), dtype=dt, device=q.device)
    _need(o, "o", dt, (N, H, dv))
    _same_device(q.device, S, k, v, alpha, beta, lam, o)
    fn = load_library().qdelta_step_prologue if prologue else load_library().qdelta_step
    st = _call(q.device, fn, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(lam), _ptr(o), N,
               H, dk, dv, _dtype_code(q), _stream(stream, q.device))
    _check(st, "qdelta_step_prologue" if prologue else "qdelta_step")
    return o


def qd_device_status(stream=None) -> int:
    """Synchronises the stream and returns the library's device status code."""
    dev = torch.cuda.current_device()
    return load_library().qd_device_status(_stream(stream, dev))

"""Oracle: plain fp64 CPU reference of the Q-Delta / QED / EDA forwards, the
Q-Delta backward and the decode steps.

TEST INFRASTRUCTURE.  Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s
CPU-baseline / reference leg may import this package.  It shares no code with
the CUDA path and the CUDA path never calls it.

The arithmetic lives in `qdelta_oracle.c` (sequential recurrences in the pages'
step order; citations in its header).  This module only marshals numpy arrays to
fp64 and calls it.  `build()` compiles the C file with gcc (no CUDA involved).

Array layouts (all numpy, any float dtype; converted to fp64):
  q, k [B,T,H,dk]; v [B,T,H,dv]; Q-Delta gates [B,T,H]; QED g, b [B,T,H,dk],
  w [B,T,H,dv], lam_h [H]; states [B,H,dv,dk] (QED: its K x V state transposed).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qdelta_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile qdelta_oracle.c into liboracle.so (gcc, -O2, portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-shared",
                               "-fPIC", "-o", tmp, _SRC, "-lpthread", "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_qdelta_fwd.argtypes = [I] * 5 + [P] * 9 + [I]
        lib.oracle_qed_fwd.argtypes = [I] * 5 + [P] * 10 + [I]
        lib.oracle_qdelta_step.argtypes = [I] * 4 + [P] * 8 + [I]
        lib.oracle_qed_fwd_variant.argtypes = [I] * 5 + [P] * 7 + [I] + [P] * 4 + [I]
        lib.oracle_qed_step.argtypes = [I] * 4 + [P] * 8 + [I, P, P, I]
        lib.oracle_qdelta_fwd_prologue.argtypes = [I] * 5 + [P] * 9 + [I]
        lib.oracle_qdelta_bwd.argtypes = [I] * 5 + [P] * 16 + [I]
        lib.oracle_eda_fwd.argtypes = [I] * 5 + [P] * 8 + [I]
        lib.oracle_qdelta_bwd_prologue.argtypes = [I] * 5 + [P] * 16 + [I]
        lib.oracle_qdelta_bwd_prologue.restype = I
        for f in (lib.oracle_qdelta_fwd, lib.oracle_qed_fwd, lib.oracle_qdelta_step, lib.oracle_qed_fwd_variant,
                  lib.oracle_qed_step, lib.oracle_qdelta_fwd_prologue, lib.oracle_qdelta_bwd, lib.oracle_eda_fwd):
            f.restype = I
        _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def qdelta_fwd(q, k, v, alpha, beta, lam, S0=None, nthreads: int = 0):
    """Sequential Q-Delta forward.  alpha None = 1, lam None = 0, S0 None = 0.
    Returns (o [B,T,H,dv], S_final [B,H,dv,dk]) in fp64."""
    q, k, v, alpha, beta, lam, S0 = map(_f64, (q, k, v, alpha, beta, lam, S0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    S = np.zeros((B, H, dv, dk))
    rc = _load().oracle_qdelta_fwd(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                   _ptr(beta), _ptr(lam), _ptr(S0), _ptr(o), _ptr(S), nthreads)
    if rc:
        raise MemoryError("oracle_qdelta_fwd failed")
    return o, S


def qdelta_bwd(q, k, v, alpha, beta, lam, S0, dO, dS_final=None, nthreads: int = 0):
    """Backward of qdelta_fwd: gradients of sum(dO * o) + sum(dS_final * S_final)
    (dS_final None = 0).  Returns a dict dq, dk, dv, dalpha (None when alpha is None),
    dbeta, dlam (None when lam is None), dS0, all fp64 in the inputs' shapes."""
    q, k, v, alpha, beta, lam, S0, dO, dS_final = map(_f64, (q, k, v, alpha, beta, lam, S0, dO, dS_final))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    g = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
         "dalpha": None if alpha is None else np.zeros((B, T, H)), "dbeta": np.zeros((B, T, H)),
         "dlam": None if lam is None else np.zeros((B, T, H)), "dS0": np.zeros((B, H, dv, dk))}
    rc = _load().oracle_qdelta_bwd(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(lam),
                                   _ptr(S0), _ptr(dO), _ptr(dS_final), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                                   _ptr(g["dalpha"]), _ptr(g["dbeta"]), _ptr(g["dlam"]), _ptr(g["dS0"]), nthreads)
    if rc:
        raise MemoryError("oracle_qdelta_bwd failed")
    return g


def qdelta_bwd_prologue(q_raw, k_raw, v, a_logit, b_logit, l_logit, S0, dO, dS_final=None, nthreads: int = 0):
    """Backward of qdelta_fwd_prologue: gradients with respect to the projections and
    gate logits (dq, dk are of q_raw, k_raw; dalpha, dbeta, dlam of the logits)."""
    args = map(_f64, (q_raw, k_raw, v, a_logit, b_logit, l_logit, S0, dO, dS_final))
    q_raw, k_raw, v, a_logit, b_logit, l_logit, S0, dO, dS_final = args
    B, T, H, dk = q_raw.shape
    dv = v.shape[-1]
    g = {"dq": np.zeros_like(q_raw), "dk": np.zeros_like(k_raw), "dv": np.zeros_like(v),
         "dalpha": None if a_logit is None else np.zeros((B, T, H)), "dbeta": np.zeros((B, T, H)),
         "dlam": None if l_logit is None else np.zeros((B, T, H)), "dS0": np.zeros((B, H, dv, dk))}
    rc = _load().oracle_qdelta_bwd_prologue(B, T, H, dk, dv, _ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(a_logit),
                                            _ptr(b_logit), _ptr(l_logit), _ptr(S0), _ptr(dO), _ptr(dS_final),
                                            _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dalpha"]),
                                            _ptr(g["dbeta"]), _ptr(g["dlam"]), _ptr(g["dS0"]), nthreads)
    if rc:
        raise MemoryError("oracle_qdelta_bwd_prologue failed")
    return g


def eda_fwd(q, k, v, e, beta=None, S0=None, nthreads: int = 0):
    """Sequential EDA forward (erase along e, then the Delta write along k; beta None
    = the page's unit step).  Returns (o [B,T,H,dv], S_final [B,H,dv,dk] = M^T)."""
    q, k, v, e, beta, S0 = map(_f64, (q, k, v, e, beta, S0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    S = np.zeros((B, H, dv, dk))
    rc = _load().oracle_eda_fwd(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(e), _ptr(beta), _ptr(S0),
                                _ptr(o), _ptr(S), nthreads)
    if rc:
        raise MemoryError("oracle_eda_fwd failed")
    return o, S


def qed_fwd(q, k, v, g, b, w, lam_h, S0=None, nthreads: int = 0):
    """Sequential QED forward (GDN-2 with the query-derived erase direction).
    Returns (o [B,T,H,dv], S_final [B,H,dv,dk] = QED's K x V state transposed)."""
    q, k, v, g, b, w, lam_h, S0 = map(_f64, (q, k, v, g, b, w, lam_h, S0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    S = np.zeros((B, H, dv, dk))
    rc = _load().oracle_qed_fwd(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b),
                                _ptr(w), _ptr(lam_h), _ptr(S0), _ptr(o), _ptr(S), nthreads)
    if rc:
        raise MemoryError("oracle_qed_fwd failed")
    return o, S


def qdelta_fwd_prologue(q_raw, k_raw, v, a_logit, b_logit, l_logit, S0=None, nthreads: int = 0):
    """Q-Delta forward from the projections: q, k = SiLU(x)/|SiLU(x)|, beta, lambda =
    sigmoid(logit), alpha = exp(-softplus(logit)) (None logits: alpha 1, lambda 0)."""
    q_raw, k_raw, v, a_logit, b_logit, l_logit, S0 = map(_f64, (q_raw, k_raw, v, a_logit, b_logit, l_logit, S0))
    B, T, H, dk = q_raw.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    S = np.zeros((B, H, dv, dk))
    rc = _load().oracle_qdelta_fwd_prologue(B, T, H, dk, dv, _ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(a_logit),
                                            _ptr(b_logit), _ptr(l_logit), _ptr(S0), _ptr(o), _ptr(S), nthreads)
    if rc:
        raise MemoryError("oracle_qdelta_fwd_prologue failed")
    return o, S


QED_VARIANTS = {"full": 0, "nogate": 1, "nogate_noproj": 2, "rand": 3}


def qed_fwd_variant(q, k, v, g, b, w, lam_h, variant="full", z=None, S0=None, nthreads: int = 0):
    """QED forward for one ablation arm ("The Query Knows What to Forget", Table 1):
    full, nogate, nogate_noproj or rand (z [H,dk] the per-head fixed vector)."""
    vid = QED_VARIANTS[variant]
    q, k, v, g, b, w, lam_h, z, S0 = map(_f64, (q, k, v, g, b, w, lam_h, z, S0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    S = np.zeros((B, H, dv, dk))
    rc = _load().oracle_qed_fwd_variant(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b),
                                        _ptr(w), _ptr(lam_h), vid, _ptr(z), _ptr(S0), _ptr(o), _ptr(S), nthreads)
    if rc:
        raise ValueError(f"oracle_qed_fwd_variant failed ({rc})")
    return o, S


def qed_step(S, q, k, v, g, b, w, lam_h, variant="full", z=None, nthreads: int = 0):
    """One QED decode step.  S [N,H,dv,dk] fp64 numpy array (QED's state transposed),
    updated IN PLACE; q, k, g, b [N,H,dk]; v, w [N,H,dv]; lam_h [H].  Returns o [N,H,dv]."""
    if not (isinstance(S, np.ndarray) and S.dtype == np.float64 and S.flags.c_contiguous):
        raise TypeError("S must be a C-contiguous float64 numpy array (updated in place)")
    vid = QED_VARIANTS[variant]
    q, k, v, g, b, w, lam_h, z = map(_f64, (q, k, v, g, b, w, lam_h, z))
    N, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((N, H, dv))
    rc = _load().oracle_qed_step(N, H, dk, dv, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b),
                                 _ptr(w), _ptr(lam_h), vid, _ptr(z), _ptr(o), nthreads)
    if rc:
        raise ValueError(f"oracle_qed_step failed ({rc})")
    return o


def qdelta_step(S, q, k, v, alpha, beta, lam, nthreads: int = 0):
    """One decode step.  S [N,H,dv,dk] fp64 numpy array, updated IN PLACE;
    tokens [N,H,d], gates [N,H].  Returns o [N,H,dv]."""
    if not (isinstance(S, np.ndarray) and S.dtype == np.float64 and S.flags.c_contiguous):
        raise TypeError("S must be a C-contiguous float64 numpy array (updated in place)")
    q, k, v, alpha, beta, lam = map(_f64, (q, k, v, alpha, beta, lam))
    N, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((N, H, dv))
    rc = _load().oracle_qdelta_step(N, H, dk, dv, _ptr(S), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(alpha), _ptr(beta), _ptr(lam), _ptr(o), nthreads)
    if rc:
        raise MemoryError("oracle_qdelta_step failed")
    return o

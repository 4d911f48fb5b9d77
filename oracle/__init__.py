"""CPU fp64 oracle for the fused TP-reduce + MoE finalize + residual + RMSNorm.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``tp_reduce_moe_gb300``) never imports, links or calls it, and this package
never imports the product: the two share no code.

The arithmetic lives in ``ar_oracle.c`` (plain C, binary64, OpenMP over token
rows); this module only builds it with gcc and marshals numpy arrays.  The
exact rational brute force that pins it is ``oracle.brute``.

Every function takes bf16 data as ``numpy.uint16`` arrays of raw bf16 bit
patterns, fp32 routing weights as ``numpy.float32`` and int32 perm as
``numpy.int32``; results come back as ``numpy.float64`` (unrounded).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "ar_oracle.c")
_LIB = os.path.join(_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``ar_oracle.c`` into ``liboracle.so`` beside it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.oracle_ar_finalize_rmsnorm.restype = ctypes.c_int
    lib.oracle_ar_finalize_rmsnorm.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
        P, P, P, P, P, P, ctypes.c_double, ctypes.c_double, ctypes.c_int,
        P, P, P]
    lib.oracle_ar_finalize_rmsnorm_gated.restype = ctypes.c_int
    lib.oracle_ar_finalize_rmsnorm_gated.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
        P, P, P, P, P, P, P, ctypes.c_double, ctypes.c_double, ctypes.c_int,
        P, P, P]
    lib.oracle_ar_mhc_post.restype = ctypes.c_int
    lib.oracle_ar_mhc_post.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                       P, P, P, P, P]
    lib.oracle_round_bf16.restype = ctypes.c_double
    lib.oracle_round_bf16.argtypes = [ctypes.c_double]
    lib.oracle_round_bf16_array.restype = None
    lib.oracle_round_bf16_array.argtypes = [P, P, ctypes.c_int64]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


@contextlib.contextmanager
def _swap_library(path: str):
    """Run the wrappers against another build of the oracle source (used only
    by the test that plants mistakes in a copy of ``ar_oracle.c``)."""
    global _lib
    old = _load()
    with _lock:
        _lib = _bind(path)
    try:
        yield
    finally:
        with _lock:
            _lib = old


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _ptr_table(arrs):
    tab = (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])
    return tab


def _u16(a, shape=None) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 data must be uint16 bit patterns, got {a.dtype}")
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"shape {a.shape} != {tuple(shape)}")
    return a


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def round_bf16(x) -> np.ndarray:
    """Round binary64 values to the nearest bfloat16 value (ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_round_bf16_array(_ptr(x), _ptr(y), x.size)
    return y


def ar_finalize_rmsnorm_ref(E, perm, w, S, residual, gamma, weight_bias, eps,
                            h_bf16_before_norm=False, want_abs=False, shared_gate=None):
    """fp64 oracle of the fused boundary op for all T rows.

    E: list of R arrays [rows_e, H] (bf16 bits), or None/[] when K == 0.
    perm: int32 [T, K]; w: float32 [T, K]; S: list of R arrays [T, H] or None.
    residual: [T, H]; gamma: [H].  shared_gate: optional float32 [T] gate
    logits (the shared term of token t is scaled by sigmoid(shared_gate[t])).
    Returns dict with float64 ``h`` (the unrounded residual_out), ``out`` and,
    with ``want_abs``, ``abs`` (sum of |terms| per element).
    """
    residual = _u16(residual)
    T, H = residual.shape
    gamma = _u16(gamma, (H,))
    if E:
        E = [_u16(e) for e in E]
        R = len(E)
        rows_e = E[0].shape[0]
        for e in E:
            if e.shape != (rows_e, H):
                raise ValueError("all E_r must have the same [rows_e, H] shape")
        perm = np.ascontiguousarray(perm, dtype=np.int32)
        K = perm.shape[1] if perm.ndim == 2 else 0
        if perm.shape != (T, K):
            raise ValueError(f"perm shape {perm.shape} != {(T, K)}")
        w = np.ascontiguousarray(w, dtype=np.float32)
        if w.shape != (T, K):
            raise ValueError(f"w shape {w.shape} != {(T, K)}")
    else:
        R, K, rows_e = (len(S) if S else 0), 0, 0
        perm = np.zeros((1,), np.int32)
        w = np.zeros((1,), np.float32)
    if S:
        S = [_u16(s, (T, H)) for s in S]
        if R and len(S) != R:
            raise ValueError("S must have R entries")
        R = len(S)
    h = np.empty((T, H), np.float64)
    out = np.empty((T, H), np.float64)
    ab = np.empty((T, H), np.float64) if want_abs else None
    e_tab = _ptr_table(E) if E else None
    s_tab = _ptr_table(S) if S else None
    common_head = (R, K, H, T, rows_e,
                   ctypes.cast(e_tab, ctypes.c_void_p) if e_tab is not None else None,
                   _ptr(perm), _ptr(w),
                   ctypes.cast(s_tab, ctypes.c_void_p) if s_tab is not None else None)
    common_tail = (_ptr(residual), _ptr(gamma), float(weight_bias), float(eps),
                   1 if h_bf16_before_norm else 0,
                   _ptr(h), _ptr(out), _ptr(ab) if ab is not None else None)
    if shared_gate is not None:
        gate = np.ascontiguousarray(shared_gate, dtype=np.float32)
        if gate.shape != (T,):
            raise ValueError(f"shared_gate shape {gate.shape} != {(T,)}")
        rc = _load().oracle_ar_finalize_rmsnorm_gated(*common_head, _ptr(gate), *common_tail)
    else:
        rc = _load().oracle_ar_finalize_rmsnorm(*common_head, *common_tail)
    if rc == -2:
        raise IndexError("perm value outside [0, rows_e)")
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")
    res = {"h": h, "out": out}
    if want_abs:
        res["abs"] = ab
    return res


def ar_rmsnorm_ref(partials, residual, gamma, weight_bias, eps,
                   h_bf16_before_norm=False, want_abs=False):
    """fp64 oracle of the K = 0 case: sum of R partials + residual, RMSNorm."""
    return ar_finalize_rmsnorm_ref(None, None, None, partials, residual, gamma,
                                   weight_bias, eps, h_bf16_before_norm, want_abs)


def ar_mhc_post_ref(partials, x, post, comb):
    """fp64 oracle of the all-reduce + mHC residual write-back (hc_post).

    partials: list of R arrays [T, H] (bf16 bits); x: [T, hc, H] (bf16 bits,
    the incoming residual streams); post: float32 [T, hc]; comb: float32
    [T, hc, hc].  Returns float64 out [T, hc, H] (unrounded):
    out[t,i,j] = post[t,i] * sum_r P_r[t,j] + sum_k comb[t,i,k] * x[t,k,j].
    PARITY UNPINNED: the pages do not define hc_post (see ar_oracle.c).
    """
    x = _u16(x)
    T, hc, H = x.shape
    partials = [_u16(p, (T, H)) for p in partials]
    post = np.ascontiguousarray(post, dtype=np.float32)
    comb = np.ascontiguousarray(comb, dtype=np.float32)
    if post.shape != (T, hc) or comb.shape != (T, hc, hc):
        raise ValueError(f"post {post.shape} / comb {comb.shape} do not match T={T}, hc={hc}")
    out = np.empty((T, hc, H), np.float64)
    tab = _ptr_table(partials)
    rc = _load().oracle_ar_mhc_post(len(partials), H, hc, T, ctypes.cast(tab, ctypes.c_void_p),
                                    _ptr(x), _ptr(post), _ptr(comb), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")
    return out

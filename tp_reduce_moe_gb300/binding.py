"""Thin ctypes binding of libarfuse (include/arfuse.h): argument marshalling only.

Every step of the operator runs in the CUDA library; this module turns torch
tensors into device pointers and sizes, checks that their shapes agree with
the sizes passed (the C ABI sees only pointers), and raises on any status
other than AR_OK.  There is no CPU path: if the library is missing, loading it
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
import weakref

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libarfuse.so")

AR_OK = 0
AR_ERR_INVALID_ARG = 1
AR_ERR_ALIGNMENT = 2
AR_ERR_UNSUPPORTED = 3
AR_ERR_CAPACITY = 4
AR_ERR_CUDA = 5
AR_ERR_DEVICE_CHECK = 6
AR_VALIDATED = 7

AR_WS_DRY_RUN = 0x1
AR_WS_NORM_BF16_H = 0x2
AR_WS_PDL = 0x4
AR_DEVERR_PERM_RANGE = 0x1
AR_DEVERR_TIMEOUT = 0x2
AR_REGIME_AUTO = 0
AR_REGIME_CLUSTER = 1
AR_REGIME_STREAM = 2
AR_REGIME_ONESHOT = 3
AR_REGIME_SPLIT = 4

AR_MAX_RANKS = 16
AR_MAX_TOP_K = 16
AR_MAX_HIDDEN = 16384

_lock = threading.Lock()
_lib = None


class ArfuseError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {ar_status_string(status)} (status {status})")


def load_library(path: str | None = None):
    """Load libarfuse.so (built by ``tp_reduce_moe_gb300.build``).  Raises if
    it is missing: there is no fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libarfuse.so not found at {p}; build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        P, I, I64, F, U = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                           ctypes.c_uint)
        lib.ar_workspace_create.restype = I
        lib.ar_workspace_create.argtypes = [I, I, I, I, I64, F, U, ctypes.POINTER(P)]
        lib.ar_workspace_destroy.restype = I
        lib.ar_workspace_destroy.argtypes = [P]
        lib.ar_finalize_rmsnorm.restype = I
        lib.ar_finalize_rmsnorm.argtypes = [P, P, I64, P, P, P, P, P, F, F, I64, I, I, I,
                                            P, P, I, P]
        lib.ar_finalize_rmsnorm_gated.restype = I
        lib.ar_finalize_rmsnorm_gated.argtypes = [P, P, I64, P, P, P, P, P, P, F, F, I64, I, I, I,
                                                  P, P, I, P]
        lib.ar_rmsnorm.restype = I
        lib.ar_rmsnorm.argtypes = [P, P, I, P, P, F, F, I64, I, P, P, I, P]
        lib.ar_workspace_device_error.restype = I
        lib.ar_workspace_device_error.argtypes = [P, ctypes.POINTER(I)]
        lib.ar_workspace_set_regime.restype = I
        lib.ar_workspace_set_regime.argtypes = [P, I]
        lib.ar_workspace_set_stage_bytes.restype = I
        lib.ar_workspace_set_stage_bytes.argtypes = [P, I]
        lib.ar_workspace_set_split_rows.restype = I
        lib.ar_workspace_set_split_rows.argtypes = [P, I]
        lib.ar_workspace_inject_wait_timeout.restype = I
        lib.ar_workspace_inject_wait_timeout.argtypes = [P, I64]
        lib.ar_workspace_set_producer_warps.restype = I
        lib.ar_workspace_set_producer_warps.argtypes = [P, I]
        lib.ar_workspace_set_split_column_groups.restype = I
        lib.ar_workspace_set_split_column_groups.argtypes = [P, I]
        lib.ar_mhc_post.restype = I
        lib.ar_mhc_post.argtypes = [P, P, I, P, P, P, I64, I, I, P, P]
        lib.ar_workspace_set_regime_table.restype = I
        lib.ar_workspace_set_regime_table.argtypes = [P, P, I]
        lib.ar_workspace_get_regime_table.restype = I
        lib.ar_workspace_get_regime_table.argtypes = [P, P, I, ctypes.POINTER(I)]
        lib.ar_workspace_set_cluster_size.restype = I
        lib.ar_workspace_set_cluster_size.argtypes = [P, I]
        lib.ar_workspace_last_regime.restype = I
        lib.ar_workspace_last_regime.argtypes = [P, ctypes.POINTER(I)]
        lib.ar_workspace_last_grid.restype = I
        lib.ar_workspace_last_grid.argtypes = [P]
        lib.ar_workspace_last_plan.restype = I
        lib.ar_workspace_last_plan.argtypes = [P, P]
        lib.ar_status_string.restype = ctypes.c_char_p
        lib.ar_status_string.argtypes = [I]
        _lib = lib
        return lib


def ar_status_string(status: int) -> str:
    """Text of an ar_status code (\"unknown status\" for other values)."""
    return load_library().ar_status_string(int(status)).decode()


def _check(status: int, where: str, ok=(AR_OK,)):
    if status not in ok:
        raise ArfuseError(status, where)
    return status


class Workspace:
    """Owner of one ``ar_workspace*`` (fixed R, K, H, eps, max_tokens)."""

    def __init__(self, handle: int, R: int, K: int, H: int, max_tokens: int, eps: float,
                 device: int, dry_run: bool):
        self.handle = handle
        self.R, self.K, self.H = R, K, H
        self.max_tokens, self.eps, self.device, self.dry_run = max_tokens, eps, device, dry_run
        self._fin = weakref.finalize(self, _destroy_handle, handle)

    def destroy(self):
        self._fin()

    @property
    def alive(self) -> bool:
        return self._fin.alive


def _destroy_handle(handle):
    if handle:
        load_library().ar_workspace_destroy(ctypes.c_void_p(handle))


def ar_workspace_create(ranks: int, top_k: int, hidden: int, max_tokens: int, eps: float,
                        device: int | None = None, flags: int = 0) -> Workspace:
    """Workspace for one model shape (R rank partials, top_k, hidden, eps),
    shared by its layers; `device` defaults to the current CUDA device,
    `flags` takes AR_WS_* (AR_WS_DRY_RUN: no GPU state, calls only validate).
    Installs the built-in regime table when the library has one for the
    shape."""
    lib = load_library()
    dry = bool(flags & AR_WS_DRY_RUN)
    if device is None:
        device = torch.cuda.current_device() if not dry else 0
    h = ctypes.c_void_p()
    _check(lib.ar_workspace_create(int(device), int(ranks), int(top_k), int(hidden),
                                   int(max_tokens), float(eps), int(flags), ctypes.byref(h)),
           "ar_workspace_create")
    return Workspace(h.value, ranks, top_k, hidden, max_tokens, eps, device, dry)


def ar_workspace_destroy(ws: Workspace) -> None:
    """Free the workspace (no call on it may still be running)."""
    ws.destroy()


def ar_workspace_set_regime(ws: Workspace, regime: int) -> None:
    """Force AR_REGIME_CLUSTER / _STREAM / _ONESHOT / _SPLIT for later calls
    (a call it cannot plan raises AR_ERR_UNSUPPORTED); AR_REGIME_AUTO restores
    the regime table and the heuristic."""
    _check(load_library().ar_workspace_set_regime(ctypes.c_void_p(ws.handle), int(regime)),
           "ar_workspace_set_regime")


def ar_workspace_set_cluster_size(ws: Workspace, ctas_per_row: int) -> None:
    """Force the CTAs per row (2..16) of the cluster, split and one-shot
    regimes (one-shot: a power of two); 0 = automatic."""
    _check(load_library().ar_workspace_set_cluster_size(ctypes.c_void_p(ws.handle),
                                                        int(ctas_per_row)),
           "ar_workspace_set_cluster_size")


def ar_workspace_set_stage_bytes(ws: Workspace, nbytes: int) -> None:
    """Target ring-slot size of the streaming kernels (tuning); 0 = automatic."""
    _check(load_library().ar_workspace_set_stage_bytes(ctypes.c_void_p(ws.handle), int(nbytes)),
           "ar_workspace_set_stage_bytes")


class RegimeRule(ctypes.Structure):
    """One rule of a regime table (``ar_regime_rule``)."""
    _fields_ = [("max_tokens", ctypes.c_int64), ("regime", ctypes.c_int32),
                ("ctas_per_row", ctypes.c_int32), ("stage_bytes", ctypes.c_int32),
                ("producer_warps", ctypes.c_int32)]


AR_MAX_REGIME_RULES = 32


def ar_workspace_set_regime_table(ws: Workspace, rules) -> None:
    """Replace the workspace's regime table: ``[(max_tokens, regime, ctas_per_row
    [, stage_bytes, producer_warps]), ...]`` with strictly ascending max_tokens
    (empty: heuristic only); omitted fields are 0 (automatic)."""
    rules = [tuple(r) + (0,) * (5 - len(r)) for r in rules]
    arr = (RegimeRule * max(1, len(rules)))(*[RegimeRule(*[int(x) for x in r]) for r in rules])
    _check(load_library().ar_workspace_set_regime_table(ctypes.c_void_p(ws.handle),
                                                        ctypes.cast(arr, ctypes.c_void_p), len(rules)),
           "ar_workspace_set_regime_table")


def ar_workspace_get_regime_table(ws: Workspace):
    """The workspace's regime table as ``[(max_tokens, regime, ctas_per_row,
    stage_bytes, producer_warps), ...]``."""
    arr = (RegimeRule * AR_MAX_REGIME_RULES)()
    n = ctypes.c_int(0)
    _check(load_library().ar_workspace_get_regime_table(ctypes.c_void_p(ws.handle),
                                                        ctypes.cast(arr, ctypes.c_void_p),
                                                        AR_MAX_REGIME_RULES, ctypes.byref(n)),
           "ar_workspace_get_regime_table")
    return [(int(arr[i].max_tokens), int(arr[i].regime), int(arr[i].ctas_per_row),
             int(arr[i].stage_bytes), int(arr[i].producer_warps))
            for i in range(min(n.value, AR_MAX_REGIME_RULES))]


AR_MAX_SPLIT_PARTS = 8


def ar_workspace_set_split_rows(ws: Workspace, max_parts: int) -> None:
    """Cap how many CTAs share each row of whole-row streaming's last, partial
    wave (0 or 1: never split; default AR_MAX_SPLIT_PARTS)."""
    _check(load_library().ar_workspace_set_split_rows(ctypes.c_void_p(ws.handle), int(max_parts)),
           "ar_workspace_set_split_rows")


def ar_workspace_set_split_column_groups(ws: Workspace, groups: int) -> None:
    """Column groups per row of the split kernel (1..8, a divisor of the
    cluster size; tuning); 0 = automatic."""
    _check(load_library().ar_workspace_set_split_column_groups(ctypes.c_void_p(ws.handle), int(groups)),
           "ar_workspace_set_split_column_groups")


def ar_workspace_set_producer_warps(ws: Workspace, warps: int) -> None:
    """Cap the streaming kernels' producer warps (1..4; tuning); 0 = automatic."""
    _check(load_library().ar_workspace_set_producer_warps(ctypes.c_void_p(ws.handle), int(warps)),
           "ar_workspace_set_producer_warps")


def ar_workspace_inject_wait_timeout(ws: Workspace, limit_ns: int) -> None:
    """Failure injection for tests (0 = off): whole-row streaming calls make
    their consumers wait on a barrier nothing arrives on, for limit_ns, so the
    call takes the device-side timeout path (AR_DEVERR_TIMEOUT, outputs of
    that call undefined); other regimes decline while it is set."""
    _check(load_library().ar_workspace_inject_wait_timeout(ctypes.c_void_p(ws.handle), int(limit_ns)),
           "ar_workspace_inject_wait_timeout")


def ar_workspace_last_regime(ws: Workspace):
    """(regime, CTAs per row -- or the grid for whole-row streaming) of the
    last launched (dry run: validated) call; (0, 0) before the first."""
    n = ctypes.c_int(0)
    r = load_library().ar_workspace_last_regime(ctypes.c_void_p(ws.handle), ctypes.byref(n))
    return int(r), int(n.value)


def ar_workspace_last_grid(ws: Workspace) -> int:
    """CTAs launched by the last call (0 before the first)."""
    return int(load_library().ar_workspace_last_grid(ctypes.c_void_p(ws.handle)))


class PlanInfo(ctypes.Structure):
    """The launch plan of a call (``ar_plan_info``)."""
    _fields_ = [(name, ctypes.c_int32) for name in (
        "regime", "ctas_per_row", "grid", "block", "smem_bytes", "column_groups", "copy_rounds",
        "ring_slots", "ring_slot_bytes", "producer_warps", "loads_per_thread")]


def ar_workspace_last_plan(ws: Workspace) -> dict:
    """The last launched (dry run: validated) call's launch plan as a dict of
    the ``ar_plan_info`` fields (regime, CTAs per row, grid, block, shared
    memory, split column groups and copy rounds, ring slots and slot bytes,
    producer warps, one-shot loads per thread); all zero before the first."""
    info = PlanInfo()
    _check(load_library().ar_workspace_last_plan(ctypes.c_void_p(ws.handle), ctypes.byref(info)),
           "ar_workspace_last_plan")
    return {name: int(getattr(info, name)) for name, _ in PlanInfo._fields_}


def ar_workspace_device_error(ws: Workspace) -> int:
    """Synchronise, read and clear the device error word (AR_DEVERR_* bits)."""
    code = ctypes.c_int(0)
    st = load_library().ar_workspace_device_error(ctypes.c_void_p(ws.handle), ctypes.byref(code))
    _check(st, "ar_workspace_device_error", ok=(AR_OK, AR_ERR_DEVICE_CHECK))
    return int(code.value)


# ------------------------------------------------------------------ marshalling
def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _need(t, dtype, shape, name, index=None):
    if isinstance(t, int):       # raw device address: the caller vouches for it
        return
    # one combined test on the common path (a call checks ~20 tensors); the
    # name is formatted only for the error
    if t.dtype is dtype and t.shape == shape and t.is_contiguous():
        return
    if index is not None:
        name = f"{name}[{index}]"
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    raise ValueError(f"{name}: must be contiguous")


def _ptr_array(ts):
    return (ctypes.c_void_p * len(ts))(*[t if isinstance(t, int) else t.data_ptr() for t in ts])


def _stream_handle(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def ar_finalize_rmsnorm(ws: Workspace, expert_out, perm, topk_w, shared_out, residual, gamma,
                        weight_bias: float, eps: float, out=None, residual_out=None,
                        residual_out_fp32: bool = False, stream=None, rows_e: int | None = None,
                        T: int | None = None, shared_gate=None):
    """Fused MoE finalize + shared add + rank sum + residual + RMSNorm.

    expert_out: list of R bf16 [rows_e, H] tensors; perm int32 [T, K]; topk_w
    fp32 [T, K]; shared_out: list of R bf16 [T, H] or None; residual bf16
    [T, H]; gamma bf16 [H].  shared_gate: optional fp32 [T] gate logits (calls
    ar_finalize_rmsnorm_gated: shared partials scaled by sigmoid(gate[t])).
    Returns (out, residual_out); outputs are allocated when not given.
    ``residual_out`` may be ``residual`` (in place, bf16 only).
    """
    R, K, H = ws.R, ws.K, ws.H
    if T is None:
        T = residual.shape[0]
    if K == 0 and not expert_out:
        expert_out = []
    elif len(expert_out) != R:
        raise ValueError(f"expert_out has {len(expert_out)} entries, workspace has R={R}")
    if rows_e is None:
        rows_e = expert_out[0].shape[0] if K > 0 else 0
    for r, e in enumerate(expert_out):
        _need(e, torch.bfloat16, (rows_e, H), "expert_out", r)
    if K > 0:
        _need(perm, torch.int32, (T, K), "perm")
        _need(topk_w, torch.float32, (T, K), "topk_w")
    if shared_out is not None:
        if len(shared_out) != R:
            raise ValueError("shared_out must have R entries")
        for r, s in enumerate(shared_out):
            _need(s, torch.bfloat16, (T, H), "shared_out", r)
    _need(residual, torch.bfloat16, (T, H), "residual")
    _need(gamma, torch.bfloat16, (H,), "gamma")
    if shared_gate is not None:
        _need(shared_gate, torch.float32, (T,), "shared_gate")
    dev = residual.device if not isinstance(residual, int) else None
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if residual_out is None:
        residual_out = torch.empty((T, H), dtype=torch.float32 if residual_out_fp32 else torch.bfloat16,
                                   device=dev)
    _need(out, torch.bfloat16, (T, H), "out")
    _need(residual_out, torch.float32 if residual_out_fp32 else torch.bfloat16, (T, H),
          "residual_out")
    e_arr = _ptr_array(expert_out) if K > 0 else None
    s_arr = _ptr_array(shared_out) if shared_out is not None else None
    head = (ctypes.c_void_p(ws.handle),
            ctypes.addressof(e_arr) if e_arr is not None else None,
            int(rows_e), _ptr(perm) if K > 0 else None, _ptr(topk_w) if K > 0 else None,
            ctypes.addressof(s_arr) if s_arr is not None else None)
    tail = (_ptr(residual), _ptr(gamma), float(weight_bias), float(eps), int(T), int(R), int(K),
            int(H), _ptr(out), _ptr(residual_out), 1 if residual_out_fp32 else 0,
            _stream_handle(stream, dev) if not ws.dry_run else None)
    lib = load_library()
    if shared_gate is not None:
        st = lib.ar_finalize_rmsnorm_gated(*head, _ptr(shared_gate), *tail)
        where = "ar_finalize_rmsnorm_gated"
    else:
        st = lib.ar_finalize_rmsnorm(*head, *tail)
        where = "ar_finalize_rmsnorm"
    _check(st, where, ok=(AR_OK, AR_VALIDATED) if ws.dry_run else (AR_OK,))
    return out, residual_out


def ar_rmsnorm(ws: Workspace, partials, residual, gamma, weight_bias: float, eps: float, out=None,
               residual_out=None, residual_out_fp32: bool = False, stream=None,
               T: int | None = None):
    """Trailing all-reduce + residual RMSNorm (no MoE term): h = sum_r partials[r]
    + residual, out = RMSNorm(h).  Returns (out, residual_out)."""
    R, H = ws.R, ws.H
    if T is None:
        T = residual.shape[0]
    if len(partials) != R:
        raise ValueError(f"partials has {len(partials)} entries, workspace has R={R}")
    for r, s in enumerate(partials):
        _need(s, torch.bfloat16, (T, H), "partials", r)
    _need(residual, torch.bfloat16, (T, H), "residual")
    _need(gamma, torch.bfloat16, (H,), "gamma")
    dev = residual.device if not isinstance(residual, int) else None
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if residual_out is None:
        residual_out = torch.empty((T, H), dtype=torch.float32 if residual_out_fp32 else torch.bfloat16,
                                   device=dev)
    _need(out, torch.bfloat16, (T, H), "out")
    _need(residual_out, torch.float32 if residual_out_fp32 else torch.bfloat16, (T, H),
          "residual_out")
    p_arr = _ptr_array(partials)
    st = load_library().ar_rmsnorm(
        ctypes.c_void_p(ws.handle), ctypes.addressof(p_arr), int(R), _ptr(residual),
        _ptr(gamma), float(weight_bias), float(eps), int(T), int(H), _ptr(out), _ptr(residual_out),
        1 if residual_out_fp32 else 0, _stream_handle(stream, dev) if not ws.dry_run else None)
    _check(st, "ar_rmsnorm", ok=(AR_OK, AR_VALIDATED) if ws.dry_run else (AR_OK,))
    return out, residual_out


AR_MAX_HC_STREAMS = 8


def ar_mhc_post(ws: Workspace, partials, streams, post, comb, out=None, stream=None,
                T: int | None = None, hc: int | None = None):
    """All-reduce + mHC residual write-back: out[t,i] = post[t,i] * sum_r partials[r][t]
    + sum_k comb[t,i,k] * streams[t,k].  partials: R bf16 [T, H]; streams bf16
    [T, hc, H]; post fp32 [T, hc]; comb fp32 [T, hc, hc].  ``out`` may be
    ``streams`` (in place).  Returns out."""
    R, H = ws.R, ws.H
    if len(partials) != R:
        raise ValueError(f"partials has {len(partials)} entries, workspace has R={R}")
    if T is None:
        T = streams.shape[0]
    if hc is None:
        hc = streams.shape[1] if not isinstance(streams, int) else post.shape[1]
    for r, p in enumerate(partials):
        _need(p, torch.bfloat16, (T, H), "partials", r)
    _need(streams, torch.bfloat16, (T, hc, H), "streams")
    _need(post, torch.float32, (T, hc), "post")
    _need(comb, torch.float32, (T, hc, hc), "comb")
    dev = streams.device if not isinstance(streams, int) else None
    if out is None:
        out = torch.empty((T, hc, H), dtype=torch.bfloat16, device=dev)
    _need(out, torch.bfloat16, (T, hc, H), "out")
    arr = _ptr_array(partials)
    st = load_library().ar_mhc_post(ctypes.c_void_p(ws.handle), ctypes.cast(arr, ctypes.c_void_p), int(R),
                                    _ptr(streams), _ptr(post), _ptr(comb), int(T), int(H), int(hc),
                                    _ptr(out), _stream_handle(stream, dev) if not ws.dry_run else None)
    _check(st, "ar_mhc_post", ok=(AR_OK, AR_VALIDATED) if ws.dry_run else (AR_OK,))
    return out

"""Host-side tests of the C ABI (no kernel launch, no GPU needed).

The library must load, export every entry point include/arfuse.h declares,
and reject bad arguments on the host before anything could launch.  Argument
checks run against a dry-run workspace (AR_WS_DRY_RUN), whose calls validate
and then return AR_VALIDATED; fake, suitably aligned addresses stand in for
device pointers and are never dereferenced.
"""
import ctypes
import os
import re
import subprocess

import pytest

import tp_reduce_moe_gb300 as arf
from tp_reduce_moe_gb300 import binding

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(os.path.dirname(HERE), "include", "arfuse.h")


@pytest.fixture(scope="module")
def lib():
    from tp_reduce_moe_gb300 import build
    build.build()
    return arf.load_library()


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"ARFUSE_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"ar_workspace_create", "ar_workspace_destroy", "ar_finalize_rmsnorm", "ar_rmsnorm",
            "ar_workspace_device_error", "ar_status_string"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in arfuse.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("ar_")}
    assert exported == set(declared_functions())


def test_status_strings(lib):
    for s in range(0, 8):
        assert arf.ar_status_string(s)
    assert arf.ar_status_string(99) == "unknown status"


def test_destroy_null_is_ok(lib):
    assert lib.ar_workspace_destroy(None) == arf.AR_OK


def test_null_workspace_is_rejected(lib):
    assert lib.ar_workspace_device_error(None, None) == arf.AR_ERR_INVALID_ARG
    assert lib.ar_workspace_set_regime(None, 0) == arf.AR_ERR_INVALID_ARG
    assert lib.ar_workspace_last_regime(None, None) == 0
    assert lib.ar_rmsnorm(None, None, 2, None, None, 0.0, 1e-6, 1, 8, None, None, 0, None) \
        == arf.AR_ERR_INVALID_ARG


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="needs a machine without a GPU")
def test_create_without_gpu_fails_cleanly(lib):
    h = ctypes.c_void_p()
    st = lib.ar_workspace_create(0, 2, 2, 256, 16, 1e-6, 0, ctypes.byref(h))
    assert st == arf.AR_ERR_CUDA and not h.value


@pytest.mark.parametrize("args,status", [
    ((2, 2, 256, 0, 1e-6, 0), arf.AR_ERR_INVALID_ARG),       # max_tokens
    ((2, 2, 256, 16, -1.0, 0), arf.AR_ERR_INVALID_ARG),      # eps
    ((2, 2, 256, 16, float("nan"), 0), arf.AR_ERR_INVALID_ARG),
    ((2, 2, 260, 16, 1e-6, 0), arf.AR_ERR_ALIGNMENT),        # H % 8
    ((17, 2, 256, 16, 1e-6, 0), arf.AR_ERR_UNSUPPORTED),     # R
    ((0, 2, 256, 16, 1e-6, 0), arf.AR_ERR_UNSUPPORTED),
    ((2, 17, 256, 16, 1e-6, 0), arf.AR_ERR_UNSUPPORTED),     # K
    ((2, 2, 16392, 16, 1e-6, 0), arf.AR_ERR_UNSUPPORTED),    # H
    ((2, 2, 256, 16, 1e-6, 0x8), arf.AR_ERR_INVALID_ARG),    # unknown flag
])
def test_create_rejects(lib, args, status):
    h = ctypes.c_void_p()
    R, K, H, T, eps, flags = args
    st = lib.ar_workspace_create(0, R, K, H, T, eps, flags | arf.AR_WS_DRY_RUN, ctypes.byref(h))
    assert st == status and not h.value


# ------------------------------------------------------------ dry-run validation
R, K, H, TMAX, EPS = 2, 2, 256, 64, 1e-6
BASE = 1 << 40            # fake device addresses, 16-byte aligned, far apart
MB = 1 << 20


class Fake:
    """Fake, non-overlapping, 16-byte-aligned device addresses for one call."""

    def __init__(self, T=4, rows_e=None):
        self.T = T
        self.rows_e = rows_e if rows_e is not None else T * K
        a = iter(range(BASE, BASE + 64 * MB, MB))
        self.E = [next(a) for _ in range(R)]
        self.S = [next(a) for _ in range(R)]
        self.perm, self.w, self.res, self.gamma = next(a), next(a), next(a), next(a)
        self.out, self.rout = next(a), next(a)

    def call(self, lib, ws, **over):
        f = dict(E=self.E, rows_e=self.rows_e, perm=self.perm, w=self.w, S=self.S, res=self.res,
                 gamma=self.gamma, wb=0.0, eps=EPS, T=self.T, R=R, K=K, H=H, out=self.out,
                 rout=self.rout, f32=0)
        f.update(over)
        E = (ctypes.c_void_p * len(f["E"]))(*f["E"]) if f["E"] is not None else None
        S = (ctypes.c_void_p * len(f["S"]))(*f["S"]) if f["S"] is not None else None
        return lib.ar_finalize_rmsnorm(ctypes.c_void_p(ws.handle), ctypes.cast(E, ctypes.c_void_p) if E else None,
                                       f["rows_e"], f["perm"], f["w"],
                                       ctypes.cast(S, ctypes.c_void_p) if S else None, f["res"],
                                       f["gamma"], f["wb"], f["eps"], f["T"], f["R"], f["K"], f["H"],
                                       f["out"], f["rout"], f["f32"], None)


@pytest.fixture()
def ws(lib):
    w = arf.ar_workspace_create(R, K, H, TMAX, EPS, flags=arf.AR_WS_DRY_RUN)
    yield w
    w.destroy()


def test_valid_call_validates(lib, ws):
    f = Fake()
    assert f.call(lib, ws) == arf.AR_VALIDATED
    assert f.call(lib, ws, S=None) == arf.AR_VALIDATED            # no shared term
    assert f.call(lib, ws, rout=f.res) == arf.AR_VALIDATED        # in-place bf16 residual
    assert f.call(lib, ws, f32=1) == arf.AR_VALIDATED
    assert f.call(lib, ws, rows_e=1) == arf.AR_VALIDATED          # perm is checked on device


def test_zero_tokens_is_a_noop(lib, ws):
    f = Fake()
    assert f.call(lib, ws, T=0, res=None, out=None, rout=None) == arf.AR_OK


@pytest.mark.parametrize("over,status", [
    (dict(res=None), arf.AR_ERR_INVALID_ARG),                  # residual is mandatory
    (dict(gamma=None), arf.AR_ERR_INVALID_ARG),
    (dict(out=None), arf.AR_ERR_INVALID_ARG),
    (dict(rout=None), arf.AR_ERR_INVALID_ARG),
    (dict(perm=None), arf.AR_ERR_INVALID_ARG),
    (dict(w=None), arf.AR_ERR_INVALID_ARG),
    (dict(E=None), arf.AR_ERR_INVALID_ARG),
    (dict(rows_e=0), arf.AR_ERR_INVALID_ARG),
    (dict(R=3, E=[BASE] * 3, S=[BASE] * 3), arf.AR_ERR_INVALID_ARG),   # R differs from workspace
    (dict(K=1), arf.AR_ERR_INVALID_ARG),                      # K differs
    (dict(H=512), arf.AR_ERR_INVALID_ARG),                    # H differs
    (dict(eps=1e-5), arf.AR_ERR_INVALID_ARG),                 # eps differs
    (dict(T=-1), arf.AR_ERR_INVALID_ARG),
    (dict(T=TMAX + 1), arf.AR_ERR_CAPACITY),
    (dict(f32=2), arf.AR_ERR_INVALID_ARG),
    (dict(R=17), arf.AR_ERR_INVALID_ARG),
    (dict(K=17), arf.AR_ERR_INVALID_ARG),
])
def test_call_rejects(lib, ws, over, status):
    assert Fake().call(lib, ws, **over) == status


@pytest.mark.parametrize("field", ["res", "gamma", "out", "rout"])
def test_misaligned_pointer(lib, ws, field):
    f = Fake()
    assert f.call(lib, ws, **{field: getattr(f, field) + 8}) == arf.AR_ERR_ALIGNMENT


def test_misaligned_expert_and_shared_and_meta(lib, ws):
    f = Fake()
    assert f.call(lib, ws, E=[f.E[0], f.E[1] + 2]) == arf.AR_ERR_ALIGNMENT
    assert f.call(lib, ws, S=[f.S[0] + 4, f.S[1]]) == arf.AR_ERR_ALIGNMENT
    assert f.call(lib, ws, perm=f.perm + 2) == arf.AR_ERR_ALIGNMENT
    assert f.call(lib, ws, w=f.w + 1) == arf.AR_ERR_ALIGNMENT
    assert f.call(lib, ws, perm=f.perm + 4) == arf.AR_VALIDATED   # 4-byte alignment is enough


def test_null_entries_in_pointer_tables(lib, ws):
    f = Fake()
    assert f.call(lib, ws, E=[f.E[0], 0]) == arf.AR_ERR_INVALID_ARG
    assert f.call(lib, ws, S=[0, f.S[1]]) == arf.AR_ERR_INVALID_ARG


def test_overlapping_outputs_are_rejected(lib, ws):
    f = Fake()
    assert f.call(lib, ws, out=f.rout) == arf.AR_ERR_INVALID_ARG          # out == residual_out
    assert f.call(lib, ws, out=f.res) == arf.AR_ERR_INVALID_ARG           # out over the residual
    assert f.call(lib, ws, rout=f.res, f32=1) == arf.AR_ERR_INVALID_ARG   # fp32 cannot alias
    assert f.call(lib, ws, rout=f.res + 16) == arf.AR_ERR_INVALID_ARG     # partial alias
    assert f.call(lib, ws, out=f.E[1] + 32) == arf.AR_ERR_INVALID_ARG     # inside an expert buffer
    assert f.call(lib, ws, rout=f.S[0]) == arf.AR_ERR_INVALID_ARG
    assert f.call(lib, ws, out=f.gamma) == arf.AR_ERR_INVALID_ARG
    assert f.call(lib, ws, out=f.perm) == arf.AR_ERR_INVALID_ARG


def test_nothing_to_reduce(lib):
    w = arf.ar_workspace_create(R, 0, H, TMAX, EPS, flags=arf.AR_WS_DRY_RUN)
    try:
        f = Fake()
        assert f.call(lib, w, K=0, E=None, perm=None, w=None, S=None) == arf.AR_ERR_INVALID_ARG
        assert f.call(lib, w, K=0, E=None, perm=None, w=None) == arf.AR_VALIDATED
    finally:
        w.destroy()


def test_ar_rmsnorm_validation(lib):
    w = arf.ar_workspace_create(R, 4, H, TMAX, EPS, flags=arf.AR_WS_DRY_RUN)
    try:
        f = Fake()
        P = (ctypes.c_void_p * R)(*f.S)
        h = ctypes.c_void_p(w.handle)
        call = lambda **o: lib.ar_rmsnorm(h, o.get("P", ctypes.cast(P, ctypes.c_void_p)), o.get("R", R),
                                          o.get("res", f.res), f.gamma, 0.0, o.get("eps", EPS),
                                          o.get("T", 4), o.get("H", H), o.get("out", f.out),
                                          o.get("rout", f.rout), 0, None)
        assert call() == arf.AR_VALIDATED              # the workspace's top_k is not used
        assert call(P=None) == arf.AR_ERR_INVALID_ARG
        assert call(res=None) == arf.AR_ERR_INVALID_ARG
        assert call(R=1) == arf.AR_ERR_INVALID_ARG
        assert call(H=128) == arf.AR_ERR_INVALID_ARG
        assert call(eps=0.5) == arf.AR_ERR_INVALID_ARG
        assert call(T=TMAX + 1) == arf.AR_ERR_CAPACITY
        assert call(out=f.S[1]) == arf.AR_ERR_INVALID_ARG
    finally:
        w.destroy()


def test_regime_setter(lib, ws):
    assert arf.ar_workspace_last_regime(ws) == (0, 0)     # nothing planned yet
    for r in (arf.AR_REGIME_AUTO, arf.AR_REGIME_CLUSTER, arf.AR_REGIME_STREAM, arf.AR_REGIME_ONESHOT):
        arf.ar_workspace_set_regime(ws, r)
        assert Fake().call(lib, ws) == arf.AR_VALIDATED
        if r != arf.AR_REGIME_AUTO:                       # a dry run records its plan
            assert arf.ar_workspace_last_regime(ws)[0] == r
    with pytest.raises(arf.ArfuseError):
        arf.ar_workspace_set_regime(ws, 7)
    assert arf.ar_workspace_last_regime(ws)[0] == arf.AR_REGIME_ONESHOT


def test_cluster_size_setter(lib, ws):
    arf.ar_workspace_set_regime(ws, arf.AR_REGIME_CLUSTER)
    for c in (0, 2, 4, 8, 16):
        arf.ar_workspace_set_cluster_size(ws, c)
        assert Fake().call(lib, ws) == arf.AR_VALIDATED
    for c in (1, -2, 17, 32):
        with pytest.raises(arf.ArfuseError):
            arf.ar_workspace_set_cluster_size(ws, c)


def test_stage_bytes_setter(lib, ws):
    for b in (0, 1024, 16384, 131072):
        arf.ar_workspace_set_stage_bytes(ws, b)
        assert Fake().call(lib, ws) == arf.AR_VALIDATED
    for b in (-1, 1023, 131073):
        with pytest.raises(arf.ArfuseError):
            arf.ar_workspace_set_stage_bytes(ws, b)


def test_producer_warps_setter(lib, ws):
    for n in (0, 1, 2, 3, 4):
        arf.ar_workspace_set_producer_warps(ws, n)
        assert Fake().call(lib, ws) == arf.AR_VALIDATED
    for n in (-1, 5, 32):
        with pytest.raises(arf.ArfuseError):
            arf.ar_workspace_set_producer_warps(ws, n)


def test_cluster_regime_needs_two_chunks(lib):
    """A row of one 16-byte chunk cannot be split over a cluster: a clean decline."""
    w = arf.ar_workspace_create(1, 1, 8, 4, EPS, flags=arf.AR_WS_DRY_RUN)
    try:
        f = Fake()
        arf.ar_workspace_set_regime(w, arf.AR_REGIME_CLUSTER)
        assert f.call(lib, w, R=1, K=1, H=8, E=f.E[:1], S=f.S[:1]) == arf.AR_ERR_UNSUPPORTED
        arf.ar_workspace_set_regime(w, arf.AR_REGIME_STREAM)
        assert f.call(lib, w, R=1, K=1, H=8, E=f.E[:1], S=f.S[:1]) == arf.AR_VALIDATED
    finally:
        w.destroy()


def test_dry_run_device_error_is_clear(lib, ws):
    assert arf.ar_workspace_device_error(ws) == 0


def test_binding_checks_shapes(lib, ws):
    import torch
    x = lambda *s, dt=torch.bfloat16: torch.zeros(s, dtype=dt)
    E = [x(8, H), x(8, H)]
    with pytest.raises(ValueError):
        arf.ar_finalize_rmsnorm(ws, E, torch.zeros(4, 2, dtype=torch.int32), x(4, 2, dt=torch.float32),
                                None, x(4, H), x(H + 8), 0.0, EPS)
    with pytest.raises(TypeError):
        arf.ar_finalize_rmsnorm(ws, E, torch.zeros(4, 2, dtype=torch.int64), x(4, 2, dt=torch.float32),
                                None, x(4, H), x(H), 0.0, EPS)
    # the message names the tensor, with its index in a list
    perm, w = torch.zeros(4, 2, dtype=torch.int32), x(4, 2, dt=torch.float32)
    with pytest.raises(TypeError, match=r"expert_out\[1\]: dtype"):
        arf.ar_finalize_rmsnorm(ws, [E[0], x(8, H, dt=torch.float16)], perm, w, None, x(4, H), x(H), 0.0, EPS)
    with pytest.raises(ValueError, match=r"expert_out\[0\]: must be contiguous"):
        arf.ar_finalize_rmsnorm(ws, [x(H, 8).t(), E[1]], perm, w, None, x(4, H), x(H), 0.0, EPS)
    with pytest.raises(ValueError, match=r"shared_out\[1\]: shape"):
        arf.ar_finalize_rmsnorm(ws, E, perm, w, [x(4, H), x(3, H)], x(4, H), x(H), 0.0, EPS)


# ------------------------------------------------------------ gated shared expert
def _gated(lib, ws, f, gate, **over):
    a = dict(E=f.E, rows_e=f.rows_e, perm=f.perm, w=f.w, S=f.S, res=f.res, gamma=f.gamma, T=f.T,
             R=R, K=K, H=H, out=f.out, rout=f.rout, f32=0)
    a.update(over)
    E = ctypes.cast((ctypes.c_void_p * len(a["E"]))(*a["E"]), ctypes.c_void_p)
    S = ctypes.cast((ctypes.c_void_p * len(a["S"]))(*a["S"]), ctypes.c_void_p) if a["S"] else None
    return lib.ar_finalize_rmsnorm_gated(ctypes.c_void_p(ws.handle), E, a["rows_e"], a["perm"], a["w"],
                                         S, gate, a["res"], a["gamma"], 0.0, EPS, a["T"], a["R"], a["K"],
                                         a["H"], a["out"], a["rout"], a["f32"], None)


def test_gated_validation(lib, ws):
    f = Fake()
    gate = BASE + 40 * MB
    assert _gated(lib, ws, f, gate) == arf.AR_VALIDATED
    assert _gated(lib, ws, f, None) == arf.AR_ERR_INVALID_ARG           # gate required
    assert _gated(lib, ws, f, gate, S=None) == arf.AR_ERR_INVALID_ARG   # shared term required
    assert _gated(lib, ws, f, gate + 2) == arf.AR_ERR_ALIGNMENT
    assert _gated(lib, ws, f, f.out) == arf.AR_ERR_INVALID_ARG          # overlaps an output
    assert _gated(lib, ws, f, gate, T=0, res=None) == arf.AR_OK


def test_norm_bf16_h_flag_is_accepted(lib):
    w = arf.ar_workspace_create(R, K, H, TMAX, EPS, flags=arf.AR_WS_DRY_RUN | arf.AR_WS_NORM_BF16_H)
    try:
        assert Fake().call(lib, w) == arf.AR_VALIDATED
    finally:
        w.destroy()


# ------------------------------------------------ all-reduce + mHC write-back
def _mhc_call(lib, ws, **over):
    a = iter(range(BASE, BASE + 64 * MB, MB))
    f = dict(P=[next(a) for _ in range(R)], R=R, x=next(a), post=next(a), comb=next(a), T=4, H=H, hc=4,
             out=next(a))
    f.update(over)
    P = (ctypes.c_void_p * len(f["P"]))(*f["P"]) if f["P"] is not None else None
    return lib.ar_mhc_post(ctypes.c_void_p(ws.handle) if ws else None,
                           ctypes.cast(P, ctypes.c_void_p) if P else None, f["R"], f["x"], f["post"],
                           f["comb"], f["T"], f["H"], f["hc"], f["out"], None)


def test_mhc_post_validation(lib, ws):
    assert _mhc_call(lib, ws) == arf.AR_VALIDATED
    x = BASE + 40 * MB
    assert _mhc_call(lib, ws, x=x, out=x) == arf.AR_VALIDATED            # in place
    assert _mhc_call(lib, ws, x=x, out=x + 16) == arf.AR_ERR_INVALID_ARG  # partial overlap
    assert _mhc_call(lib, ws, T=0) == arf.AR_OK
    assert _mhc_call(lib, ws, T=TMAX + 1) == arf.AR_ERR_CAPACITY
    assert _mhc_call(lib, ws, R=R + 1, P=[BASE + i * MB for i in range(R + 1)]) == arf.AR_ERR_INVALID_ARG
    assert _mhc_call(lib, ws, H=H + 8) == arf.AR_ERR_INVALID_ARG
    for hc in (0, arf.AR_MAX_HC_STREAMS + 1):
        assert _mhc_call(lib, ws, hc=hc) == arf.AR_ERR_INVALID_ARG
    assert _mhc_call(lib, ws, hc=1) == arf.AR_VALIDATED
    assert _mhc_call(lib, ws, hc=arf.AR_MAX_HC_STREAMS) == arf.AR_VALIDATED
    for field in ("x", "out"):
        assert _mhc_call(lib, ws, **{field: BASE + 50 * MB + 8}) == arf.AR_ERR_ALIGNMENT
    for field in ("post", "comb"):
        assert _mhc_call(lib, ws, **{field: BASE + 50 * MB + 2}) == arf.AR_ERR_ALIGNMENT
    assert _mhc_call(lib, ws, P=[BASE + 8] + [BASE + (i + 1) * MB for i in range(R - 1)]) == arf.AR_ERR_ALIGNMENT
    for field in ("x", "post", "comb", "out"):
        assert _mhc_call(lib, ws, **{field: None}) == arf.AR_ERR_INVALID_ARG
    assert _mhc_call(lib, ws, P=None) == arf.AR_ERR_INVALID_ARG
    assert _mhc_call(lib, None) == arf.AR_ERR_INVALID_ARG
    # the output overlapping a partial, post or comb
    p0 = BASE + 30 * MB
    assert _mhc_call(lib, ws, P=[p0] + [BASE + (i + 1) * MB for i in range(R - 1)], out=p0) == arf.AR_ERR_INVALID_ARG
    assert _mhc_call(lib, ws, post=BASE + 41 * MB, out=BASE + 41 * MB) == arf.AR_ERR_INVALID_ARG
    assert _mhc_call(lib, ws, comb=BASE + 42 * MB, out=BASE + 42 * MB) == arf.AR_ERR_INVALID_ARG


def test_split_rows_setter(lib, ws):
    for n in (0, 1, 2, arf.AR_MAX_SPLIT_PARTS):
        arf.ar_workspace_set_split_rows(ws, n)
        assert Fake().call(lib, ws) == arf.AR_VALIDATED
    for n in (-1, arf.AR_MAX_SPLIT_PARTS + 1):
        with pytest.raises(arf.ArfuseError):
            arf.ar_workspace_set_split_rows(ws, n)


def test_split_column_groups_setter(lib, ws):
    for n in range(9):
        arf.ar_workspace_set_split_column_groups(ws, n)
        assert Fake().call(lib, ws) == arf.AR_VALIDATED
    for n in (-1, 9, 16):
        with pytest.raises(arf.ArfuseError):
            arf.ar_workspace_set_split_column_groups(ws, n)
    arf.ar_workspace_set_split_column_groups(ws, 0)


def test_pdl_flag_is_accepted(lib):
    w = arf.ar_workspace_create(R, K, H, TMAX, EPS, flags=arf.AR_WS_DRY_RUN | arf.AR_WS_PDL)
    try:
        assert Fake().call(lib, w) == arf.AR_VALIDATED
    finally:
        w.destroy()
    h = ctypes.c_void_p()
    assert lib.ar_workspace_create(0, R, K, H, TMAX, EPS, arf.AR_WS_DRY_RUN | 0x8, ctypes.byref(h)) == \
        arf.AR_ERR_INVALID_ARG


def test_wait_timeout_injection_setter(lib):
    w = arf.ar_workspace_create(R, K, H, TMAX, EPS, flags=arf.AR_WS_DRY_RUN)
    try:
        arf.ar_workspace_inject_wait_timeout(w, 50_000)
        # the injected wait exists only in whole-row streaming: any other regime declines
        for regime in (arf.AR_REGIME_CLUSTER, arf.AR_REGIME_ONESHOT, arf.AR_REGIME_SPLIT):
            arf.ar_workspace_set_regime(w, regime)
            assert Fake().call(lib, w) == arf.AR_ERR_UNSUPPORTED
        arf.ar_workspace_set_regime(w, arf.AR_REGIME_STREAM)
        assert Fake().call(lib, w) == arf.AR_VALIDATED
        arf.ar_workspace_inject_wait_timeout(w, 0)
        arf.ar_workspace_set_regime(w, arf.AR_REGIME_SPLIT)
        assert Fake().call(lib, w) == arf.AR_VALIDATED
        for bad in (-1, 1_000_000_001):
            with pytest.raises(arf.ArfuseError):
                arf.ar_workspace_inject_wait_timeout(w, bad)
    finally:
        w.destroy()
    assert lib.ar_workspace_inject_wait_timeout(None, 1) == arf.AR_ERR_INVALID_ARG


def test_header_is_plain_c_and_the_library_links_from_c(lib, tmp_path):
    """include/arfuse.h compiles as C11 with warnings as errors, and a C
    program linked to libarfuse.so drives a dry-run workspace through the
    ABI (tests/host/abi_check.c)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("gcc not available")
    lib_dir = os.path.dirname(arf.LIB_PATH)
    exe = tmp_path / "abi_check"
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER),
                    os.path.join(HERE, "host", "abi_check.c"), "-L", lib_dir, "-larfuse",
                    "-Wl,-rpath," + lib_dir, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout

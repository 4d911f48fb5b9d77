"""Seeded random shapes against the CPU fp64 oracle (needs a GB300).

Each case draws (R, K, H, T, shared partials, weight_bias, eps) at random --
hidden sizes anywhere from one 16-byte chunk to the maximum, ragged against
every tile and group width -- and runs every kernel regime (forced, and the
automatic choice), both residual_out types, the split kernel under random
column-group counts (powers of two or not), and the forced regimes at a
random cluster size (odd sizes included).  A forced regime with no launch plan for the
shape must decline cleanly (AR_ERR_UNSUPPORTED, nothing launched).
Tolerances as in test_gpu_parity.
"""
import random

import pytest
import torch

import tp_reduce_moe_gb300 as arf
from gen import Config, make_inputs
from tests._util import check_bf16, check_f32, run_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
REGIMES = (arf.AR_REGIME_AUTO, arf.AR_REGIME_CLUSTER, arf.AR_REGIME_STREAM, arf.AR_REGIME_ONESHOT,
           arf.AR_REGIME_SPLIT)
N_CASES = 24
MAX_ELEMS = 24 << 20  # bf16 input elements per case (keeps the CPU side to seconds)


def _draw(i):
    rng = random.Random(1000 + i)
    while True:
        R = rng.randint(1, 16)
        K = rng.choice([0, 1, 2, 3, 5, 8, 10, 16])
        H = 8 * rng.choice([1, 2, 7, 33, 64, 129, 257, 448, 768, 896, 1024, 1537, 2048])
        T = rng.choice([1, 2, 3, 5, 8, 13, 16, 21, 40])
        shared = True if K == 0 else rng.random() < 0.7
        if (R * K * T + R * T + 2 * T) * H <= MAX_ELEMS:
            break
    wb = rng.choice([0.0, 0.0, 1.0])
    eps = rng.choice([1e-6, 1e-5])
    groups = rng.choice([0, 1, 2, 3, 4, 5, 6])
    csize = rng.choice([0, 0, 3, 5, 6, 9, 12])
    cfg = Config(f"fuzz{i}", 200 + i, R=R, K=K, H=H, Ts=(T,), eps=eps,
                 weights="softmax" if K > 0 else "none", s_sigma=1.0, has_shared=shared, weight_bias=wb)
    return cfg, T, groups, csize


CASES = [_draw(i) for i in range(N_CASES)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tp_reduce_moe_gb300 import build
    build.build()
    arf.load_library()
    torch.cuda.set_device(0)


def _to_dev(inp):
    d = dict(inp)
    for key in ("E", "S"):
        if inp[key] is not None:
            d[key] = [x.to(DEV) for x in inp[key]]
    for key in ("perm", "w", "residual", "gamma"):
        if inp[key] is not None:
            d[key] = inp[key].to(DEV)
    return d


@pytest.mark.parametrize("case", range(N_CASES),
                         ids=[f"R{c.R}K{c.K}H{c.H}T{t}S{int(c.has_shared)}G{g}C{cs}" for c, t, g, cs in CASES])
def test_random_shape(case):
    cfg, T, groups, csize = CASES[case]
    inp = make_inputs(cfg, T, seed=7 + case)
    ref = run_oracle(inp, want_abs=True)
    d = _to_dev(inp)
    ws = arf.ar_workspace_create(cfg.R, cfg.K, cfg.H, T, cfg.eps, device=0)
    ran = 0
    try:
        arf.ar_workspace_set_split_column_groups(ws, groups)
        arf.ar_workspace_set_cluster_size(ws, csize)
        for regime in REGIMES:
            arf.ar_workspace_set_regime(ws, regime)
            for fp32 in (False, True):
                try:
                    if cfg.K == 0:
                        out, r_out = arf.ar_rmsnorm(ws, d["S"], d["residual"], d["gamma"], cfg.weight_bias,
                                                    cfg.eps, residual_out_fp32=fp32)
                    else:
                        out, r_out = arf.ar_finalize_rmsnorm(
                            ws, d["E"], d["perm"], d["w"], d["S"], d["residual"], d["gamma"], cfg.weight_bias,
                            cfg.eps, residual_out_fp32=fp32, rows_e=d["rows_e"])
                except arf.ArfuseError as e:
                    assert regime != arf.AR_REGIME_AUTO and e.status == arf.AR_ERR_UNSUPPORTED, \
                        (regime, arf.ar_status_string(e.status))
                    continue
                torch.cuda.synchronize()
                ran += 1
                tag = f"fuzz {cfg.name} R={cfg.R} K={cfg.K} H={cfg.H} T={T} regime={regime} fp32={fp32}"
                check_bf16(out, ref["out"], tag + " out")
                if fp32:
                    check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
                else:
                    check_bf16(r_out, ref["h"], tag + " residual_out")
        assert ran >= 2  # at least the automatic choice, both residual_out types
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()

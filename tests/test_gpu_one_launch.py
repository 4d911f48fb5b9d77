"""One operator, one launch (needs a GB300).

The fused op replaces a finalize, a shared-expert add, a collective and an
RMSNorm; every call of it, in every regime, must be exactly one kernel launch
on the caller's stream -- no memset, no copy, no helper kernel (the split
rows of whole-row streaming reset their own counters on the device).  Counted
with the CUDA activity of torch's profiler.
"""
import pytest
import torch

import tp_reduce_moe_gb300 as arf
from gen import make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
OUR_KERNELS = ("stream_rows_kernel", "split_rows_kernel", "cluster_rows_kernel", "mhc_post_kernel")


def _to_dev(inp):
    d = dict(inp)
    for key in ("E", "S"):
        if inp[key] is not None:
            d[key] = [x.to(DEV) for x in inp[key]]
    for key in ("perm", "w", "residual", "gamma"):
        if inp[key] is not None:
            d[key] = inp[key].to(DEV)
    return d


def _device_activities(fn):
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    names = []
    for e in prof.events():
        if getattr(e, "device_type", None) == torch.autograd.DeviceType.CUDA:
            names.append(e.name)
    return names


@pytest.fixture(scope="module", autouse=True)
def _profiler_ready():
    """The first profiling session of a process may record no device activity
    while the profiler starts up: run one over a torch kernel first."""
    x = torch.ones(1024, device=DEV)
    for _ in range(3):
        if _device_activities(lambda: x.mul_(1.0)):
            return
    pytest.skip("the CUDA profiler records no device activity on this machine")


@pytest.mark.parametrize("cfg,T,regime", [
    ("dsv3_decode", 4, arf.AR_REGIME_AUTO),      # split kernel
    ("dsv3_decode", 64, arf.AR_REGIME_AUTO),     # column tiles over a cluster
    ("prefill", 200, arf.AR_REGIME_STREAM),      # whole rows, last wave split over CTAs
    ("dsv3_decode", 4, arf.AR_REGIME_ONESHOT),   # one-shot kernel
    ("ar_only", 16, arf.AR_REGIME_AUTO),         # K = 0 entry point
    ("tp16", 9, arf.AR_REGIME_AUTO),             # split kernel in two copy rounds
])
def test_one_call_is_one_kernel_launch(cfg, T, regime):
    if cfg == "tp16":
        from gen import Config
        cfg = Config("tp16", 97, R=16, K=10, H=8192, Ts=(T,), eps=1e-6, weights="softmax", has_shared=True)
    inp = make_inputs(cfg, T)
    d = _to_dev(inp)
    ws = arf.ar_workspace_create(inp["R"], inp["K"], inp["H"], T, inp["eps"], device=0)
    try:
        arf.ar_workspace_set_regime(ws, regime)
        out = torch.empty((T, inp["H"]), dtype=torch.bfloat16, device=DEV)
        r_out = torch.empty((T, inp["H"]), dtype=torch.bfloat16, device=DEV)

        def call():
            if inp["K"] == 0:
                arf.ar_rmsnorm(ws, d["S"], d["residual"], d["gamma"], d["weight_bias"], d["eps"],
                               out=out, residual_out=r_out)
            else:
                arf.ar_finalize_rmsnorm(ws, d["E"], d["perm"], d["w"], d["S"], d["residual"], d["gamma"],
                                        d["weight_bias"], d["eps"], out=out, residual_out=r_out,
                                        rows_e=d["rows_e"])

        call()  # first call: one-time set-up outside the profiled region
        names = _device_activities(call)
        ours = [n for n in names if any(k in n for k in OUR_KERNELS)]
        assert len(ours) == 1, names
        assert len(names) == 1, names      # nothing else on the device: no memset, no copy
    finally:
        ws.destroy()

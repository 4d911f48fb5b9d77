"""The device-side timeout path, driven without a GPU fault (needs a GB300).

Every pipeline wait in the kernels is bounded; when one runs out the kernel
records AR_DEVERR_TIMEOUT, skips its remaining waits, waits for its own bulk
copies still in flight and returns, so the caller can run the step on its own
unfused path (sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with
final RMSNorm", Changes: a decline must leave the owed reduction to the
caller).  Here the host injects the failure: with
ar_workspace_inject_wait_timeout set, whole-row streaming makes its consumers
wait on a barrier nothing arrives on, bounded by a short limit.  The call must
return, the error word must carry the timeout bit, and the next call without
the injection must match the oracle -- which also shows that the split-row
counters of the workspace were left (or reset) at zero.
"""
import pytest
import torch

import tp_reduce_moe_gb300 as arf
from gen import make_inputs
from tests._util import check_bf16, check_f32, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tp_reduce_moe_gb300 import build
    build.build()
    arf.load_library()
    torch.cuda.set_device(0)


def _call(ws, d, fp32):
    return arf.ar_finalize_rmsnorm(ws, d["E"], d["perm"], d["w"], d["S"], d["residual"], d["gamma"],
                                   d["weight_bias"], d["eps"], residual_out_fp32=fp32)


# tiny: whole rows only; prefill T = 3: every row split over 8 CTAs (last-wave
# split rows, which meet through the workspace's counters); dsv3 T = 200: one
# full wave of whole rows plus split rows of the last wave
@pytest.mark.parametrize("cfg,T", [("tiny", 4), ("prefill", 3), ("dsv3_decode", 200)])
def test_injected_wait_timeout_is_reported_and_the_next_call_is_clean(cfg, T):
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    d = {k: v for k, v in inp.items()}
    for key in ("E", "S"):
        d[key] = [x.cuda() for x in inp[key]]
    for key in ("perm", "w", "residual", "gamma"):
        d[key] = inp[key].cuda()
    ws = arf.ar_workspace_create(d["R"], d["K"], d["H"], T, d["eps"], device=0)
    try:
        arf.ar_workspace_set_regime(ws, arf.AR_REGIME_STREAM)
        assert arf.ar_workspace_device_error(ws) == 0
        arf.ar_workspace_inject_wait_timeout(ws, 50_000)  # 50 us
        for fp32 in (False, True):
            _call(ws, d, fp32)                 # returns AR_OK: the launch itself is fine
            err = arf.ar_workspace_device_error(ws)   # synchronises: the kernel has returned
            assert err & arf.AR_DEVERR_TIMEOUT, f"timeout bit not set (error word {err:#x})"
            assert not err & arf.AR_DEVERR_PERM_RANGE
        # other regimes decline while the injection is set
        arf.ar_workspace_set_regime(ws, arf.AR_REGIME_SPLIT if d["H"] // 8 >= 2 else arf.AR_REGIME_ONESHOT)
        with pytest.raises(arf.ArfuseError) as e:
            _call(ws, d, False)
        assert e.value.status == arf.AR_ERR_UNSUPPORTED
        # injection off: the same workspace computes the oracle's result again
        arf.ar_workspace_inject_wait_timeout(ws, 0)
        arf.ar_workspace_set_regime(ws, arf.AR_REGIME_STREAM)
        for fp32 in (False, True):
            out, r_out = _call(ws, d, fp32)
            torch.cuda.synchronize()
            check_bf16(out, ref["out"], f"{cfg} T={T} out after a timeout")
            if fp32:
                check_f32(r_out, ref["h"], ref["abs"], f"{cfg} T={T} residual_out after a timeout")
            else:
                check_bf16(r_out, ref["h"], f"{cfg} T={T} residual_out after a timeout")
        assert arf.ar_workspace_device_error(ws) == 0
        # the automatic choice works on the same workspace too
        arf.ar_workspace_set_regime(ws, arf.AR_REGIME_AUTO)
        out, r_out = _call(ws, d, False)
        torch.cuda.synchronize()
        check_bf16(out, ref["out"], f"{cfg} T={T} out (automatic regime) after a timeout")
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()

"""The allocation-free entry point, ar_finalize_rmsnorm_noalloc, through the C ABI.

Callers that may not allocate device memory -- code running while an engine
captures a CUDA graph, plugins whose host engine owns all device memory
through its own pool, deployments with a fixed memory budget -- cannot create
a workspace, because that allocates a small device block.  They call this
entry point instead; it keeps its one status word in a fixed array inside the
library.  Every case runs twice in a row on the same inputs, and each result
must match the CPU oracle with the parity suite's acceptance (bf16 outputs at
rtol = atol = 1e-2, fp32 residual_out at 1e-5 scaled by the condition of the
sum).  The cases reach every plan the automatic choice makes for these shapes:
the split kernel, 16-, 8- and 4-CTA column tiles, the one-shot kernel (K = 0),
whole-row streaming with a ragged last wave (which this entry point never
splits) and several waves.  This file is collected last so that a run stopping
at the first failure has run every other test first; it also passes on its own
in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import tp_reduce_moe_gb300 as arf
from gen import Config, make_inputs
from tests._util import check_bf16, check_f32, run_oracle, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def noalloc():
    from tp_reduce_moe_gb300 import build
    build.build()
    lib = arf.load_library()
    f = lib.ar_finalize_rmsnorm_noalloc
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    f.restype = I
    f.argtypes = [P, I64, P, P, P, P, P, F, F, I64, I, I, I, P, P, I, P]
    torch.cuda.set_device(0)
    return f


def _table(ts):
    if ts is None:
        return None
    return ctypes.cast((ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts]), ctypes.c_void_p)


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _call(f, d, out, r_out, fp32, T=None):
    stream = torch.cuda.current_stream().cuda_stream
    return f(_table(d["E"]), d["rows_e"] if d["K"] > 0 else 0, _ptr(d["perm"]), _ptr(d["w"]),
             _table(d["S"]), d["residual"].data_ptr(), d["gamma"].data_ptr(),
             float(d["weight_bias"]), float(d["eps"]), d["T"] if T is None else T, d["R"], d["K"],
             d["H"], out.data_ptr(), r_out.data_ptr(), 1 if fp32 else 0, stream)


def _to_dev(inp):
    d = dict(inp)
    for key in ("E", "S"):
        if inp[key] is not None:
            d[key] = [x.cuda() for x in inp[key]]
    for key in ("perm", "w", "residual", "gamma"):
        if inp[key] is not None:
            d[key] = inp[key].cuda()
    return d


def _outputs(d, fp32):
    T, H = d["T"], d["H"]
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    r_out = torch.full((T, H), float("nan"), dtype=torch.float32 if fp32 else torch.bfloat16,
                       device="cuda")
    return out, r_out


def _check(out, r_out, ref, fp32, tag):
    check_bf16(out, ref["out"], tag + " out")
    if fp32:
        check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
    else:
        check_bf16(r_out, ref["h"], tag + " residual_out")


# The plans the automatic choice makes: dsv3 T = 16 the split kernel in twelve-CTA clusters,
# T = 24 / 48 / 72 eight-CTA tiles (64 KB and 24 KB ring slots) and four-CTA tiles; prefill
# shape T = 64 four-CTA tiles with 48 KB slots and three producer warps, T = 200 eight-CTA tiles
# with 24 KB slots, T = 300 (past the table) whole rows with a ragged last wave (300 mod 152);
# glm T = 1 the split kernel in sixteen-CTA clusters; tiny T = 4 (six summands) and ar_only
# T = 16 / 200 the one-shot kernel in sixteen-, eight- and two-CTA clusters; the TP16 routing
# profile (R = 16, K = 10, H = 8192) at T = 9 the split kernel in two copy rounds
CASES = [("tiny", 4), ("dsv3_decode", 16), ("dsv3_decode", 24), ("dsv3_decode", 48),
         ("dsv3_decode", 72), ("prefill", 64), ("glm_gemma", 1), ("ar_only", 16), ("ar_only", 200),
         ("prefill", 200), ("prefill", 300), ("tp16", 9)]
TP16 = Config("tp16", 97, R=16, K=10, H=8192, Ts=(9,), eps=1e-6, weights="softmax", has_shared=True)


@pytest.mark.parametrize("cfg,T", CASES, ids=[f"{c}-T{t}" for c, t in CASES])
@pytest.mark.parametrize("fp32", [False, True])
def test_noalloc_matches_the_oracle(noalloc, cfg, T, fp32):
    inp = make_inputs(TP16 if cfg == "tp16" else cfg, T)
    ref = run_oracle(inp, want_abs=True)
    d = _to_dev(inp)
    for call in range(2):  # two calls in a row share the library's array
        out, r_out = _outputs(d, fp32)
        assert _call(noalloc, d, out, r_out, fp32) == arf.AR_OK
        torch.cuda.synchronize()
        _check(out, r_out, ref, fp32, f"noalloc {cfg} T={T} fp32={fp32} call {call}")


@pytest.mark.parametrize("fp32", [False, True])
def test_noalloc_several_waves_sampled(noalloc, fp32):
    # prefill T = 2048: whole-row streaming over more than one wave of CTAs;
    # sampled rows against the oracle
    T = 2048
    d = make_inputs("prefill", T, device="cuda")
    rng = np.random.default_rng(T)
    rows = sorted(set([0, 1, 151, 152, T // 2, T - 2, T - 1] + rng.integers(0, T, 25).tolist()))
    ref = run_oracle(sample_rows(d, rows), want_abs=True)
    idx = torch.as_tensor(rows, device="cuda")
    for call in range(2):
        out, r_out = _outputs(d, fp32)
        assert _call(noalloc, d, out, r_out, fp32) == arf.AR_OK
        torch.cuda.synchronize()
        _check(out[idx], r_out[idx], ref, fp32, f"noalloc prefill T={T} fp32={fp32} call {call}")
        del out, r_out


def test_noalloc_rejects_sizes_beyond_its_limits(noalloc):
    d = _to_dev(make_inputs("tiny", 4))
    out = torch.empty(4, 256, dtype=torch.bfloat16, device="cuda")
    r_out = torch.empty(4, 256, dtype=torch.bfloat16, device="cuda")
    assert _call(noalloc, d, out, r_out, False, T=(1 << 26) + 1) == arf.AR_ERR_CAPACITY
    assert _call(noalloc, dict(d, R=17), out, r_out, False) == arf.AR_ERR_INVALID_ARG
    assert _call(noalloc, dict(d, K=17), out, r_out, False) == arf.AR_ERR_INVALID_ARG
    assert _call(noalloc, dict(d, H=16392), out, r_out, False) == arf.AR_ERR_UNSUPPORTED
    assert _call(noalloc, dict(d, T=0), out, r_out, False) == arf.AR_OK  # nothing to do

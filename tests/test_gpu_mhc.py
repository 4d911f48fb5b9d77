"""GPU parity of ar_mhc_post (all-reduce + mHC residual write-back) against the
CPU fp64 oracle (needs a GB300).

Acceptance: every output stream within rtol = atol = 1e-2 of the oracle value
rounded to bf16 (the bf16 bar of the main op).  The oracle itself is pinned
only to this library's reading of hc_post (the pages give no formula), so
this parity is parity with that reading.
"""
import pytest
import torch

import oracle
import tp_reduce_moe_gb300 as arf
from gen import MHC_SHAPES, bf16_bits, make_mhc_inputs
from tests._util import check_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tp_reduce_moe_gb300 import build
    build.build()
    arf.load_library()
    torch.cuda.set_device(0)


def _ref(inp):
    return oracle.ar_mhc_post_ref([bf16_bits(p) for p in inp["P"]], bf16_bits(inp["x"]),
                                  inp["post"].numpy(), inp["comb"].numpy())


def _dev(inp):
    return ([p.to(DEV) for p in inp["P"]], inp["x"].to(DEV), inp["post"].to(DEV), inp["comb"].to(DEV))


def _run(R, H, hc, T, seed=777, inplace=False, max_tokens=None):
    inp = make_mhc_inputs(R, H, hc, T, seed=seed)
    ref = _ref(inp)
    ws = arf.ar_workspace_create(R, 0, H, max_tokens or max(T, 1), 1e-6, device=0)
    try:
        P, x, post, comb = _dev(inp)
        out = x if inplace else None
        got = arf.ar_mhc_post(ws, P, x, post, comb, out=out)
        torch.cuda.synchronize()
        assert arf.ar_workspace_device_error(ws) == 0
        return got, ref
    finally:
        ws.destroy()


CASES = [(s["R"], s["H"], s["hc"], T) for s in MHC_SHAPES.values() for T in s["Ts"]]


@pytest.mark.parametrize("R,H,hc,T", CASES, ids=[f"R{r}H{h}hc{c}T{t}" for r, h, c, t in CASES])
def test_mhc_shapes(R, H, hc, T):
    got, ref = _run(R, H, hc, T)
    check_bf16(got, ref, f"mhc R={R} H={H} hc={hc} T={T}")


@pytest.mark.parametrize("R,H,hc,T", [(1, 8, 1, 1), (5, 264, 3, 3), (16, 2056, 8, 33), (2, 1032, 2, 100),
                                      (4, 16384, 4, 2), (3, 120, 7, 17)])
def test_mhc_edge_shapes(R, H, hc, T):
    got, ref = _run(R, H, hc, T, seed=R * 31 + hc)
    check_bf16(got, ref, f"mhc edge R={R} H={H} hc={hc} T={T}")


def test_mhc_in_place():
    got, ref = _run(4, 5120, 4, 16, inplace=True)
    check_bf16(got, ref, "mhc in place")


def test_mhc_outputs_stay_in_bounds_and_zero_tokens():
    R, H, hc, T = 2, 264, 4, 5
    inp = make_mhc_inputs(R, H, hc, T)
    ref = _ref(inp)
    ws = arf.ar_workspace_create(R, 0, H, T, 1e-6, device=0)
    try:
        P, x, post, comb = _dev(inp)
        n = T * hc * H
        canary = torch.full((n + 2 * 64,), 12345.0, dtype=torch.bfloat16, device=DEV)
        out = canary[64:64 + n].view(T, hc, H)
        arf.ar_mhc_post(ws, P, x, post, comb, out=out)
        torch.cuda.synchronize()
        check_bf16(out, ref, "mhc canary")
        assert bool((canary[:64] == 12345.0).all()) and bool((canary[64 + n:] == 12345.0).all())
        before = out.clone()
        arf.ar_mhc_post(ws, [p[:0] for p in P], x[:0], post[:0], comb[:0], out=out[:0], T=0)
        torch.cuda.synchronize()
        assert torch.equal(out, before)
    finally:
        ws.destroy()


def test_mhc_graph_replay_and_reproducibility():
    R, H, hc, T = 4, 6144, 4, 8
    a = make_mhc_inputs(R, H, hc, T, seed=1)
    b = make_mhc_inputs(R, H, hc, T, seed=2)
    ws = arf.ar_workspace_create(R, 0, H, T, 1e-6, device=0)
    try:
        P, x, post, comb = _dev(a)
        out = torch.empty_like(x)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            arf.ar_mhc_post(ws, P, x, post, comb, out=out, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        first = out.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            arf.ar_mhc_post(ws, P, x, post, comb, out=out)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, first)
        Pb, xb, postb, combb = _dev(b)
        for dst, src in zip(P + [x, post, comb], Pb + [xb, postb, combb]):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        check_bf16(out, _ref(b), "mhc graph replay with new inputs")
    finally:
        ws.destroy()

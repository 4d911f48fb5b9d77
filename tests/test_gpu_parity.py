"""GPU parity of libarfuse against the CPU fp64 oracle (needs a GB300).

Every call goes through the C ABI (via the ctypes binding).  Acceptance:
  out and bf16 residual_out: |g - o_bf16| <= 1e-2 + 1e-2 |o_bf16|  (torch.allclose
    at rtol = atol = 1e-2 against the oracle rounded to bf16; sglang PR #37104
    "perf(mtp): fuse trailing TP all-reduce with final RMSNorm", Correctness);
  fp32 residual_out: |g - o| <= 1e-5 max(|o|, sum |terms|);
  perm handling: bit-exact (perm-decode inputs).
"""
import numpy as np
import pytest
import torch

import oracle
import tp_reduce_moe_gb300 as arf
from gen import CONFIGS, Config, make_inputs, make_perm_decode_inputs
from tests._util import check_bf16, check_f32, oracle_args, run_oracle, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
REGIMES = (arf.AR_REGIME_CLUSTER, arf.AR_REGIME_STREAM, arf.AR_REGIME_ONESHOT, arf.AR_REGIME_SPLIT,
           arf.AR_REGIME_AUTO)
KERNELS = (arf.AR_REGIME_CLUSTER, arf.AR_REGIME_STREAM, arf.AR_REGIME_ONESHOT, arf.AR_REGIME_SPLIT)
# Regimes that split a row over several CTAs cannot run a row of one 16-byte chunk.
SPLITTING = (arf.AR_REGIME_CLUSTER, arf.AR_REGIME_SPLIT)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tp_reduce_moe_gb300 import build
    build.build()
    arf.load_library()
    torch.cuda.set_device(0)


def to_dev(inp):
    d = dict(inp)
    for key in ("E", "S"):
        if inp[key] is not None:
            d[key] = [x.to(DEV) for x in inp[key]]
    for key in ("perm", "w", "residual", "gamma"):
        if inp[key] is not None:
            d[key] = inp[key].to(DEV)
    return d


def make_ws(inp, max_tokens=None):
    return arf.ar_workspace_create(inp["R"], inp["K"], inp["H"], max_tokens or max(inp["T"], 1),
                                   inp["eps"], device=0)


def run_gpu(ws, d, fp32=False, regime=arf.AR_REGIME_AUTO, **kw):
    arf.ar_workspace_set_regime(ws, regime)
    if d["K"] == 0 and kw.pop("use_rmsnorm", True):
        return arf.ar_rmsnorm(ws, d["S"], d["residual"], d["gamma"], d["weight_bias"], d["eps"],
                              residual_out_fp32=fp32, **kw)
    return arf.ar_finalize_rmsnorm(ws, d["E"] if d["E"] is not None else [], d["perm"], d["w"], d["S"],
                                   d["residual"], d["gamma"], d["weight_bias"], d["eps"],
                                   residual_out_fp32=fp32, rows_e=d["rows_e"], **kw)


def check_all(ws, d, ref, what, regimes=REGIMES, fp32s=(False, True), declines=()):
    for regime in regimes:
        for fp32 in fp32s:
            if regime in declines:   # no launch plan for this shape: a clean decline
                with pytest.raises(arf.ArfuseError) as e:
                    run_gpu(ws, d, fp32=fp32, regime=regime)
                assert e.value.status == arf.AR_ERR_UNSUPPORTED
                continue
            if regime in SPLITTING and d["H"] // 8 < 2:
                with pytest.raises(arf.ArfuseError) as e:   # one chunk cannot be split
                    run_gpu(ws, d, fp32=fp32, regime=regime)
                assert e.value.status == arf.AR_ERR_UNSUPPORTED
                continue
            out, r_out = run_gpu(ws, d, fp32=fp32, regime=regime)
            torch.cuda.synchronize()
            tag = f"{what} regime={regime} fp32={fp32}"
            check_bf16(out, ref["out"], tag + " out")
            if fp32:
                check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
            else:
                check_bf16(r_out, ref["h"], tag + " residual_out")
            got_regime, _ = arf.ar_workspace_last_regime(ws)
            if regime != arf.AR_REGIME_AUTO:
                assert got_regime == regime
    assert arf.ar_workspace_device_error(ws) == 0


# ------------------------------------------------ every config at every T, fully
FULL_CASES = [(n, T) for n, c in CONFIGS.items() for T in c.Ts if not (n == "prefill" and T > 512)]


@pytest.mark.parametrize("cfg,T", FULL_CASES, ids=[f"{n}-T{T}" for n, T in FULL_CASES])
def test_config_full(cfg, T):
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        check_all(ws, to_dev(inp), ref, f"{cfg} T={T}")
    finally:
        ws.destroy()


# ----------------------------- full-size prefill: sampled rows against the oracle
@pytest.mark.parametrize("T", [2048, 8192])
def test_prefill_full_size_sampled(T):
    d = make_inputs("prefill", T, device=DEV)
    rng = np.random.default_rng(T)
    rows = sorted(set([0, 1, T // 2, T - 2, T - 1] + rng.integers(0, T, 59).tolist()))
    ref = run_oracle(sample_rows(d, rows), want_abs=True)
    ws = make_ws(d)
    try:
        for regime in REGIMES:
            for fp32 in (False, True):
                out, r_out = run_gpu(ws, d, fp32=fp32, regime=regime)
                torch.cuda.synchronize()
                idx = torch.as_tensor(rows, device=DEV)
                tag = f"prefill T={T} regime={regime} fp32={fp32}"
                check_bf16(out[idx], ref["out"], tag + " out")
                if fp32:
                    check_f32(r_out[idx], ref["h"], ref["abs"], tag + " residual_out")
                else:
                    check_bf16(r_out[idx], ref["h"], tag + " residual_out")
                # a property that holds at any size: every row of out has the
                # RMS of gamma-scaled unit rows, so no row was skipped
                assert torch.isfinite(out.float()).all()
                del out, r_out
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# -------------------------------------------------- perm decode, bit-exact
DECODE_CASES = [(2, 2, 256, 4), (2, 8, 7168, 128), (8, 8, 7168, 128), (8, 8, 6144, 16),
                (8, 10, 8192, 8192), (8, 10, 8192, 512), (16, 16, 256, 37), (1, 1, 64, 3)]


@pytest.mark.parametrize("R,K,H,T", DECODE_CASES, ids=[f"R{r}K{k}H{h}T{t}" for r, k, h, t in DECODE_CASES])
def test_perm_decode_bit_exact(R, K, H, T):
    ws = arf.ar_workspace_create(R, K, H, T, 1e-6, device=0)
    try:
        for shift in range(min(K, 3)):
            d = make_perm_decode_inputs(R, K, H, T, hot_shift=shift, seed=shift, device=DEV)
            D = d["digits"]
            want = d["perm"][torch.arange(T, device=DEV), d["hot"]].long()
            cols = torch.arange(H, device=DEV)
            expect = (want.view(-1, 1) >> (4 * (cols % D)).view(1, -1)) & 15
            for regime in KERNELS:
                for fp32 in (False, True):
                    _, r_out = run_gpu(ws, d, fp32=fp32, regime=regime)
                    torch.cuda.synchronize()
                    got = r_out.float()
                    assert torch.equal(got, got.round())
                    bad = (got.long() != expect)
                    assert not bad.any(), (f"perm decode mismatch regime={regime} fp32={fp32}: "
                                           f"{int(bad.sum())} elements, first row "
                                           f"{int(bad.any(1).nonzero()[0])}")
            del d
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# ------------------------------------------------------------------ edge cases
EDGE = [
    # (R, K, H, T, shared)
    (1, 1, 8, 1, False),        # smallest row: one 16-byte chunk
    (1, 1, 56, 5, True),        # 7 chunks: no cluster split divides it
    (3, 5, 264, 9, True),       # odd everything, 33 chunks
    (16, 16, 128, 3, True),     # maximum R and K
    (16, 16, 2048, 40, False),
    (2, 3, 16384, 20, True),    # maximum hidden (4 chunks per stream consumer)
    (4, 2, 12296, 7, True),     # ragged: 1537 chunks, last consumer warp partial
    (8, 8, 7168, 333, True),    # T not a multiple of the SM count, both kernels
    (16, 16, 16384, 3, True),   # the heaviest row the library takes: 273 segments of 32 KB
]
# Forced regimes with no launch plan for a shape, which must decline cleanly: at the heaviest row
# the one-shot kernel would need more than 768 threads per CTA, and the split kernel more than 32
# segments per CTA or more shared memory than an SM has.
EDGE_DECLINES = {(16, 16, 16384, 3, True): (arf.AR_REGIME_ONESHOT, arf.AR_REGIME_SPLIT)}


@pytest.mark.parametrize("R,K,H,T,shared", EDGE, ids=[f"R{a}K{b}H{c}T{d}S{int(e)}" for a, b, c, d, e in EDGE])
def test_edge_shapes(R, K, H, T, shared):
    from gen import Config
    cfg = Config("edge", 99, R=R, K=K, H=H, Ts=(T,), eps=1e-6, weights="softmax",
                 has_shared=shared)
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp, max_tokens=T + 5)
    try:
        check_all(ws, to_dev(inp), ref, f"edge R={R} K={K} H={H} T={T}",
                  declines=EDGE_DECLINES.get((R, K, H, T, shared), ()))
    finally:
        ws.destroy()


def test_k0_through_finalize_entry_point():
    inp = make_inputs("ar_only", 16)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        out, r_out = run_gpu(ws, d, use_rmsnorm=False)
        out2, r_out2 = run_gpu(ws, d)
        torch.cuda.synchronize()
        check_bf16(out, ref["out"], "K=0 via ar_finalize_rmsnorm")
        assert torch.equal(out, out2) and torch.equal(r_out, r_out2)
    finally:
        ws.destroy()


def test_gemma_raw_checkpoint_weight_bias():
    """weight_bias = 1 with the raw checkpoint gamma equals the stored +1 form."""
    inp = make_inputs("glm_gemma", 8)
    g_plus = (torch.rand(inp["H"], generator=torch.Generator().manual_seed(1)) + 1.0).to(torch.bfloat16)
    g_ckpt = (g_plus.float() - 1.0).to(torch.bfloat16)
    inp["gamma"] = g_ckpt
    inp["weight_bias"] = 1.0
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        check_all(ws, d, ref, "gemma raw checkpoint", fp32s=(False,))
        a, _ = run_gpu(ws, d)
        d2 = dict(d, gamma=g_plus.to(DEV), weight_bias=0.0)
        b, _ = run_gpu(ws, d2)
        torch.cuda.synchronize()
        assert (a.float() - b.float()).abs().max().item() <= 2 ** -6 * a.float().abs().max().item()
    finally:
        ws.destroy()


def test_in_place_residual():
    inp = make_inputs("dsv3_decode", 16)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        for regime in KERNELS:
            d = to_dev(inp)
            out, r_out = run_gpu(ws, d, regime=regime, residual_out=d["residual"])
            torch.cuda.synchronize()
            assert r_out.data_ptr() == d["residual"].data_ptr()
            check_bf16(out, ref["out"], f"in-place out regime={regime}")
            check_bf16(d["residual"], ref["h"], f"in-place residual regime={regime}")
    finally:
        ws.destroy()


@pytest.mark.parametrize("perm_kind", ["expert_sorted", "duplicates", "wide_rows"])
def test_perm_structures(perm_kind):
    inp = make_inputs("dsv3_decode", 64, perm_kind="expert_sorted" if perm_kind == "expert_sorted" else "random")
    if perm_kind == "duplicates":
        g = torch.Generator().manual_seed(3)
        inp["perm"] = torch.randint(0, 5, inp["perm"].shape, generator=g, dtype=torch.int32)
    if perm_kind == "wide_rows":   # expert buffers with more rows than T*K (padding)
        extra = 77
        inp["E"] = [torch.cat([e, torch.randn(extra, inp["H"]).to(torch.bfloat16)]) for e in inp["E"]]
        inp["rows_e"] += extra
        inp["perm"] = (inp["perm"] + extra).to(torch.int32)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        check_all(ws, to_dev(inp), ref, f"perm {perm_kind}")
    finally:
        ws.destroy()


def test_perm_out_of_range_sets_error_and_never_faults():
    inp = make_inputs("dsv3_decode", 4)
    bad = inp["perm"].clone()
    bad[2, 3] = inp["rows_e"] + 1000
    bad[3, 0] = -7
    ws = make_ws(inp)
    try:
        for regime in KERNELS:
            d = to_dev(dict(inp, perm=bad))
            out, _ = run_gpu(ws, d, regime=regime)
            code = arf.ar_workspace_device_error(ws)
            assert code & arf.AR_DEVERR_PERM_RANGE
            assert arf.ar_workspace_device_error(ws) == 0          # read clears it
            # untouched rows are still right
            ref = run_oracle(dict(inp))
            check_bf16(out[:2], ref["out"][:2], f"rows before the bad slots regime={regime}")
    finally:
        ws.destroy()


def test_outputs_stay_in_bounds():
    """Canary bytes around out and residual_out are never written."""
    inp = make_inputs("glm_gemma", 16)
    ws = make_ws(inp)
    T, H = inp["T"], inp["H"]
    try:
        for regime in KERNELS:
            for fp32 in (False, True):
                pad = 4096
                dt = torch.float32 if fp32 else torch.bfloat16
                ob = torch.full((2 * pad + T * H,), -7.0, dtype=torch.bfloat16, device=DEV)
                rb = torch.full((2 * pad + T * H,), -7.0, dtype=dt, device=DEV)
                out = ob[pad:pad + T * H].view(T, H)
                r_out = rb[pad:pad + T * H].view(T, H)
                run_gpu(ws, to_dev(inp), fp32=fp32, regime=regime, out=out, residual_out=r_out)
                torch.cuda.synchronize()
                for buf in (ob, rb):
                    assert (buf[:pad] == -7).all() and (buf[pad + T * H:] == -7).all()
    finally:
        ws.destroy()


def test_cuda_graph_replay_with_changing_inputs():
    """Capture once, then replay after overwriting the inputs in place."""
    ws = arf.ar_workspace_create(8, 8, 7168, 16, 1e-6, device=0)
    try:
        for regime in KERNELS:
            d = to_dev(make_inputs("dsv3_decode", 16, seed=1))
            out = torch.empty(16, 7168, dtype=torch.bfloat16, device=DEV)
            r_out = torch.empty(16, 7168, dtype=torch.bfloat16, device=DEV)
            arf.ar_workspace_set_regime(ws, regime)
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                run_gpu(ws, d, regime=regime, out=out, residual_out=r_out)   # warm-up
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                run_gpu(ws, d, regime=regime, out=out, residual_out=r_out)
            for seed in (2, 3):
                new = make_inputs("dsv3_decode", 16, seed=seed)
                for key in ("E", "S"):
                    for dst, src in zip(d[key], new[key]):
                        dst.copy_(src)
                for key in ("perm", "w", "residual", "gamma"):
                    d[key].copy_(new[key])
                g.replay()
                torch.cuda.synchronize()
                ref = run_oracle(new, want_abs=True)
                check_bf16(out, ref["out"], f"graph replay seed={seed} regime={regime}")
                check_bf16(r_out, ref["h"], f"graph replay residual seed={seed} regime={regime}")
            del g
    finally:
        ws.destroy()


def test_side_stream_and_back_to_back_calls():
    inp = make_inputs("dsv3_decode", 4)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        s = torch.cuda.Stream()
        outs = []
        with torch.cuda.stream(s):
            for regime in KERNELS * 3:
                outs.append(run_gpu(ws, d, regime=regime, stream=s)[0])
        s.synchronize()
        for o in outs:
            check_bf16(o, ref["out"], "side stream")
    finally:
        ws.destroy()


def test_wrong_device_or_mismatch_is_a_clean_decline():
    inp = make_inputs("tiny", 4)
    ws = arf.ar_workspace_create(2, 2, 256, 2, inp["eps"], device=0)
    try:
        with pytest.raises(arf.ArfuseError) as e:
            run_gpu(ws, to_dev(inp))          # T=4 > max_tokens=2
        assert e.value.status == arf.AR_ERR_CAPACITY
    finally:
        ws.destroy()


# ------------------------------------------- every cluster size of the cluster regime
@pytest.mark.parametrize("cfg,T", [("dsv3_decode", 4), ("glm_gemma", 16), ("prefill", 3), ("ar_only", 37)])
def test_every_cluster_size(cfg, T):
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        for c in (2, 4, 8, 16):
            arf.ar_workspace_set_cluster_size(ws, c)
            for fp32 in (False, True):
                out, r_out = run_gpu(ws, d, fp32=fp32, regime=arf.AR_REGIME_CLUSTER)
                torch.cuda.synchronize()
                assert arf.ar_workspace_last_regime(ws) == (arf.AR_REGIME_CLUSTER, c)
                check_bf16(out, ref["out"], f"{cfg} T={T} C={c} out")
                if fp32:
                    check_f32(r_out, ref["h"], ref["abs"], f"{cfg} T={T} C={c} residual_out")
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# ------------------------------------- gated shared expert (Qwen-style shared gate)
@pytest.mark.parametrize("cfg,T", [("tiny", 4), ("dsv3_decode", 4), ("glm_gemma", 16),
                                   ("dsv3_decode", 128), ("prefill", 512)])
def test_gated_shared_expert(cfg, T):
    from gen import make_gate_logits
    inp = make_inputs(cfg, T)
    gate = make_gate_logits(T)
    a = oracle_args(inp)
    ref = oracle.ar_finalize_rmsnorm_ref(a["E"], a["perm"], a["w"], a["S"], a["residual"], a["gamma"],
                                         a["weight_bias"], a["eps"], want_abs=True,
                                         shared_gate=gate.numpy())
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        g = gate.to(DEV)
        for regime in KERNELS:
            for fp32 in (False, True):
                out, r_out = run_gpu(ws, d, fp32=fp32, regime=regime, shared_gate=g)
                torch.cuda.synchronize()
                tag = f"gated {cfg} T={T} regime={regime} fp32={fp32}"
                check_bf16(out, ref["out"], tag + " out")
                if fp32:
                    check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
                else:
                    check_bf16(r_out, ref["h"], tag + " residual_out")
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# -------------------------------- the norm of bf16-rounded h (workspace flag)
@pytest.mark.parametrize("cfg,T", [("dsv3_decode", 16), ("ar_only", 8), ("prefill", 512)])
def test_norm_reads_bf16_h(cfg, T):
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True, h_bf16_before_norm=True)
    ws = arf.ar_workspace_create(inp["R"], inp["K"], inp["H"], T, inp["eps"], device=0,
                                 flags=arf.AR_WS_NORM_BF16_H)
    plain = make_ws(inp)
    try:
        d = to_dev(inp)
        for regime in KERNELS:
            out, r_out = run_gpu(ws, d, fp32=True, regime=regime)
            out0, _ = run_gpu(plain, d, fp32=True, regime=regime)
            torch.cuda.synchronize()
            check_bf16(out, ref["out"], f"bf16-h {cfg} T={T} regime={regime} out")
            check_f32(r_out, ref["h"], ref["abs"], f"bf16-h {cfg} T={T} regime={regime} residual_out")
            assert not torch.equal(out, out0)          # the flag changes the result ...
            assert (out.float() - out0.float()).abs().max().item() < 0.05   # ... within a few ulps
    finally:
        ws.destroy()
        plain.destroy()


def test_results_are_bitwise_reproducible():
    """Fixed summation order: repeated calls give identical bits, per kernel."""
    inp = make_inputs("dsv3_decode", 64)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        for regime in KERNELS:
            first = run_gpu(ws, d, regime=regime)
            for _ in range(3):
                again = run_gpu(ws, d, regime=regime)
                torch.cuda.synchronize()
                assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
    finally:
        ws.destroy()



@pytest.mark.parametrize("cfg,T", [("dsv3_decode", 4), ("glm_gemma", 16), ("prefill", 3), ("ar_only", 5),
                                   ("tiny", 4)])
def test_every_split_cluster_size(cfg, T):
    """The split regime at every cluster size whose plan fits shared memory; a
    size that does not fit is a clean AR_ERR_UNSUPPORTED."""
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    ran = 0
    try:
        d = to_dev(inp)
        for c in (2, 4, 8, 16):
            arf.ar_workspace_set_cluster_size(ws, c)
            for fp32 in (False, True):
                try:
                    out, r_out = run_gpu(ws, d, fp32=fp32, regime=arf.AR_REGIME_SPLIT)
                except arf.ArfuseError as e:
                    assert e.status == arf.AR_ERR_UNSUPPORTED
                    continue
                torch.cuda.synchronize()
                ran += 1
                assert arf.ar_workspace_last_regime(ws) == (arf.AR_REGIME_SPLIT, c)
                check_bf16(out, ref["out"], f"split {cfg} T={T} C={c} out")
                if fp32:
                    check_f32(r_out, ref["h"], ref["abs"], f"split {cfg} T={T} C={c} residual_out")
        assert ran >= 2
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


@pytest.mark.parametrize("cfg,T", [("dsv3_decode", 4), ("glm_gemma", 3), ("prefill", 2), ("tiny", 4),
                                   ("dsv3_decode", 48)])
def test_split_column_groups(cfg, T):
    """Split plans with column groups: C CTAs in G groups of C/G.  Every column
    is summed exactly as by the C/G-CTA split without groups (the same
    segments per CTA, the same slice order), so residual_out is bitwise
    identical to it; out differs from it only through the order of the tile
    sums of squares.  Oracle parity for every plan that fits."""
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        base = {}
        arf.ar_workspace_set_split_column_groups(ws, 1)
        for c in (2, 4, 8, 16):
            arf.ar_workspace_set_cluster_size(ws, c)
            try:
                out, r_out = run_gpu(ws, d, fp32=True, regime=arf.AR_REGIME_SPLIT)
            except arf.ArfuseError as e:
                assert e.status == arf.AR_ERR_UNSUPPORTED
                continue
            torch.cuda.synchronize()
            check_bf16(out, ref["out"], f"split {cfg} T={T} C={c} one group out")
            check_f32(r_out, ref["h"], ref["abs"], f"split {cfg} T={T} C={c} one group residual_out")
            base[c] = (out.clone(), r_out.clone())
        ran = 0
        for groups in (2, 4, 8):
            arf.ar_workspace_set_split_column_groups(ws, groups)
            for c in (4, 8, 16):
                arf.ar_workspace_set_cluster_size(ws, c)
                try:
                    out, r_out = run_gpu(ws, d, fp32=True, regime=arf.AR_REGIME_SPLIT)
                except arf.ArfuseError as e:
                    assert e.status == arf.AR_ERR_UNSUPPORTED
                    continue
                torch.cuda.synchronize()
                ran += 1
                tag = f"split {cfg} T={T} C={c} groups={groups}"
                assert arf.ar_workspace_last_regime(ws) == (arf.AR_REGIME_SPLIT, c), tag
                check_bf16(out, ref["out"], tag + " out")
                check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
                if c // groups in base:
                    assert torch.equal(r_out, base[c // groups][1]), tag
                    assert (out.float() - base[c // groups][0].float()).abs().max().item() < 0.05, tag
        assert ran >= 2
        arf.ar_workspace_set_split_column_groups(ws, 0)
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


SPLIT_EDGE = [
    # (R, K, H, T, shared): column groups of unequal width
    (3, 5, 264, 3, True),       # 33 chunks: groups of 17 + 16, 9 + 9 + 9 + 6, ...
    (2, 3, 2056, 5, True),      # 257 chunks: eight groups of 33, the last of 26
    (4, 2, 12296, 2, True),     # 1537 chunks: four groups of 385, the last of 382
    (1, 6, 1032, 4, False),     # 129 chunks, no shared partials
]


@pytest.mark.parametrize("R,K,H,T,shared", SPLIT_EDGE,
                         ids=[f"R{a}K{b}H{c}T{d}S{int(e)}" for a, b, c, d, e in SPLIT_EDGE])
def test_split_column_groups_ragged(R, K, H, T, shared):
    """Forced column groups on widths that do not divide evenly: oracle parity
    for every (cluster size, groups) with a plan, both residual_out types."""
    from gen import Config
    cfg = Config("split_edge", 98, R=R, K=K, H=H, Ts=(T,), eps=1e-6, weights="softmax",
                 has_shared=shared)
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp, max_tokens=T)
    ran = 0
    try:
        d = to_dev(inp)
        for groups in (2, 4, 8):
            arf.ar_workspace_set_split_column_groups(ws, groups)
            for c in (4, 8, 16):
                arf.ar_workspace_set_cluster_size(ws, c)
                for fp32 in (False, True):
                    try:
                        out, r_out = run_gpu(ws, d, fp32=fp32, regime=arf.AR_REGIME_SPLIT)
                    except arf.ArfuseError as e:
                        assert e.status == arf.AR_ERR_UNSUPPORTED
                        continue
                    torch.cuda.synchronize()
                    ran += 1
                    tag = f"split edge R={R} K={K} H={H} T={T} C={c} groups={groups} fp32={fp32}"
                    check_bf16(out, ref["out"], tag + " out")
                    if fp32:
                        check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
                    else:
                        check_bf16(r_out, ref["h"], tag + " residual_out")
        assert ran >= 4
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


@pytest.mark.parametrize("cfg,T,split_c", [("glm_gemma", 8, 8), ("tiny", 4, 4)])
def test_regime_table_routes_calls(cfg, T, split_c):
    """AR_REGIME_AUTO under a regime table runs the rule's regime and cluster
    size, with the same results as every other regime."""
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        for regime, ctas in ((arf.AR_REGIME_STREAM, 0), (arf.AR_REGIME_CLUSTER, 4),
                             (arf.AR_REGIME_ONESHOT, 0), (arf.AR_REGIME_SPLIT, split_c)):
            arf.ar_workspace_set_regime_table(ws, [(T, regime, ctas)])
            out, r_out = run_gpu(ws, d, fp32=True)
            torch.cuda.synchronize()
            got = arf.ar_workspace_last_regime(ws)
            assert got[0] == regime and (ctas == 0 or got[1] == ctas), (regime, ctas, got)
            check_bf16(out, ref["out"], f"table {cfg} T={T} regime={regime} out")
            check_f32(r_out, ref["h"], ref["abs"], f"table {cfg} T={T} regime={regime} residual_out")
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


@pytest.mark.parametrize("cfg,T", [("dsv3_decode", 16), ("tiny", 400), ("ar_only", 128)])
def test_tuning_controls_leave_results_unchanged(cfg, T):
    """Producer warps and slot sizes change only who issues which bulk copy and
    how copies are grouped, never the summation order: bitwise-identical
    outputs for every setting, in both streaming regimes, and oracle parity."""
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        for regime, ctas in ((arf.AR_REGIME_STREAM, 0), (arf.AR_REGIME_CLUSTER, 4)):
            arf.ar_workspace_set_cluster_size(ws, ctas)
            base = None
            for warps in (0, 1, 2, 3, 4):
                for stage in (0, 4096, 32768):
                    arf.ar_workspace_set_producer_warps(ws, warps)
                    arf.ar_workspace_set_stage_bytes(ws, stage)
                    out, r_out = run_gpu(ws, d, fp32=True, regime=regime)
                    torch.cuda.synchronize()
                    if base is None:
                        base = (out.clone(), r_out.clone())
                        check_bf16(out, ref["out"], f"{cfg} T={T} regime={regime} out")
                        check_f32(r_out, ref["h"], ref["abs"], f"{cfg} T={T} regime={regime} residual_out")
                    else:
                        assert torch.equal(out, base[0]) and torch.equal(r_out, base[1]), \
                            (regime, warps, stage)
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# a small heavy-row shape (37 segments per row: up to four parts) for split-row tests
SPLIT_CFG = Config("split_small", 9, R=4, K=8, H=512, Ts=(160,), eps=1e-6, weights="softmax")


@pytest.mark.parametrize("cfg,T", [(SPLIT_CFG, 153), (SPLIT_CFG, 170), (SPLIT_CFG, 7), ("dsv3_decode", 16),
                                   ("dsv3_decode", 64), ("glm_gemma", 16)],
                         ids=["small-T153", "small-T170", "small-T7", "dsv3-T16", "dsv3-T64", "glm-T16"])
def test_split_rows_of_the_last_wave(cfg, T):
    """Whole-row streaming with the last wave's rows split over several CTAs
    (partial rows meet in the workspace scratch, the last arriving CTA
    finishes the row): parity at every split cap, both residual_out types, and
    back-to-back calls (the arrival counters must come back to zero)."""
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        grids = set()
        for parts in (0, 2, 3, arf.AR_MAX_SPLIT_PARTS):
            arf.ar_workspace_set_split_rows(ws, parts)
            for fp32 in (False, True):
                for rep in range(3):
                    out, r_out = run_gpu(ws, d, fp32=fp32, regime=arf.AR_REGIME_STREAM)
                    torch.cuda.synchronize()
                    tag = f"split rows {getattr(cfg, 'name', cfg)} T={T} parts<={parts} fp32={fp32} call {rep}"
                    check_bf16(out, ref["out"], tag + " out")
                    if fp32:
                        check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
                    else:
                        check_bf16(r_out, ref["h"], tag + " residual_out")
            grids.add(arf.ar_workspace_last_regime(ws)[1])
        if T < torch.cuda.get_device_properties(0).multi_processor_count:
            assert len(grids) >= 2, grids   # the cap changed the launch (more CTAs per row)
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


@pytest.mark.parametrize("cfg,T", [("dsv3_decode", 4), ("dsv3_decode", 64), ("ar_only", 16), ("prefill", 3),
                                   ("dsv3_decode", 200)])
def test_pdl_chain_reads_the_previous_calls_output(cfg, T):
    """With AR_WS_PDL, calls launched back to back without a host sync, each
    reading the previous call's residual_out as its residual: every call must
    see its input complete (griddepcontrol.wait before the first global
    access).  Each step is checked against the oracle run on the residual the
    GPU actually fed it."""
    inp = make_inputs(cfg, T)
    ws = arf.ar_workspace_create(inp["R"], inp["K"], inp["H"], T, inp["eps"], device=0, flags=arf.AR_WS_PDL)
    try:
        d = to_dev(inp)
        steps = 5
        res = [d["residual"].clone()] + [torch.empty_like(d["residual"]) for _ in range(steps)]
        outs = [torch.empty_like(d["residual"]) for _ in range(steps)]
        for n in range(steps):
            dn = dict(d)
            dn["residual"] = res[n]
            run_gpu(ws, dn, out=outs[n], residual_out=res[n + 1])
        torch.cuda.synchronize()
        assert arf.ar_workspace_device_error(ws) == 0
        for n in range(steps):
            step = dict(inp)
            step["residual"] = res[n].cpu()
            ref = run_oracle(step)
            check_bf16(outs[n], ref["out"], f"pdl chain {cfg} T={T} step {n} out")
            check_bf16(res[n + 1], ref["h"], f"pdl chain {cfg} T={T} step {n} residual_out")
    finally:
        ws.destroy()


# ------------------------------- split kernel with more rows than resident clusters
@pytest.mark.parametrize("cfg,T,csize", [("dsv3_decode", 64, 16), ("dsv3_decode", 100, 8), ("glm_gemma", 40, 16),
                                         ("prefill", 30, 16), ("tiny", 1000, 4)])
def test_split_launch_of_more_rows_than_resident_clusters(cfg, T, csize):
    """When T exceeds the clusters the device runs at once, the split kernel's
    clusters (one row each) run in several waves -- or, for rows whose
    segments leave one CTA per SM, in the two-copy-round form when the device
    holds more of its clusters."""
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        arf.ar_workspace_set_cluster_size(ws, csize)
        d = to_dev(inp)
        for fp32 in (False, True):
            out, r_out = run_gpu(ws, d, fp32=fp32, regime=arf.AR_REGIME_SPLIT)
            torch.cuda.synchronize()
            assert arf.ar_workspace_last_regime(ws) == (arf.AR_REGIME_SPLIT, csize)
            tag = f"{cfg} T={T} split C={csize} fp32={fp32}"
            check_bf16(out, ref["out"], tag + " out")
            if fp32:
                check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
            else:
                check_bf16(r_out, ref["h"], tag + " residual_out")
        # the same call twice gives the same bits (fixed order whatever the grid)
        a1 = run_gpu(ws, d, fp32=True, regime=arf.AR_REGIME_SPLIT)
        a2 = run_gpu(ws, d, fp32=True, regime=arf.AR_REGIME_SPLIT)
        torch.cuda.synchronize()
        assert torch.equal(a1[0], a2[0]) and torch.equal(a1[1], a2[1])
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# ------------------------ trailing all-reduce of eight partials (K = 0, TP8)
@pytest.mark.parametrize("T", [16, 128, 256])
def test_eight_partial_allreduce_both_oneshot_forms(T):
    """The one-shot kernel's eight-load forms: 80 registers within one wave
    (T = 16), 64 registers once the launch no longer fits one wave of the
    80-register form (T = 128, 256; the switch itself is checked on the host)."""
    from gen import Config
    cfg = Config("ar8", 77, R=8, K=0, H=7168, Ts=(T,), eps=1e-6, weights="none", has_shared=True)
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        check_all(ws, to_dev(inp), ref, f"R=8 K=0 T={T}", regimes=(arf.AR_REGIME_ONESHOT, arf.AR_REGIME_AUTO))
    finally:
        ws.destroy()


# --------------------- regime-table rules with their own ring slots / producer warps
@pytest.mark.parametrize("cfg,T,ctas", [("dsv3_decode", 48, 8), ("dsv3_decode", 96, 8), ("glm_gemma", 96, 8),
                                        ("dsv3_decode", 128, 128), ("dsv3_decode", 192, 8), ("prefill", 64, 4)])
def test_builtin_rules_with_ring_variants(cfg, T, ctas):
    """The built-in tables run 24 KB slots and two producer warps for some
    clustered rules, and two producer warps for some whole-row rules; those
    plans meet the oracle like the default ones."""
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        rules = arf.ar_workspace_get_regime_table(ws)
        rule = next(r for r in rules if T <= r[0])
        assert rule[3:] != (0, 0)   # the rule sets its own slot size and/or producer warps
        for fp32 in (False, True):
            out, r_out = run_gpu(ws, d, fp32=fp32)
            torch.cuda.synchronize()
            assert arf.ar_workspace_last_regime(ws) == (rule[1], ctas)
            tag = f"{cfg} T={T} rule {rule} fp32={fp32}"
            check_bf16(out, ref["out"], tag + " out")
            if fp32:
                check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
            else:
                check_bf16(r_out, ref["h"], tag + " residual_out")
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# --------------------- clustered grids capped at the clusters the device co-schedules
@pytest.mark.parametrize("T,ctas,stage,producers", [(96, 4, 0, 0), (192, 4, 24576, 2), (256, 8, 24576, 2),
                                                     (48, 8, 32768, 2), (64, 4, 49152, 3)])
def test_clustered_grid_capped_at_coresident_clusters(T, ctas, stage, producers):
    """Clustered streaming plans whose shared-memory estimate asks for more
    clusters than a GB300 co-schedules (a cluster lives in one GPC) run on a
    grid capped at the co-resident count, each cluster taking more rows
    round-robin; the results meet the oracle like any other plan."""
    inp = make_inputs("dsv3_decode", T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        arf.ar_workspace_set_regime_table(ws, [(T, arf.AR_REGIME_CLUSTER, ctas, stage, producers)])
        d = to_dev(inp)
        for fp32 in (False, True):
            out, r_out = run_gpu(ws, d, fp32=fp32)
            torch.cuda.synchronize()
            assert arf.ar_workspace_last_regime(ws) == (arf.AR_REGIME_CLUSTER, ctas)
            grid = arf.ar_workspace_last_grid(ws)
            assert grid % ctas == 0 and 0 < grid <= T * ctas
            if (T, ctas, stage) == (192, 4, 24576):
                # 24 KB slots: three CTAs per SM by shared memory, 114 four-CTA clusters by that
                # estimate; a GB300 co-schedules fewer (clusters live in one GPC)
                assert grid < 456, grid
            tag = f"dsv3 T={T} tiles C={ctas} slots {stage} producers {producers} fp32={fp32}"
            check_bf16(out, ref["out"], tag + " out")
            if fp32:
                check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
            else:
                check_bf16(r_out, ref["h"], tag + " residual_out")
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# --------------------- the one-shot kernel at every cluster size
@pytest.mark.parametrize("cfg,T", [("ar_only", 1), ("ar_only", 37), ("tiny", 5), ("dsv3_decode", 2)])
def test_one_shot_every_cluster_size(cfg, T):
    """A rule or the workspace may fix the one-shot kernel's cluster size
    (fewer, larger CTAs per row); every power of two meets the oracle."""
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        d = to_dev(inp)
        for c in (2, 4, 8, 16):
            arf.ar_workspace_set_cluster_size(ws, c)
            for fp32 in (False, True):
                try:
                    out, r_out = run_gpu(ws, d, fp32=fp32, regime=arf.AR_REGIME_ONESHOT)
                except arf.ArfuseError as e:   # more CTAs than 16-byte chunks, or blocks too large
                    assert e.status == arf.AR_ERR_UNSUPPORTED
                    continue
                torch.cuda.synchronize()
                assert arf.ar_workspace_last_regime(ws) == (arf.AR_REGIME_ONESHOT, c)
                tag = f"one-shot {cfg} T={T} C={c} fp32={fp32}"
                check_bf16(out, ref["out"], tag + " out")
                if fp32:
                    check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
                else:
                    check_bf16(r_out, ref["h"], tag + " residual_out")
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# --------------------- split kernel: cluster sizes and column groups beyond powers of two
@pytest.mark.parametrize("cfg,T,combos", [
    ("dsv3_decode", 3, [(9, 3), (12, 3), (10, 2), (15, 5), (15, 3), (6, 2), (14, 2)]),
    ("glm_gemma", 5, [(9, 3), (12, 4), (12, 6), (10, 2)]),
    ("prefill", 2, [(9, 3), (12, 3), (10, 5)]),
    ("tiny", 7, [(6, 3), (9, 3), (12, 6), (10, 5)]),
])
def test_split_any_cluster_size_and_groups(cfg, T, combos):
    """Any cluster size 2..16 with column groups that divide it (ragged group
    widths included) meets the oracle; a combination whose CTAs would hold
    more than 32 segments is declined as AR_ERR_UNSUPPORTED."""
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    ran = 0
    try:
        d = to_dev(inp)
        for c, g in combos:
            arf.ar_workspace_set_cluster_size(ws, c)
            arf.ar_workspace_set_split_column_groups(ws, g)
            for fp32 in (False, True):
                try:
                    out, r_out = run_gpu(ws, d, fp32=fp32, regime=arf.AR_REGIME_SPLIT)
                except arf.ArfuseError as e:
                    assert e.status == arf.AR_ERR_UNSUPPORTED
                    continue
                torch.cuda.synchronize()
                assert arf.ar_workspace_last_regime(ws) == (arf.AR_REGIME_SPLIT, c)
                ran += 1
                tag = f"split {cfg} T={T} C={c} G={g} fp32={fp32}"
                check_bf16(out, ref["out"], tag + " out")
                if fp32:
                    check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
                else:
                    check_bf16(r_out, ref["h"], tag + " residual_out")
        assert ran > 0
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# --------------------- the TP16 routing profile (R = 16, K = 10, H = 8192) through its table
@pytest.mark.parametrize("T", [3, 9, 12, 32, 72])
def test_tp16_table_plans_meet_the_oracle(T):
    """Sixteen rank partials of top-10 rows at H = 8192 (177 segments per
    row): the built-in table's plan at decode and mid-range T -- split, tiles
    with default and smaller ring slots -- against the oracle."""
    from gen import Config
    cfg = Config("tp16", 97, R=16, K=10, H=8192, Ts=(T,), eps=1e-6, weights="softmax", has_shared=True)
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        assert arf.ar_workspace_get_regime_table(ws), "a built-in table for this shape"
        check_all(ws, to_dev(inp), ref, f"tp16 T={T}", regimes=(arf.AR_REGIME_AUTO,))
        plan = arf.ar_workspace_last_plan(ws)
        if T <= 12:   # the split kernel: one copy round while its clusters fit one wave, else two
            assert plan["regime"] == arf.AR_REGIME_SPLIT
            assert plan["copy_rounds"] == (1 if T <= 6 else 2)
    finally:
        ws.destroy()


# --------------------- split kernel in two copy rounds (half the segment buffers)
TWO_ROUND_CASES = [
    # (R, K, H, T, cluster size, column groups): two rounds because one round
    # has no plan (more than 32 segments for a CTA), or -- groups 0 at T >= 8 --
    # because the device holds more of the two-round form's clusters
    (16, 10, 8192, 1, 16, 4),
    (16, 10, 8192, 9, 16, 4),
    (16, 10, 8192, 8, 16, 0),
    (16, 10, 8192, 13, 16, 0),
    (8, 8, 7168, 1, 16, 8),
    (8, 8, 7168, 5, 16, 8),
    (8, 8, 7168, 3, 4, 2),
    (12, 12, 6144, 2, 12, 3),      # twelve-CTA clusters in three groups, 40 segments per CTA
    (10, 14, 6152, 3, 12, 3),      # ragged column groups (769 chunks), 38 segments per CTA
]


@pytest.mark.parametrize("R,K,H,T,csize,groups", TWO_ROUND_CASES,
                         ids=[f"R{c[0]}K{c[1]}H{c[2]}T{c[3]}C{c[4]}G{c[5]}" for c in TWO_ROUND_CASES])
def test_split_two_rounds_meets_the_oracle(R, K, H, T, csize, groups):
    """The split kernel with buffers for the first half of a CTA's segments:
    the second routed half is fetched into them once every consumer warp has
    folded the first.  Both residual_out types against the oracle, the error
    word clean, and the same bits on a second call."""
    from gen import Config
    cfg = Config("two_rounds", 98, R=R, K=K, H=H, Ts=(T,), eps=1e-6, weights="softmax", has_shared=True)
    inp = make_inputs(cfg, T)
    ref = run_oracle(inp, want_abs=True)
    ws = make_ws(inp)
    try:
        arf.ar_workspace_set_cluster_size(ws, csize)
        arf.ar_workspace_set_split_column_groups(ws, groups)
        d = to_dev(inp)
        check_all(ws, d, ref, f"two rounds R={R} K={K} H={H} T={T} C={csize} G={groups}",
                  regimes=(arf.AR_REGIME_SPLIT,))
        assert arf.ar_workspace_last_regime(ws) == (arf.AR_REGIME_SPLIT, csize)
        assert arf.ar_workspace_last_plan(ws)["copy_rounds"] == 2
        a1 = run_gpu(ws, d, fp32=True, regime=arf.AR_REGIME_SPLIT)
        a2 = run_gpu(ws, d, fp32=True, regime=arf.AR_REGIME_SPLIT)
        torch.cuda.synchronize()
        assert torch.equal(a1[0], a2[0]) and torch.equal(a1[1], a2[1])
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


@pytest.mark.parametrize("bf16_h", [False, True])
def test_split_two_rounds_gated_and_bf16_h(bf16_h):
    """Two copy rounds combined with the variants that change the first
    round's coefficients (a gated shared expert: the shared partials scaled by
    sigmoid(gate[t])) and the epilogue (the norm reading h rounded to bf16),
    both residual_out types, against the oracle."""
    from gen import make_gate_logits
    R, K, H, T = 16, 10, 8192, 9
    cfg = Config("two_rounds_gated", 99, R=R, K=K, H=H, Ts=(T,), eps=1e-6, weights="softmax", has_shared=True)
    inp = make_inputs(cfg, T)
    gate = make_gate_logits(T)
    a = oracle_args(inp)
    ref = oracle.ar_finalize_rmsnorm_ref(a["E"], a["perm"], a["w"], a["S"], a["residual"], a["gamma"],
                                         a["weight_bias"], a["eps"], want_abs=True, shared_gate=gate.numpy(),
                                         h_bf16_before_norm=bf16_h)
    ws = arf.ar_workspace_create(R, K, H, T, inp["eps"], device=0,
                                 flags=arf.AR_WS_NORM_BF16_H if bf16_h else 0)
    try:
        arf.ar_workspace_set_cluster_size(ws, 16)
        arf.ar_workspace_set_split_column_groups(ws, 4)
        d = to_dev(inp)
        g = gate.to(DEV)
        for fp32 in (False, True):
            out, r_out = run_gpu(ws, d, fp32=fp32, regime=arf.AR_REGIME_SPLIT, shared_gate=g)
            torch.cuda.synchronize()
            assert arf.ar_workspace_last_plan(ws)["copy_rounds"] == 2
            tag = f"two rounds gated bf16_h={bf16_h} fp32={fp32}"
            check_bf16(out, ref["out"], tag + " out")
            if fp32:
                check_f32(r_out, ref["h"], ref["abs"], tag + " residual_out")
            else:
                check_bf16(r_out, ref["h"], tag + " residual_out")
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


# ------------------------- independent callers: a workspace each, own streams and threads
def test_two_workspaces_on_two_streams_and_threads():
    """Two callers, each with its own workspace and stream -- whole rows whose
    last wave splits rows over CTAs (the workspace's scratch and counters)
    and column tiles over clusters -- launched interleaved without host syncs,
    first from one host thread, then from two threads at once (the library's
    shared host state: plan caches, occupancy queries).  Every output against
    the oracle; the error words stay clean."""
    import threading
    cases = [("prefill", 300), ("dsv3_decode", 64)]
    inps = [make_inputs(c, T) for c, T in cases]
    refs = [run_oracle(x) for x in inps]
    wss = [make_ws(x) for x in inps]
    streams = [torch.cuda.Stream() for _ in cases]
    try:
        devs = [to_dev(x) for x in inps]
        outs = [(torch.empty_like(d["residual"]), torch.empty_like(d["residual"])) for d in devs]

        def call(i):
            with torch.cuda.stream(streams[i]):
                run_gpu(wss[i], devs[i], out=outs[i][0], residual_out=outs[i][1], stream=streams[i])

        torch.cuda.synchronize()
        for _ in range(10):           # one host thread, interleaved on two streams
            call(0)
            call(1)
        torch.cuda.synchronize()
        for i, (c, T) in enumerate(cases):
            check_bf16(outs[i][0], refs[i]["out"], f"interleaved {c} T={T} out")
            check_bf16(outs[i][1], refs[i]["h"], f"interleaved {c} T={T} residual_out")
            outs[i][0].zero_()
            outs[i][1].zero_()
        torch.cuda.synchronize()
        errors = []

        def worker(i):
            try:
                for _ in range(25):
                    call(i)
                streams[i].synchronize()
            except Exception as e:  # noqa: BLE001 -- reported by the main thread
                errors.append(e)

        threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        assert not errors, errors
        torch.cuda.synchronize()
        for i, (c, T) in enumerate(cases):
            check_bf16(outs[i][0], refs[i]["out"], f"threads {c} T={T} out")
            check_bf16(outs[i][1], refs[i]["h"], f"threads {c} T={T} residual_out")
            assert arf.ar_workspace_device_error(wss[i]) == 0
    finally:
        for ws in wss:
            ws.destroy()


def test_cuda_graph_capture_of_a_first_call_with_plan_switch():
    """The first call of a fresh shape captured straight into a CUDA graph,
    no warm-up call: its plan needs the device's occupancy queries (here the
    split kernel's switch to two copy rounds, R = 15, K = 10, H = 8192 -- a
    shape no other test plans), which must be legal during stream capture.
    Replays after overwriting the inputs meet the oracle."""
    R, K, H, T = 15, 10, 8192, 9
    cfg = Config("capture_first", 100, R=R, K=K, H=H, Ts=(T,), eps=1e-6, weights="softmax", has_shared=True)
    inp = make_inputs(cfg, T, seed=1)
    ws = arf.ar_workspace_create(R, K, H, T, 1e-6, device=0)
    try:
        arf.ar_workspace_set_cluster_size(ws, 16)
        d = to_dev(inp)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
        r_out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run_gpu(ws, d, regime=arf.AR_REGIME_SPLIT, out=out, residual_out=r_out)
        assert arf.ar_workspace_last_plan(ws)["copy_rounds"] == 2
        for seed in (2, 3):
            new = make_inputs(cfg, T, seed=seed)
            for key in ("E", "S"):
                for dst, src in zip(d[key], new[key]):
                    dst.copy_(src)
            for key in ("perm", "w", "residual", "gamma"):
                d[key].copy_(new[key])
            g.replay()
            torch.cuda.synchronize()
            ref = run_oracle(new)
            check_bf16(out, ref["out"], f"captured first call seed={seed} out")
            check_bf16(r_out, ref["h"], f"captured first call seed={seed} residual_out")
        del g
        assert arf.ar_workspace_device_error(ws) == 0
    finally:
        ws.destroy()


def test_pdl_chain_through_two_round_split_plans():
    """AR_WS_PDL with the split kernel in two copy rounds (the TP16 table at
    T = 9): calls launched back to back, each reading the previous call's
    residual_out, every step against the oracle."""
    R, K, H, T = 16, 10, 8192, 9
    cfg = Config("tp16", 97, R=R, K=K, H=H, Ts=(T,), eps=1e-6, weights="softmax", has_shared=True)
    inp = make_inputs(cfg, T)
    ws = arf.ar_workspace_create(R, K, H, T, inp["eps"], device=0, flags=arf.AR_WS_PDL)
    try:
        d = to_dev(inp)
        steps = 4
        res = [d["residual"].clone()] + [torch.empty_like(d["residual"]) for _ in range(steps)]
        outs = [torch.empty_like(d["residual"]) for _ in range(steps)]
        for n in range(steps):
            dn = dict(d)
            dn["residual"] = res[n]
            run_gpu(ws, dn, out=outs[n], residual_out=res[n + 1])
        torch.cuda.synchronize()
        plan = arf.ar_workspace_last_plan(ws)
        assert plan["regime"] == arf.AR_REGIME_SPLIT and plan["copy_rounds"] == 2
        assert arf.ar_workspace_device_error(ws) == 0
        for n in range(steps):
            step = dict(inp)
            step["residual"] = res[n].cpu()
            ref = run_oracle(step)
            check_bf16(outs[n], ref["out"], f"pdl two-round chain step {n} out")
            check_bf16(res[n + 1], ref["h"], f"pdl two-round chain step {n} residual_out")
    finally:
        ws.destroy()

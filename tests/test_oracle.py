"""Pins of the CPU fp64 oracle against facts fixed by the definition, the
mathematics and independent routines (no GPU).

The operator (sglang PR #37196 "[Comm] Share the CuTe DSL AR fusion core and
wire it for DeepSeek-V3 / GLM-5.x", Motivation and Modifications sections 1-2;
sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with final RMSNorm",
Changes):
    h   = sum_r (sum_k w[t,k] E_r[perm[t,k]] + S_r[t]) + residual[t]
    out = h / sqrt(mean(h^2) + eps) * (gamma + weight_bias)
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gen import bf16_bits, make_inputs, make_perm_decode_inputs
from oracle.brute import bf16_bits_to_float, brute_ar_finalize_rmsnorm
from tests._util import BF16_ATOL, BF16_RTOL, oracle_args, run_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_bf16_bits(rng, shape, sigma=1.0):
    x = torch.from_numpy((rng.standard_normal(shape) * sigma).astype(np.float32))
    return bf16_bits(x.to(torch.bfloat16))


def _small_problem(rng, T, H, K, R, shared=True, dup=False, rows_e=None):
    rows_e = rows_e or max(1, T * K)
    E = [_rand_bf16_bits(rng, (rows_e, H)) for _ in range(R)] if K else None
    if K:
        if dup:
            perm = rng.integers(0, rows_e, size=(T, K)).astype(np.int32)
        else:
            perm = rng.permutation(rows_e)[: T * K].reshape(T, K).astype(np.int32)
        w = rng.random((T, K)).astype(np.float32)
    else:
        perm = w = None
    S = [_rand_bf16_bits(rng, (T, H), 0.5) for _ in range(R)] if shared else None
    res = _rand_bf16_bits(rng, (T, H))
    gamma = bf16_bits(torch.from_numpy(rng.uniform(0.5, 1.5, H).astype(np.float32)).to(torch.bfloat16))
    return E, perm, w, S, res, gamma


# ---------------------------------------------------------------- I1 brute force
@pytest.mark.parametrize("R", [1, 2])
@pytest.mark.parametrize("K", [0, 1, 2])
@pytest.mark.parametrize("shared", [True, False])
@pytest.mark.parametrize("dup", [False, True])
def test_brute_force_2x4(R, K, shared, dup):
    if K == 0 and not shared:
        pytest.skip("nothing to reduce")
    rng = np.random.default_rng(1000 * R + 100 * K + 10 * shared + dup)
    E, perm, w, S, res, gamma = _small_problem(rng, 2, 4, K, R, shared, dup, rows_e=5 if K else None)
    for wb, eps in [(0.0, 1e-6), (0.25, 0.5)]:
        h_ex, out_ex = brute_ar_finalize_rmsnorm(E, perm, w, S, res, gamma, wb, eps)
        got = oracle.ar_finalize_rmsnorm_ref(E, perm, w, S, res, gamma, wb, eps, want_abs=True)
        for t in range(2):
            for j in range(4):
                assert abs(got["h"][t, j] - float(h_ex[t][j])) <= 1e-15 * got["abs"][t, j] + 1e-300
                assert math.isclose(got["out"][t, j], out_ex[t][j], rel_tol=1e-12, abs_tol=1e-300)


def test_brute_force_tiny_config():
    """Whole tiny config (T=4, H=256, K=2, R=2) against the exact rational sum."""
    inp = make_inputs("tiny", 4)
    a = oracle_args(inp)
    h_ex, out_ex = brute_ar_finalize_rmsnorm(a["E"], a["perm"], a["w"], a["S"], a["residual"],
                                             a["gamma"], a["weight_bias"], a["eps"])
    got = run_oracle(inp, want_abs=True)
    h_ex = np.array([[float(x) for x in row] for row in h_ex])
    assert np.all(np.abs(got["h"] - h_ex) <= 1e-15 * got["abs"])
    np.testing.assert_allclose(got["out"], np.array(out_ex), rtol=1e-12, atol=0)


# ------------------------------------------------------------ I2 exact sum (fsum)
@pytest.mark.parametrize("cfg,T", [("dsv3_decode", 2), ("glm_gemma", 1), ("prefill", 1), ("ar_only", 3)])
def test_residual_out_is_exact_sum(cfg, T):
    inp = make_inputs(cfg, T)
    a = oracle_args(inp)
    got = run_oracle(inp, want_abs=True)
    rng = np.random.default_rng(7)
    H, R, K = inp["H"], inp["R"], inp["K"]
    dec = lambda b: bf16_bits_to_float(int(b))
    for _ in range(64):
        t, j = int(rng.integers(T)), int(rng.integers(H))
        terms = []
        for r in range(R):
            for k in range(K):
                terms.append(float(a["w"][t, k]) * dec(a["E"][r][a["perm"][t, k], j]))
            terms.append(dec(a["S"][r][t, j]))
        terms.append(dec(a["residual"][t, j]))
        exact = math.fsum(terms)
        assert abs(got["h"][t, j] - exact) <= 2.0 ** -50 * got["abs"][t, j]


# ------------------------------------------------------------ I3 constant gamma
@pytest.mark.parametrize("c", [1.0, 0.5, -2.0])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.1])
def test_constant_gamma_rms(c, eps):
    inp = make_inputs("dsv3_decode", 3)
    inp["gamma"] = torch.full((inp["H"],), c, dtype=torch.bfloat16)
    inp["eps"] = eps
    got = run_oracle(inp)
    ms = np.mean(got["h"] ** 2, axis=1)
    rms_out = np.sqrt(np.mean(got["out"] ** 2, axis=1))
    np.testing.assert_allclose(rms_out, abs(c) * np.sqrt(ms / (ms + np.float32(eps))), rtol=1e-13)


# ------------------------------------------------------ I4 permutation invariance
def test_permutation_invariance():
    inp = make_inputs("dsv3_decode", 4)
    a = oracle_args(inp)
    base = run_oracle(inp)
    rng = np.random.default_rng(3)
    R, T, K = inp["R"], inp["T"], inp["K"]
    rank_p = rng.permutation(R)                     # relabel ranks
    slot_p = np.stack([rng.permutation(K) for _ in range(T)])   # per-token slot order
    sigma = rng.permutation(inp["rows_e"])          # move E rows: E'[sigma[i]] = E[i]
    E2 = []
    for r in rank_p:
        e = np.empty_like(a["E"][r])
        e[sigma] = a["E"][r]
        E2.append(e)
    perm2 = sigma[np.take_along_axis(a["perm"], slot_p, axis=1)].astype(np.int32)
    w2 = np.take_along_axis(a["w"], slot_p, axis=1)
    S2 = [a["S"][r] for r in rank_p]
    got = oracle.ar_finalize_rmsnorm_ref(E2, perm2, w2, S2, a["residual"], a["gamma"],
                                         a["weight_bias"], a["eps"], want_abs=True)
    assert np.all(np.abs(got["h"] - base["h"]) <= 1e-14 * got["abs"])
    np.testing.assert_allclose(got["out"], base["out"], rtol=1e-12, atol=1e-13)


# -------------------------------------------- I5 reduces to plain residual RMSNorm
def test_reduces_to_plain_rms_norm():
    """R=1, K=1, w=1, S absent: out = rms_norm(E[perm] + residual) (torch, fp64)."""
    rng = np.random.default_rng(5)
    T, H = 6, 512
    E, perm, _, _, res, gamma = _small_problem(rng, T, H, 1, 1, shared=False)
    w = np.ones((T, 1), np.float32)
    eps = 1e-5
    got = oracle.ar_finalize_rmsnorm_ref(E, perm, w, None, res, gamma, 0.0, eps)
    to64 = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double()
    x = to64(E[0])[torch.from_numpy(perm[:, 0].astype(np.int64))] + to64(res)
    want = torch.nn.functional.rms_norm(x, (H,), weight=to64(gamma), eps=eps)
    np.testing.assert_allclose(got["h"], x.numpy(), rtol=0, atol=0)
    np.testing.assert_allclose(got["out"], want.numpy(), rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------ I6 Gemma equivalence
def test_gemma_weight_bias_equivalence():
    """(gamma_ckpt, weight_bias=1) == (gamma_ckpt + 1, weight_bias=0) exactly."""
    inp = make_inputs("glm_gemma", 2)
    g = torch.rand((inp["H"],), generator=torch.Generator().manual_seed(9)) + 1.0
    g_plus = g.to(torch.bfloat16)                   # in [1, 2]
    g_ckpt = (g_plus.float() - 1.0).to(torch.bfloat16)  # exact: fewer bits needed
    assert torch.equal(g_ckpt.float() + 1.0, g_plus.float())
    inp["gamma"] = g_plus
    inp["weight_bias"] = 0.0
    a = run_oracle(inp)
    inp["gamma"] = g_ckpt
    inp["weight_bias"] = 1.0
    b = run_oracle(inp)
    assert np.array_equal(a["out"], b["out"])
    inp["weight_bias"] = 0.0                        # and the bias really enters
    c = run_oracle(inp)
    assert np.abs(c["out"] - a["out"]).max() > 0.1


# -------------------------------------------------------------- I7 exactly once
def test_shared_partial_counted_once_per_rank():
    """Replicating one S into all R ranks contributes R*S, not S."""
    rng = np.random.default_rng(11)
    T, H, R = 3, 64, 4
    s = _rand_bf16_bits(rng, (T, H))
    zeros = np.zeros((T, H), np.uint16)
    gamma = bf16_bits(torch.ones(H, dtype=torch.bfloat16))
    got = oracle.ar_rmsnorm_ref([s] * R, zeros, gamma, 0.0, 1e-6)
    sv = torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(got["h"], R * sv)


def test_ar_rmsnorm_is_finalize_with_k0():
    inp = make_inputs("ar_only", 5)
    a = oracle_args(inp)
    x = oracle.ar_rmsnorm_ref(a["S"], a["residual"], a["gamma"], 0.0, a["eps"])
    y = oracle.ar_finalize_rmsnorm_ref(None, None, None, a["S"], a["residual"], a["gamma"], 0.0, a["eps"])
    assert np.array_equal(x["h"], y["h"]) and np.array_equal(x["out"], y["out"])


def test_nothing_to_reduce_is_rejected():
    z = np.zeros((1, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.ar_finalize_rmsnorm_ref(None, None, None, None, z, z[0], 0.0, 1e-6)


def test_perm_out_of_range_is_rejected():
    rng = np.random.default_rng(2)
    E, perm, w, S, res, gamma = _small_problem(rng, 2, 8, 2, 1)
    perm[1, 1] = 4
    with pytest.raises(IndexError):
        oracle.ar_finalize_rmsnorm_ref(E, perm, w, S, res, gamma, 0.0, 1e-6)


# --------------------------------------------------------------------- I8 scale
@pytest.mark.parametrize("m", [-3, 4])
def test_power_of_two_scaling(m):
    inp = make_inputs("glm_gemma", 2)
    inp["eps"] = 0.0
    base = run_oracle(inp)
    f = 2.0 ** m
    sc = lambda t: (t.float() * f).to(torch.bfloat16)   # exact for these magnitudes
    inp2 = dict(inp, E=[sc(e) for e in inp["E"]], S=[sc(s) for s in inp["S"]],
                residual=sc(inp["residual"]))
    got = run_oracle(inp2)
    assert np.array_equal(got["h"], f * base["h"])
    np.testing.assert_allclose(got["out"], base["out"], rtol=1e-14, atol=0)


def test_zero_row_gives_zero_output():
    inp = make_inputs("tiny", 4)
    for e in inp["E"]:
        e[inp["perm"][2].long()] = 0
    for s in inp["S"]:
        s[2] = 0
    inp["residual"][2] = 0
    got = run_oracle(inp)
    assert np.all(got["h"][2] == 0) and np.all(got["out"][2] == 0)
    assert np.any(got["out"][1] != 0)


# ---------------------------------------------------------------- I9 perm decode
@pytest.mark.parametrize("R,K,H,T", [(2, 2, 256, 4), (8, 8, 64, 16), (8, 10, 96, 40), (3, 5, 64, 1)])
def test_perm_decode_exact(R, K, H, T):
    for shift in range(K):
        inp = make_perm_decode_inputs(R, K, H, T, hot_shift=shift, seed=shift)
        got = run_oracle(inp)
        D = inp["digits"]
        h = got["h"]
        assert np.array_equal(h, np.round(h))
        cols = np.arange(H)
        weights = 16 ** (cols % D)
        want = inp["perm"].numpy()[np.arange(T), inp["hot"].numpy()].astype(np.int64)
        for t in range(T):
            # every column holds one digit of the gathered row index
            digits = h[t].astype(np.int64)
            for d in range(D):
                assert np.all(digits[cols % D == d] == (want[t] >> (4 * d)) & 15)
            assert int((digits[:D] * weights[:D]).sum()) == want[t]


# --------------------------------------------------------- bf16 rounding helper
def test_round_bf16_matches_fp32_to_bf16_for_fp32_values():
    """For binary32-exact inputs the one-step rounding equals torch's fp32->bf16
    conversion (round to nearest even), including ties and subnormals."""
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # add exact ties between neighbouring bf16 values and subnormals
    ties = (np.arange(1, 5000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([1e-40, -3e-39, 3.3895e38, 65504.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    got = oracle.round_bf16(x.astype(np.float64))
    assert np.array_equal(np.isinf(got), np.isinf(want))
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin])


def test_round_bf16_is_single_rounding():
    """A binary64 value just above a bf16 tie must round up, though its binary32
    rounding lands exactly on the tie (which would then round to even, down)."""
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40       # halfway between 1 and 1+2^-7, plus a hair
    assert float(np.float32(x)) == 1.0 + 2.0 ** -8
    assert oracle.round_bf16(np.array([x]))[0] == 1.0 + 2.0 ** -7


# ------------------------------------------------------ the bf16-h reading stays in tolerance
def test_h_rounded_before_norm_reading_is_within_tolerance():
    inp = make_inputs("dsv3_decode", 4)
    a = run_oracle(inp)
    b = run_oracle(inp, h_bf16_before_norm=True)
    o = oracle.round_bf16(a["out"])
    assert np.all(np.abs(oracle.round_bf16(b["out"]) - o) <= BF16_ATOL + BF16_RTOL * np.abs(o))
    assert not np.array_equal(a["out"], b["out"])


# ------------------------------------------------------------- golden fixture
def test_page_tolerance_fixture():
    """The pages' reported fused-vs-split difference passes the stated check."""
    with open(os.path.join(GOLDEN, "p2_correctness_tolerance.json")) as f:
        g = json.load(f)
    d, rtol, atol = g["max_abs_diff"], g["rtol"], g["atol"]
    # one bf16 ulp in [2, 4) is exactly the reported difference ...
    assert d == 2.0 ** (1 - 7)
    # ... and it passes allclose for every magnitude in [2, 4) and above
    for v in (2.0, 3.99, 100.0):
        assert d <= atol + rtol * v
    assert (rtol, atol) == (BF16_RTOL, BF16_ATOL)


# ------------------------------------------------ gated shared expert (Qwen-style)
# PR #37196 "[Comm] Share the CuTe DSL AR fusion core ...", Modifications
# section 2: the Qwen-style shared expert carries a per-token sigmoid gate,
# applied to the shared output before the fused add.
@pytest.mark.parametrize("R,K", [(1, 1), (2, 2), (2, 0)])
def test_gated_brute_force_2x4(R, K):
    rng = np.random.default_rng(77 + R + 10 * K)
    E, perm, w, S, res, gamma = _small_problem(rng, 2, 4, K, R, True, False, rows_e=5 if K else None)
    gate = rng.normal(0, 2, 2).astype(np.float32)
    h_ex, out_ex = brute_ar_finalize_rmsnorm(E, perm, w, S, res, gamma, 0.0, 1e-6, shared_gate=gate)
    got = oracle.ar_finalize_rmsnorm_ref(E, perm, w, S, res, gamma, 0.0, 1e-6, want_abs=True,
                                         shared_gate=gate)
    for t in range(2):
        for j in range(4):
            assert abs(got["h"][t, j] - float(h_ex[t][j])) <= 1e-14 * got["abs"][t, j] + 1e-300
            assert math.isclose(got["out"][t, j], out_ex[t][j], rel_tol=1e-12, abs_tol=1e-300)


def test_gate_limits_are_exact():
    """sigmoid(+50) == 1 and sigmoid(-800) == 0 in binary64; sigmoid(0) == 1/2."""
    inp = make_inputs("dsv3_decode", 3)
    a = oracle_args(inp)
    T = inp["T"]
    call = lambda S, gate: oracle.ar_finalize_rmsnorm_ref(a["E"], a["perm"], a["w"], S, a["residual"],
                                                          a["gamma"], 0.0, a["eps"], shared_gate=gate)
    plain = call(a["S"], None)
    no_shared = call(None, None)
    assert np.array_equal(call(a["S"], np.full(T, 50, np.float32))["h"], plain["h"])
    assert np.array_equal(call(a["S"], np.full(T, -800, np.float32))["h"], no_shared["h"])
    half_S = [bf16_bits((torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).float() * 0.5)
                        .to(torch.bfloat16)) for s in a["S"]]
    np.testing.assert_allclose(call(a["S"], np.zeros(T, np.float32))["h"], call(half_S, None)["h"],
                               rtol=0, atol=1e-12)


def test_gate_scales_only_the_shared_term():
    inp = make_inputs("glm_gemma", 4)
    a = oracle_args(inp)
    gate = np.array([-3.0, -0.5, 0.7, 4.0], np.float32)
    call = lambda S, g: oracle.ar_finalize_rmsnorm_ref(a["E"], a["perm"], a["w"], S, a["residual"],
                                                       a["gamma"], 0.0, a["eps"], shared_gate=g)["h"]
    base = call(None, None)
    full = call(a["S"], None)
    gated = call(a["S"], gate)
    sig = 1.0 / (1.0 + np.exp(-gate.astype(np.float64)))
    np.testing.assert_allclose(gated - base, sig[:, None] * (full - base), rtol=1e-12, atol=1e-12)


def test_gate_needs_a_shared_term():
    rng = np.random.default_rng(1)
    E, perm, w, S, res, gamma = _small_problem(rng, 2, 8, 2, 1)
    with pytest.raises(ValueError):
        oracle.ar_finalize_rmsnorm_ref(E, perm, w, None, res, gamma, 0.0, 1e-6,
                                       shared_gate=np.zeros(2, np.float32))

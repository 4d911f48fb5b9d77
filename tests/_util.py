"""Shared test helpers: marshal generator output for the oracle and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gen import bf16_bits

# Acceptance for bf16-stored results (out, bf16 residual_out): torch.allclose
# semantics with rtol = atol = 1e-2 against the oracle value rounded to bf16
# (sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with final
# RMSNorm", Correctness: BF16 allclose at rtol = atol = 1e-2).
BF16_RTOL = 1e-2
BF16_ATOL = 1e-2
# fp32 residual_out: 1e-5 relative, scaled by the condition of the sum
# (max(|o|, sum |terms|)), since plain relative error is unbounded under
# cancellation.
F32_REL = 1e-5


def oracle_args(inp):
    """numpy views of a gen.make_inputs() problem, in the oracle's argument order."""
    E = [bf16_bits(e) for e in inp["E"]] if inp["E"] is not None else None
    S = [bf16_bits(s) for s in inp["S"]] if inp["S"] is not None else None
    perm = inp["perm"].cpu().numpy() if inp["perm"] is not None else None
    w = inp["w"].cpu().numpy() if inp["w"] is not None else None
    return dict(E=E, perm=perm, w=w, S=S, residual=bf16_bits(inp["residual"]),
                gamma=bf16_bits(inp["gamma"]),
                weight_bias=float(np.float32(inp["weight_bias"])),
                eps=float(np.float32(inp["eps"])))


def run_oracle(inp, **kw):
    a = oracle_args(inp)
    return oracle.ar_finalize_rmsnorm_ref(a["E"], a["perm"], a["w"], a["S"], a["residual"],
                                          a["gamma"], a["weight_bias"], a["eps"], **kw)


def check_bf16(got: torch.Tensor, ref64: np.ndarray, what: str):
    """got (bf16 tensor) against the oracle's binary64 value rounded to bf16."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    o = oracle.round_bf16(ref64)
    err = np.abs(g - o)
    bound = BF16_ATOL + BF16_RTOL * np.abs(o)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside rtol=atol=1e-2; "
            f"first {idx.tolist()}: got {g[bad][:5]} want {o[bad][:5]}")
    return float(err.max()) if err.size else 0.0


def check_f32(got: torch.Tensor, ref64: np.ndarray, abs64: np.ndarray, what: str):
    """fp32 residual_out: |g - o| <= 1e-5 * max(|o|, sum|terms|)."""
    g = got.detach().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref64)
    bound = F32_REL * np.maximum(np.abs(ref64), abs64)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements beyond 1e-5 (condition-scaled); "
            f"first {idx.tolist()}: got {g[bad][:5]} want {ref64[bad][:5]}")
    big = np.abs(ref64) >= 1e-2
    return float((err[big] / np.abs(ref64[big])).max()) if big.any() else 0.0


def sample_rows(d, rows):
    """Compact CPU problem holding only the given token rows of a device problem
    (the gathered expert rows become a dense [len(rows)*K, H] block)."""
    dev = d["residual"].device
    idx = torch.as_tensor(rows, device=dev, dtype=torch.long)
    K = d["K"]
    comp = dict(R=d["R"], K=K, H=d["H"], T=len(rows), rows_e=len(rows) * K, eps=d["eps"],
                weight_bias=d["weight_bias"])
    if K > 0:
        gathered = d["perm"][idx].reshape(-1).long()
        comp["E"] = [e.index_select(0, gathered).cpu() for e in d["E"]]
        comp["perm"] = torch.arange(len(rows) * K, dtype=torch.int32).view(len(rows), K)
        comp["w"] = d["w"][idx].cpu()
    else:
        comp["E"], comp["perm"], comp["w"] = None, None, None
    comp["S"] = [s[idx].cpu() for s in d["S"]] if d["S"] is not None else None
    comp["residual"] = d["residual"][idx].cpu()
    comp["gamma"] = d["gamma"].cpu()
    return comp

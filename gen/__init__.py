"""Seeded synthetic inputs for the fused TP-reduce + MoE finalize + RMSNorm op.

This module only draws inputs.  It holds none of the operator's arithmetic and
is shared by the oracle tests, the GPU parity tests, ``bench.py`` and
``smoke()`` so that both sides read identical bytes.

Workloads (shapes follow the pages: hidden 7168 for the DeepSeek-V3 NextN
boundary in sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with
final RMSNorm", Performance; hidden 6144 for GLM-5.x and hidden 8192 with
top_k 10 for the GB300 routing profiles in sglang PR #37196 "[Comm] Share the
CuTe DSL AR fusion core ...", Known gaps):

=============  ==  ==  ====  =========================  ========================
name           R   K   H     T                          routing weights
=============  ==  ==  ====  =========================  ========================
tiny           2   2   256   4                          softmax over K
ar_only        2   0   7168  1,2,4,8,16,32,64,128        (none: partials only)
dsv3_decode    8   8   7168  1,4,16,64,128              top-8 of sigmoid over 256,
                                                        renormalised to sum 1
glm_gemma      8   8   6144  1,2,4,8,16                 softmax over 8
prefill        8   10  8192  512,2048,8192              softmax over 10
=============  ==  ==  ====  =========================  ========================

Value recipe: E_r ~ N(0,1), S_r ~ N(0, s_sigma) (0.5 for tiny, else 1),
residual ~ N(0,1), gamma ~ U(0.5, 1.5) (for glm_gemma this is the stored
checkpoint + 1 and weight_bias = 0), all drawn in fp32 and rounded to bf16
(round to nearest even); perm = a random permutation of the T*K expert-output
rows, shaped [T, K] token-major (or, optionally, the expert-sorted order a real
MoE permutation has).  Draw order: E_0..E_{R-1}, S_0..S_{R-1}, residual, gamma,
router logits, perm.  Seed = 1_000_003 * config_index + T unless given.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

__all__ = ["CONFIGS", "Config", "make_inputs", "make_perm_decode_inputs",
           "make_gate_logits", "make_mhc_inputs", "MHC_SHAPES", "mhc_problem_bytes",
           "bf16_bits", "problem_bytes"]


@dataclass(frozen=True)
class Config:
    name: str
    index: int
    R: int
    K: int
    H: int
    Ts: tuple
    eps: float
    weights: str            # "softmax" | "sigmoid_top_of_256" | "none"
    s_sigma: float = 1.0
    gemma: bool = False     # gamma is stored as checkpoint + 1
    has_shared: bool = True
    weight_bias: float = 0.0
    notes: str = field(default="", compare=False)


CONFIGS = {
    "tiny": Config("tiny", 0, R=2, K=2, H=256, Ts=(4,), eps=1e-6,
                   weights="softmax", s_sigma=0.5),
    "ar_only": Config("ar_only", 1, R=2, K=0, H=7168,
                      Ts=(1, 2, 4, 8, 16, 32, 64, 128), eps=1e-6, weights="none"),
    "dsv3_decode": Config("dsv3_decode", 2, R=8, K=8, H=7168,
                          Ts=(1, 4, 16, 64, 128), eps=1e-6,
                          weights="sigmoid_top_of_256"),
    "glm_gemma": Config("glm_gemma", 3, R=8, K=8, H=6144, Ts=(1, 2, 4, 8, 16),
                        eps=1e-5, weights="softmax", gemma=True),
    "prefill": Config("prefill", 4, R=8, K=10, H=8192, Ts=(512, 2048, 8192),
                      eps=1e-6, weights="softmax"),
}


def problem_bytes(R: int, K: int, H: int, T: int, residual_out_fp32: bool = False) -> int:
    """Algorithmic HBM bytes of one call: every input byte read once and every
    output byte written once (routing metadata and gamma excluded)."""
    b = R * T * K * H * 2 + R * T * H * 2 + 3 * T * H * 2
    if residual_out_fp32:
        b += T * H * 2
    return b


def bf16_bits(t: torch.Tensor):
    """CPU numpy uint16 view of the raw bits of a bf16 tensor (copied to host)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal_bf16(shape, sigma, g, device, chunk_rows=8192):
    """N(0, sigma) in fp32 rounded to bf16, drawn in row chunks to bound the
    fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    rows = shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(sigma)
        out[r0:r1].copy_(x)
    return out


def _routing(cfg: Config, T: int, g, device):
    """Routing weights [T, K] fp32 and the chosen expert ids [T, K]."""
    K = cfg.K
    if cfg.weights == "sigmoid_top_of_256":
        logits = torch.randn((T, 256), generator=g, device=device)
        scores = torch.sigmoid(logits)
        top, ids = torch.topk(scores, K, dim=1)
        w = top / top.sum(dim=1, keepdim=True)
    elif cfg.weights == "softmax":
        logits = torch.randn((T, K), generator=g, device=device)
        w = torch.softmax(logits, dim=1)
        ids = torch.argsort(torch.rand((T, 256), generator=g, device=device), dim=1)[:, :K]
    else:
        raise ValueError(cfg.weights)
    return w.to(torch.float32).contiguous(), ids


def make_inputs(cfg, T: int, seed: int | None = None, device="cpu",
                perm_kind: str = "random", shared: bool | None = None, perm_blocks: int = 1):
    """Draw one problem of config ``cfg`` (a Config or its name) with T tokens.

    Returns a dict: R, K, H, T, rows_e, eps, weight_bias, E (list of R bf16
    [T*K, H] or None), perm (int32 [T, K] or None), w (fp32 [T, K] or None),
    S (list of R bf16 [T, H] or None), residual (bf16 [T, H]), gamma (bf16 [H]).

    perm_blocks = n > 1 draws the T rows as n equal blocks, each gathering only
    from its own contiguous block of T*K/n expert rows -- n independent
    problems packed in one buffer, as n successive layers' expert outputs would
    be (perm_kind "random": a random permutation within each block;
    "expert_sorted": the slots of each block stably sorted by expert id).
    """
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    R, K, H = cfg.R, cfg.K, cfg.H
    if seed is None:
        seed = 1_000_003 * cfg.index + T
    g = _gen(seed, device)
    rows_e = T * K
    E = [_normal_bf16((rows_e, H), 1.0, g, device) for _ in range(R)] if K > 0 else None
    use_s = cfg.has_shared if shared is None else shared
    if K == 0:
        use_s = True
    S = [_normal_bf16((T, H), cfg.s_sigma, g, device) for _ in range(R)] if use_s else None
    residual = _normal_bf16((T, H), 1.0, g, device)
    gamma = (torch.rand((H,), generator=g, device=device) + 0.5).to(torch.bfloat16)
    perm = w = None
    if K > 0:
        w, ids = _routing(cfg, T, g, device)
        if perm_kind == "random" and perm_blocks > 1:
            if T % perm_blocks:
                raise ValueError("T must be a multiple of perm_blocks")
            blk = rows_e // perm_blocks
            keys = torch.rand((perm_blocks, blk), generator=g, device=device)
            local = torch.argsort(keys, dim=1)
            base = torch.arange(perm_blocks, device=device).view(-1, 1) * blk
            perm = (local + base).to(torch.int32).view(T, K)
        elif perm_kind == "random":
            perm = torch.randperm(rows_e, generator=g, device=device).to(torch.int32).view(T, K)
        elif perm_kind == "expert_sorted":
            # position of slot (t, k) after a stable sort of the slots by
            # expert id, within each of perm_blocks blocks of tokens
            if T % perm_blocks:
                raise ValueError("T must be a multiple of perm_blocks")
            blk = rows_e // perm_blocks
            order = torch.sort(ids.reshape(perm_blocks, blk), dim=1, stable=True).indices
            base = torch.arange(perm_blocks, device=device).view(-1, 1) * blk
            perm = torch.empty(rows_e, dtype=torch.int32, device=device)
            perm[(order + base).reshape(-1)] = (torch.arange(blk, device=device).view(1, -1) + base).reshape(-1).to(torch.int32)
            perm = perm.view(T, K)
        else:
            raise ValueError(perm_kind)
        perm = perm.contiguous()
    return dict(cfg=cfg, R=R, K=K, H=H, T=T, rows_e=rows_e, eps=cfg.eps,
                weight_bias=cfg.weight_bias, E=E, perm=perm, w=w, S=S,
                residual=residual, gamma=gamma)


def make_gate_logits(T: int, seed: int = 4242, device="cpu", sigma: float = 2.0):
    """Shared-expert gate logits, fp32 [T] ~ N(0, sigma) (sigmoid spans ~0.02..0.98)."""
    g = _gen(seed, device)
    return (torch.randn((T,), generator=g, device=device) * sigma).contiguous()


def hex_digits_needed(rows: int) -> int:
    n = 1
    while 16 ** n < rows:
        n += 1
    return n


def make_perm_decode_inputs(R: int, K: int, H: int, T: int, hot_shift: int = 0,
                            seed: int = 12345, device="cpu", rows_e: int | None = None):
    """Inputs whose routed sum spells out the gathered row index.

    E_r[i, c] holds hex digit (c mod D) of i when (c // D) mod R == r, else 0,
    with D = hex digits needed for rows_e; every value is a small integer, exact
    in bf16.  w is one-hot per token, hot slot k* = (t + hot_shift) mod K; S = 0,
    residual = 0, gamma = 1.  Then residual_out[t, c] must equal hex digit
    (c mod D) of perm[t, k*] exactly.  perm is a seeded random permutation.
    """
    if rows_e is None:
        rows_e = T * K
    D = hex_digits_needed(rows_e)
    if H < D * R:
        raise ValueError("H too small to hold every rank's digits")
    g = _gen(seed, device)
    i = torch.arange(rows_e, device=device, dtype=torch.int64).view(-1, 1)
    c = torch.arange(H, device=device, dtype=torch.int64).view(1, -1)
    digit = (i >> (4 * (c % D))) & 15                     # [rows_e, H]
    owner = (c // D) % R                                  # [1, H]
    E = [torch.where(owner == r, digit, torch.zeros_like(digit)).to(torch.bfloat16)
         for r in range(R)]
    del digit
    perm = torch.randperm(rows_e, generator=g, device=device)[: T * K]
    perm = perm.to(torch.int32).view(T, K).contiguous()
    hot = (torch.arange(T, device=device) + hot_shift) % K
    w = torch.zeros((T, K), dtype=torch.float32, device=device)
    w[torch.arange(T, device=device), hot] = 1.0
    S = [torch.zeros((T, H), dtype=torch.bfloat16, device=device) for _ in range(R)]
    residual = torch.zeros((T, H), dtype=torch.bfloat16, device=device)
    gamma = torch.ones((H,), dtype=torch.bfloat16, device=device)
    return dict(R=R, K=K, H=H, T=T, rows_e=rows_e, eps=1e-6, weight_bias=0.0,
                E=E, perm=perm, w=w, S=S, residual=residual, gamma=gamma,
                hot=hot, digits=D)


# All-reduce + mHC residual write-back (hc_post): four residual streams, at
# most 16 tokens in serving (sglang PR #42020, Summary and Scope; TP4 on the
# page's MI355X runs).  Hidden sizes: 5120 (the other fused all-reduce +
# hc_post the page mentions) and 6144 (GLM-5.x, sglang PR #37196, Known gaps).
MHC_SHAPES = {"mhc_h5120": dict(R=4, H=5120, hc=4, Ts=(1, 2, 4, 8, 16)),
              "mhc_h6144": dict(R=4, H=6144, hc=4, Ts=(1, 2, 4, 8, 16))}


def mhc_problem_bytes(R: int, H: int, hc: int, T: int) -> int:
    """Algorithmic HBM bytes of one all-reduce + hc_post call: R partials and hc
    streams read, hc streams written (bf16; post/comb coefficients excluded)."""
    return 2 * T * H * (R + 2 * hc)


def make_mhc_inputs(R: int, H: int, hc: int, T: int, seed: int = 777, device="cpu"):
    """Inputs for the all-reduce + mHC write-back.

    partials P_r ~ N(0,1) and incoming streams x ~ N(0,1), both fp32 rounded to
    bf16; post = 2*sigmoid(N(0,1)) in (0, 2); comb a doubly stochastic hc x hc
    matrix per token (positive entries exp(N(0,1)), rows and columns
    normalised alternately 20 times, in fp64, then fp32).  Draw order:
    P_0..P_{R-1}, x, post logits, comb logits.
    """
    g = _gen(seed, device)
    P = [_normal_bf16((T, H), 1.0, g, device) for _ in range(R)]
    x = _normal_bf16((T * hc, H), 1.0, g, device).view(T, hc, H)
    post = (2.0 * torch.sigmoid(torch.randn((T, hc), generator=g, device=device))).float()
    m = torch.exp(torch.randn((T, hc, hc), generator=g, device=device)).double()
    for _ in range(20):
        m = m / m.sum(dim=2, keepdim=True)
        m = m / m.sum(dim=1, keepdim=True)
    comb = m.float().contiguous()
    return dict(R=R, H=H, hc=hc, T=T, P=P, x=x.contiguous(), post=post.contiguous(), comb=comb)

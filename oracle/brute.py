"""Exact rational brute force of the fused boundary op (tiny inputs only).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Used to pin the C
oracle: every sum is carried out in ``fractions.Fraction`` with no rounding at
all; only the final square root is taken in binary64 on the exact mean.

Definition followed (sglang PR #37196 "[Comm] Share the CuTe DSL AR fusion
core ...", Motivation and Modifications sections 1-2; sglang PR #37104
"perf(mtp): fuse trailing TP all-reduce with final RMSNorm", Changes):

    y[t,j]   = sum_r ( sum_k w[t,k] E_r[perm[t,k], j] + S_r[t,j] )
    h[t,j]   = y[t,j] + residual[t,j]
    out[t,j] = h[t,j] / sqrt(mean_j h[t,j]^2 + eps) * (gamma[j] + weight_bias)
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction


def bf16_bits_to_float(b: int) -> float:
    """Decode one bf16 bit pattern (an int in [0, 65535])."""
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


def _fr_bf16(b) -> Fraction:
    return Fraction(bf16_bits_to_float(int(b)))


def brute_ar_finalize_rmsnorm(E, perm, w, S, residual, gamma, weight_bias, eps,
                              shared_gate=None):
    """Nested Python lists/arrays in, exact ``h`` (Fractions) and ``out`` (floats) out.

    E: list over r of [rows_e][H] bf16 bit patterns (or None when K == 0);
    perm, w: [T][K]; S: list over r of [T][H] bits, or None;
    residual: [T][H] bits; gamma: [H] bits; shared_gate: optional [T] gate
    logits -- the shared term of token t is scaled by sigmoid(gate[t]) (the
    sigmoid is taken in binary64, then used exactly).
    """
    T = len(residual)
    H = len(residual[0])
    K = len(perm[0]) if (E and len(perm) and len(perm[0])) else 0
    R = len(E) if E else len(S)
    wb = Fraction(float(weight_bias))
    ep = Fraction(float(eps))
    h = [[Fraction(0)] * H for _ in range(T)]
    out = [[0.0] * H for _ in range(T)]
    for t in range(T):
        g = Fraction(1)
        if shared_gate is not None:
            g = Fraction(1.0 / (1.0 + math.exp(-float(shared_gate[t]))))
        for j in range(H):
            y = Fraction(0)
            for r in range(R):
                for k in range(K):
                    y += Fraction(float(w[t][k])) * _fr_bf16(E[r][int(perm[t][k])][j])
                if S:
                    y += g * _fr_bf16(S[r][t][j])
            h[t][j] = y + _fr_bf16(residual[t][j])
        ms = sum(x * x for x in h[t]) / H
        root = math.sqrt(ms + ep)            # the one binary64 step
        for j in range(H):
            out[t][j] = float(h[t][j] * (_fr_bf16(gamma[j]) + wb)) / root
    return h, out


def brute_ar_mhc_post(partials, x, post, comb):
    """Exact (Fraction) all-reduce + mHC write-back on tiny inputs.

    partials: list over r of [T][H] bf16 bits; x: [T][hc][H] bits; post: [T][hc]
    floats; comb: [T][hc][hc] floats.  Returns out[t][i][j] as Fractions:
    post[t][i] * sum_r P_r[t][j] + sum_k comb[t][i][k] * x[t][k][j]
    (the reading of hc_post stated in ar_oracle.c; parity unpinned).
    """
    T = len(x)
    hc = len(x[0])
    H = len(x[0][0])
    out = [[[Fraction(0)] * H for _ in range(hc)] for _ in range(T)]
    for t in range(T):
        for j in range(H):
            y = sum((_fr_bf16(p[t][j]) for p in partials), Fraction(0))
            for i in range(hc):
                o = Fraction(float(post[t][i])) * y
                for k in range(hc):
                    o += Fraction(float(comb[t][i][k])) * _fr_bf16(x[t][k][j])
                out[t][i][j] = o
    return out

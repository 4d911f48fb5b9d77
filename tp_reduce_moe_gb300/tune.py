"""Regime crossover tuning for one problem shape (R, K, H).

The library has four launch regimes (whole-row streaming, tiled streaming over
a cluster, the one-shot cluster kernel, the split-segment cluster kernel) and
the best one depends on T and on the shape: the crossovers measured for one
hidden size do not carry over to another.  ``tune`` times every regime (and
every cluster size) through the public API on this GPU, L2-cold, at a ladder
of token counts, and reduces the winners to the rule table that
``ar_workspace_set_regime_table`` takes: ``[(max_tokens, regime,
ctas_per_row), ...]`` in ascending ``max_tokens``; a call with T tokens runs
the first rule with ``T <= max_tokens``.

Timing: a CUDA graph of one call per input set, replayed; the sets are
disjoint (each gathers only within its own block of expert rows) and together
hold at least 3x the L2 cache, so every call reads HBM.  Input values are
random (they do not affect the time); only their layout matters.

    python -m tp_reduce_moe_gb300.tune --R 8 --K 8 --H 7168
"""
from __future__ import annotations

import argparse
import json
import math
import statistics

import torch

from . import binding as arf

# Crossovers fall between powers of two (measured: four-CTA tiles at T = 72
# 11-15 % ahead of the plan that wins at T = 96), so the ladder is dense.
DEFAULT_TOKENS = (1, 2, 4, 6, 8, 10, 12, 14, 16, 20, 24, 28, 32, 36, 40, 44, 48, 56, 64, 72, 80, 96, 112, 128,
                  160, 192, 224, 256)
# A measured winner replaces the running rule only when it beats the running
# rule's own time at that T by more than this fraction (run-to-run noise is
# about 1 %), so near-equal plans do not split the table into many rules.
SWITCH_MARGIN = 0.015
REGIME_NAME = {arf.AR_REGIME_AUTO: "auto", arf.AR_REGIME_CLUSTER: "cluster",
               arf.AR_REGIME_STREAM: "stream", arf.AR_REGIME_ONESHOT: "oneshot",
               arf.AR_REGIME_SPLIT: "split"}


def candidates():
    """Every (regime, ctas_per_row, stage_bytes, producer_warps) timed; 0 = the
    library's own choice.  The streaming kernels also run with 24 KB ring
    slots and two producer warps: fewer, smaller slots and fewer threads let
    more CTAs of a clustered plan reside per SM, which wins at some T.  The
    one-shot kernel also runs with every cluster size: smaller clusters
    launch and exchange sooner than the CTA count its plan aims for."""
    out = [(arf.AR_REGIME_STREAM, 0, 0, 0), (arf.AR_REGIME_STREAM, 0, 0, 2), (arf.AR_REGIME_ONESHOT, 0, 0, 0)]
    out += [(arf.AR_REGIME_ONESHOT, c, 0, 0) for c in (2, 4, 8, 16)]
    for c in (2, 4, 8, 16):
        out += [(arf.AR_REGIME_CLUSTER, c, 0, 0), (arf.AR_REGIME_CLUSTER, c, 24576, 2)]
        if c in (4, 8):  # mid-size slots: two CTAs per SM with deeper rings than 24 KB slots
            out += [(arf.AR_REGIME_CLUSTER, c, 32768, 2), (arf.AR_REGIME_CLUSTER, c, 49152, 3)]
    # the split kernel also in twelve-CTA clusters (four groups of three): one
    # CTA per SM for more rows than sixteen-CTA clusters allow at T = 8-16
    out += [(arf.AR_REGIME_SPLIT, c, 0, 0) for c in (2, 4, 8, 12, 16)]
    return out


def problem_bytes(R: int, K: int, H: int, T: int, shared: bool = True) -> int:
    """Algorithmic HBM bytes of one call with bf16 residual_out."""
    return 2 * T * H * (R * K + (R if shared else 0) + 3)


class _Inputs:
    """n_sets disjoint input sets for T tokens, on `dev`."""

    def __init__(self, R, K, H, T, shared, n_sets, dev, seed=0):
        g = torch.Generator(device=dev).manual_seed(seed)
        self.T, self.n = T, n_sets
        rows = T * n_sets
        bf = torch.bfloat16

        def randn(*shape):
            return torch.randn(*shape, generator=g, device=dev).to(bf)

        self.E = [randn(rows * K, H) for _ in range(R)] if K else None
        if K:
            blocks = [torch.randperm(T * K, generator=g, device=dev) + i * T * K for i in range(n_sets)]
            self.perm = torch.cat(blocks).view(rows, K).to(torch.int32)
            self.w = torch.rand(rows, K, generator=g, device=dev)
        self.S = [randn(rows, H) for _ in range(R)] if shared else None
        self.residual = randn(rows, H)
        self.gamma = (torch.rand(H, generator=g, device=dev) + 0.5).to(bf)
        self.out = torch.empty(n_sets, T, H, dtype=bf, device=dev)
        self.rout = torch.empty(n_sets, T, H, dtype=bf, device=dev)
        self.rows_e = rows * K

    def call(self, ws, i, eps, stream):
        sl = slice(i * self.T, (i + 1) * self.T)
        S = [x[sl] for x in self.S] if self.S is not None else None
        if self.E is None:
            arf.ar_rmsnorm(ws, S, self.residual[sl], self.gamma, 0.0, eps, out=self.out[i],
                           residual_out=self.rout[i], stream=stream)
        else:
            arf.ar_finalize_rmsnorm(ws, self.E, self.perm[sl], self.w[sl], S, self.residual[sl],
                                    self.gamma, 0.0, eps, out=self.out[i], residual_out=self.rout[i],
                                    stream=stream, rows_e=self.rows_e)


def time_regime(ws, inp: _Inputs, eps: float, regime: int, ctas: int, dev, reps: int = 3,
                stage_bytes: int = 0, producer_warps: int = 0):
    """Median µs per call of one forced (regime, ctas_per_row, stage_bytes,
    producer_warps), or None when the library has no plan for it.  Returns
    (us, regime_run, ctas_run, plan_run) -- plan_run the nonzero fields of
    the launch plan (ar_workspace_last_plan)."""
    arf.ar_workspace_set_regime(ws, regime)
    arf.ar_workspace_set_cluster_size(ws, ctas)
    arf.ar_workspace_set_stage_bytes(ws, stage_bytes)
    arf.ar_workspace_set_producer_warps(ws, producer_warps)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    try:
        with torch.cuda.stream(side):
            for i in range(min(inp.n, 4)):
                inp.call(ws, i, eps, side)
    except arf.ArfuseError as e:
        if e.status == arf.AR_ERR_UNSUPPORTED:
            return None, regime, ctas, {}
        raise
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    ran = arf.ar_workspace_last_regime(ws)
    plan = {k: v for k, v in arf.ar_workspace_last_plan(ws).items() if v and k not in ("regime", "ctas_per_row")}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream(dev)
        for i in range(inp.n):
            inp.call(ws, i, eps, cs)
    g.replay()
    torch.cuda.synchronize(dev)
    per = []
    st = torch.cuda.current_stream(dev)
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        g.replay()
        b.record(st)
        torch.cuda.synchronize(dev)
        per.append(a.elapsed_time(b) * 1e3 / inp.n)
    del g
    return statistics.median(per), ran[0], ran[1], plan


def arf_regime(name: str) -> int:
    return {v: k for k, v in REGIME_NAME.items()}[name]


def tune(R: int, K: int, H: int, tokens=DEFAULT_TOKENS, shared: bool = True, eps: float = 1e-6,
         device: int = 0, cands=None, log=None, margin: float = SWITCH_MARGIN, pdl: bool = False):
    """Time every candidate at every T; returns (rules, points).

    rules: [(max_tokens, regime, ctas_per_row, stage_bytes, producer_warps)]:
    the fastest candidate at each T, except that the running rule is kept
    while it is within `margin` of the fastest, consecutive equal choices
    merged; points: one dict per (T, candidate) with the measured µs.
    pdl: the calls launch with programmatic dependent launch (back to back in
    the timed graph, so a call's start-up overlaps the previous call).
    """
    dev = torch.device("cuda", device)
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    cands = list(cands or candidates())
    points, winners = [], []
    for T in sorted(set(int(t) for t in tokens)):
        n_sets = int(min(4096, max(2, math.ceil(3 * l2 / problem_bytes(R, K, H, T, shared)))))
        inp = _Inputs(R, K, H, T, shared, n_sets, dev)
        ws = arf.ar_workspace_create(R, K, H, T, eps, device=device, flags=arf.AR_WS_PDL if pdl else 0)
        best = None
        for regime, ctas, sb, pw in cands:
            us, ran_regime, ran_ctas, plan = time_regime(ws, inp, eps, regime, ctas, dev, stage_bytes=sb,
                                                         producer_warps=pw)
            pt = {"T": T, "regime": REGIME_NAME[regime], "ctas_per_row": ctas, "stage_bytes": sb,
                  "producer_warps": pw, "us": us, "ran": [REGIME_NAME.get(ran_regime, "?"), ran_ctas],
                  "plan": plan}
            points.append(pt)
            if log:
                log(pt)
            if us is not None and (best is None or us < best[0]):
                best = (us, regime, ctas, sb, pw)
        ws.destroy()
        del inp
        torch.cuda.empty_cache()
        if best is not None:
            if winners:
                keep = winners[-1][1:]
                kept = [pt["us"] for pt in points
                        if pt["T"] == T and pt["us"] is not None and
                        (arf_regime(pt["regime"]), pt["ctas_per_row"], pt["stage_bytes"], pt["producer_warps"]) == keep]
                if kept and kept[0] <= best[0] * (1.0 + margin):
                    best = (kept[0],) + keep
            winners.append((T,) + best[1:])
    rules = []
    for w in winners:
        if rules and rules[-1][1:] == w[1:]:
            rules[-1] = w
        else:
            rules.append(w)
    return rules, points


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--R", type=int, required=True)
    p.add_argument("--K", type=int, required=True)
    p.add_argument("--H", type=int, required=True)
    p.add_argument("--tokens", default=",".join(str(t) for t in DEFAULT_TOKENS))
    p.add_argument("--no-shared", action="store_true", help="no shared-expert partials (K > 0 only)")
    p.add_argument("--eps", type=float, default=1e-6)
    p.add_argument("--device", type=int, default=0)
    p.add_argument("--margin", type=float, default=SWITCH_MARGIN,
                   help="keep the running rule while within this fraction of the fastest")
    p.add_argument("--pdl", action="store_true",
                   help="time calls launched with programmatic dependent launch (AR_WS_PDL), for a "
                        "table that such workspaces use")
    args = p.parse_args(argv)
    shared = not args.no_shared or args.K == 0
    rules, points = tune(args.R, args.K, args.H, [int(t) for t in args.tokens.split(",")],
                         shared=shared, eps=args.eps, device=args.device, margin=args.margin, pdl=args.pdl)
    print(json.dumps({"R": args.R, "K": args.K, "H": args.H, "shared": shared, "pdl": args.pdl,
                      "device": torch.cuda.get_device_name(args.device),
                      "rules": [[t, REGIME_NAME[r], c, sb, pw] for t, r, c, sb, pw in rules],
                      "points": points}))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())

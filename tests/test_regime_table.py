"""Host-side tests of the regime table (no GPU needed).

A dry-run workspace plans every call and records the regime it would launch
(ar_workspace_last_regime) without touching a device, so the table's lookup,
its precedence rules and its fallback to the heuristic can be checked here;
every regime meets the oracle tolerances, which the GPU parity tests check
for each regime and for calls routed by a table.
"""
import pytest

import tp_reduce_moe_gb300 as arf

SPACING = 1 << 28          # fake device addresses, far apart, 16-byte aligned
BASE = 1 << 44
EPS = 1e-6


class Shape:
    def __init__(self, R, K, H, max_tokens=512):
        self.R, self.K, self.H = R, K, H
        self.ws = arf.ar_workspace_create(R, K, H, max_tokens, EPS, flags=arf.AR_WS_DRY_RUN)
        a = iter(range(BASE, BASE + 64 * SPACING, SPACING))
        self.E = [next(a) for _ in range(R)]
        self.S = [next(a) for _ in range(R)]
        self.perm, self.w, self.res, self.gamma, self.out, self.rout = (next(a) for _ in range(6))

    def plan(self, T):
        """Validate a call with T tokens; returns (regime, ctas) it would launch."""
        if self.K == 0:
            arf.ar_rmsnorm(self.ws, self.S, self.res, self.gamma, 0.0, EPS, out=self.out,
                           residual_out=self.rout, T=T)
        else:
            arf.ar_finalize_rmsnorm(self.ws, self.E, self.perm, self.w, self.S, self.res, self.gamma,
                                    0.0, EPS, out=self.out, residual_out=self.rout, rows_e=T * self.K,
                                    T=T)
        return arf.ar_workspace_last_regime(self.ws)


@pytest.fixture()
def dsv3():
    s = Shape(8, 8, 7168)
    yield s
    s.ws.destroy()


def test_builtin_table_is_installed_for_measured_shapes(dsv3):
    rules = arf.ar_workspace_get_regime_table(dsv3.ws)
    assert len(rules) >= 2
    assert [r[0] for r in rules] == sorted({r[0] for r in rules})
    other = Shape(3, 5, 1024)
    try:
        assert arf.ar_workspace_get_regime_table(other.ws) == []
    finally:
        other.ws.destroy()


def test_table_rules_are_followed(dsv3):
    arf.ar_workspace_set_regime_table(dsv3.ws, [
        (2, arf.AR_REGIME_SPLIT, 8),
        (40, arf.AR_REGIME_CLUSTER, 4),
        (100, arf.AR_REGIME_STREAM, 0),
    ])
    assert dsv3.plan(1) == (arf.AR_REGIME_SPLIT, 8)
    assert dsv3.plan(2) == (arf.AR_REGIME_SPLIT, 8)
    assert dsv3.plan(3) == (arf.AR_REGIME_CLUSTER, 4)
    assert dsv3.plan(40) == (arf.AR_REGIME_CLUSTER, 4)
    regime, grid = dsv3.plan(41)
    assert regime == arf.AR_REGIME_STREAM and grid == 41 * 3  # each row split over 152 // 41 CTAs


def test_past_the_last_rule_and_auto_rules_use_the_heuristic(dsv3):
    arf.ar_workspace_set_regime_table(dsv3.ws, [])
    heuristic = {T: dsv3.plan(T) for T in (1, 4, 16, 64, 300)}
    arf.ar_workspace_set_regime_table(dsv3.ws, [(8, arf.AR_REGIME_STREAM, 0),
                                                (32, arf.AR_REGIME_AUTO, 0)])
    assert dsv3.plan(4)[0] == arf.AR_REGIME_STREAM
    assert dsv3.plan(16) == heuristic[16]      # AUTO rule
    assert dsv3.plan(64) == heuristic[64]      # past the last rule
    assert dsv3.plan(300) == heuristic[300]


def test_rule_without_a_plan_falls_back(dsv3):
    arf.ar_workspace_set_regime_table(dsv3.ws, [])
    h1 = dsv3.plan(1)
    # 73 segments over a 2-CTA split cluster is 37 per CTA: beyond the split
    # kernel's 32 producer lanes in one round, and two rounds would buffer 21
    # whole 14 KB rows (301 KB of shared memory), so the rule has no plan
    arf.ar_workspace_set_regime_table(dsv3.ws, [(4, arf.AR_REGIME_SPLIT, 2)])
    assert dsv3.plan(1) == h1


def test_forced_regime_takes_precedence(dsv3):
    arf.ar_workspace_set_regime_table(dsv3.ws, [(512, arf.AR_REGIME_STREAM, 0)])
    arf.ar_workspace_set_regime(dsv3.ws, arf.AR_REGIME_CLUSTER)
    arf.ar_workspace_set_cluster_size(dsv3.ws, 8)
    assert dsv3.plan(4) == (arf.AR_REGIME_CLUSTER, 8)
    arf.ar_workspace_set_regime(dsv3.ws, arf.AR_REGIME_AUTO)
    assert dsv3.plan(4)[0] == arf.AR_REGIME_STREAM


@pytest.mark.parametrize("rules", [
    [(0, arf.AR_REGIME_STREAM, 0)],                                  # max_tokens < 1
    [(8, arf.AR_REGIME_STREAM, 0), (8, arf.AR_REGIME_SPLIT, 0)],     # not strictly ascending
    [(8, arf.AR_REGIME_STREAM, 0), (4, arf.AR_REGIME_SPLIT, 0)],
    [(8, 9, 0)],                                                     # unknown regime
    [(8, arf.AR_REGIME_STREAM, 4)],                                  # ctas for a regime without
    [(8, arf.AR_REGIME_ONESHOT, 17)],
    [(8, arf.AR_REGIME_CLUSTER, 1)],                                 # ctas out of range
    [(8, arf.AR_REGIME_SPLIT, 17)],
    [(t + 1, arf.AR_REGIME_STREAM, 0) for t in range(arf.AR_MAX_REGIME_RULES + 1)],  # too long
    [(8, arf.AR_REGIME_SPLIT, 16, 32768, 0)],                        # slot size for a regime without a ring
    [(8, arf.AR_REGIME_ONESHOT, 0, 0, 2)],                           # producer warps likewise
    [(8, arf.AR_REGIME_CLUSTER, 8, 512, 0)],                         # slot size out of range
    [(8, arf.AR_REGIME_STREAM, 0, 262144, 0)],
    [(8, arf.AR_REGIME_CLUSTER, 8, 0, 5)],                           # producer warps out of range
])
def test_invalid_tables_are_rejected_and_keep_the_old_one(dsv3, rules):
    before = arf.ar_workspace_get_regime_table(dsv3.ws)
    with pytest.raises(arf.ArfuseError) as e:
        arf.ar_workspace_set_regime_table(dsv3.ws, rules)
    assert e.value.status == arf.AR_ERR_INVALID_ARG
    assert arf.ar_workspace_get_regime_table(dsv3.ws) == before


def test_table_round_trip(dsv3):
    rules = [(t, arf.AR_REGIME_CLUSTER, 2 << (t % 4), 8192 * (t % 3), t % 5)
             for t in range(1, arf.AR_MAX_REGIME_RULES + 1)]
    arf.ar_workspace_set_regime_table(dsv3.ws, rules)
    assert arf.ar_workspace_get_regime_table(dsv3.ws) == rules
    # three-field rules: slot size and producer warps automatic
    arf.ar_workspace_set_regime_table(dsv3.ws, [(4, arf.AR_REGIME_SPLIT, 8)])
    assert arf.ar_workspace_get_regime_table(dsv3.ws) == [(4, arf.AR_REGIME_SPLIT, 8, 0, 0)]


def test_get_with_small_capacity(lib_handle=None):
    import ctypes
    s = Shape(8, 8, 7168)
    try:
        lib = arf.load_library()
        n = ctypes.c_int(-1)
        assert lib.ar_workspace_get_regime_table(ctypes.c_void_p(s.ws.handle), None, 0,
                                                 ctypes.byref(n)) == arf.AR_OK
        assert n.value == len(arf.ar_workspace_get_regime_table(s.ws))
        assert lib.ar_workspace_get_regime_table(None, None, 0, ctypes.byref(n)) == arf.AR_ERR_INVALID_ARG
        assert lib.ar_workspace_get_regime_table(ctypes.c_void_p(s.ws.handle), None, 1,
                                                 ctypes.byref(n)) == arf.AR_ERR_INVALID_ARG
        assert lib.ar_workspace_set_regime_table(ctypes.c_void_p(s.ws.handle), None, 1) == \
            arf.AR_ERR_INVALID_ARG
    finally:
        s.ws.destroy()


def test_k0_table_selects_oneshot_then_stream():
    """Two partials, K = 0: the one-shot kernel's 40-register variant up to
    T = 256 (the built-in table), whole-row streaming beyond (the heuristic
    past 1.5 rows per SM)."""
    s = Shape(2, 0, 7168)
    try:
        assert s.plan(8) == (arf.AR_REGIME_ONESHOT, 8)
        assert s.plan(128) == (arf.AR_REGIME_ONESHOT, 8)
        assert s.plan(160) == (arf.AR_REGIME_ONESHOT, 4)
        assert s.plan(200) == (arf.AR_REGIME_ONESHOT, 2)
        assert s.plan(256) == (arf.AR_REGIME_ONESHOT, 4)
        assert s.plan(300)[0] == arf.AR_REGIME_STREAM
    finally:
        s.ws.destroy()


def test_whole_row_streaming_splits_the_last_wave(dsv3):
    """The last partial wave's rows go to several CTAs each: the grid grows to
    cover the idle SMs (T < SMs: T * parts CTAs; T >= SMs: the SM count)."""
    arf.ar_workspace_set_regime(dsv3.ws, arf.AR_REGIME_STREAM)
    assert dsv3.plan(16) == (arf.AR_REGIME_STREAM, 16 * 8)    # 8 parts per row
    assert dsv3.plan(64) == (arf.AR_REGIME_STREAM, 128)       # 2 parts per row
    assert dsv3.plan(100) == (arf.AR_REGIME_STREAM, 100)      # 152 // 100 = 1: whole rows
    assert dsv3.plan(300) == (arf.AR_REGIME_STREAM, 152)
    arf.ar_workspace_set_split_rows(dsv3.ws, 0)
    assert dsv3.plan(16) == (arf.AR_REGIME_STREAM, 16)
    arf.ar_workspace_set_split_rows(dsv3.ws, 3)
    assert dsv3.plan(16) == (arf.AR_REGIME_STREAM, 48)


def test_light_rows_are_never_split():
    """Three segments per row (K = 0): a split part would hold a single segment."""
    s = Shape(2, 0, 7168)
    try:
        arf.ar_workspace_set_regime(s.ws, arf.AR_REGIME_STREAM)
        assert s.plan(1) == (arf.AR_REGIME_STREAM, 1)
        assert s.plan(192) == (arf.AR_REGIME_STREAM, 152)
    finally:
        s.ws.destroy()


def test_split_column_groups_need_two_ctas_per_group(dsv3):
    """Forced column groups must leave groups of at least two CTAs.  A
    group's share of the row's segments beyond the producer's 32 lanes is
    fetched in two copy rounds of at most 32 segments each (dsv3, 2 CTAs per
    group: 37 segments, 21 + 16); past that the forced split regime has no
    plan (R = 16, K = 10: 89 segments for each of 2 CTAs per group)."""
    arf.ar_workspace_set_regime(dsv3.ws, arf.AR_REGIME_SPLIT)
    arf.ar_workspace_set_cluster_size(dsv3.ws, 16)
    for groups in (0, 1, 2, 4, 8):
        arf.ar_workspace_set_split_column_groups(dsv3.ws, groups)
        assert dsv3.plan(4) == (arf.AR_REGIME_SPLIT, 16)
        assert arf.ar_workspace_last_grid(dsv3.ws) == 4 * 16
    arf.ar_workspace_set_cluster_size(dsv3.ws, 4)
    arf.ar_workspace_set_split_column_groups(dsv3.ws, 4)    # one CTA per group
    with pytest.raises(arf.ArfuseError) as e:
        dsv3.plan(1)
    assert e.value.status == arf.AR_ERR_UNSUPPORTED
    heavy = Shape(16, 10, 8192)
    try:
        arf.ar_workspace_set_regime(heavy.ws, arf.AR_REGIME_SPLIT)
        arf.ar_workspace_set_cluster_size(heavy.ws, 16)
        for groups in (0, 2, 4):        # one round (two groups) or two rounds (four)
            arf.ar_workspace_set_split_column_groups(heavy.ws, groups)
            assert heavy.plan(1) == (arf.AR_REGIME_SPLIT, 16)
        arf.ar_workspace_set_split_column_groups(heavy.ws, 8)
        with pytest.raises(arf.ArfuseError) as e:
            heavy.plan(1)
        assert e.value.status == arf.AR_ERR_UNSUPPORTED
    finally:
        heavy.ws.destroy()


def test_one_shot_cluster_size_from_a_rule_or_the_workspace():
    """The one-shot kernel takes a rule's (or the workspace's) cluster size
    when it is a power of two; another size has no one-shot plan: a forced
    regime declines the call, a table rule falls back to the heuristic."""
    s = Shape(2, 0, 7168)
    try:
        assert s.plan(8) == (arf.AR_REGIME_ONESHOT, 8)               # built-in table
        arf.ar_workspace_set_regime_table(s.ws, [(16, arf.AR_REGIME_ONESHOT, 4)])
        assert s.plan(8) == (arf.AR_REGIME_ONESHOT, 4)
        arf.ar_workspace_set_regime_table(s.ws, [(16, arf.AR_REGIME_ONESHOT, 6)])
        assert s.plan(8) == (arf.AR_REGIME_ONESHOT, 16)              # no plan for 6: the heuristic
        arf.ar_workspace_set_regime(s.ws, arf.AR_REGIME_ONESHOT)
        for c in (2, 4, 8, 16):
            arf.ar_workspace_set_cluster_size(s.ws, c)
            assert s.plan(8) == (arf.AR_REGIME_ONESHOT, c)
        arf.ar_workspace_set_cluster_size(s.ws, 6)
        with pytest.raises(arf.ArfuseError) as e:
            s.plan(8)
        assert e.value.status == arf.AR_ERR_UNSUPPORTED
    finally:
        s.ws.destroy()


def test_eight_partial_allreduce_table_runs_the_one_shot_kernel():
    s = Shape(8, 0, 7168)
    try:
        assert arf.ar_workspace_get_regime_table(s.ws) == [(96, arf.AR_REGIME_ONESHOT, 8, 0, 0),
                                                          (112, arf.AR_REGIME_ONESHOT, 2, 0, 0),
                                                          (256, arf.AR_REGIME_ONESHOT, 8, 0, 0)]
        for T in (1, 64, 128, 256):
            assert s.plan(T) == (arf.AR_REGIME_ONESHOT, 8)
        assert s.plan(100) == (arf.AR_REGIME_ONESHOT, 2)
        assert s.plan(300)[0] == arf.AR_REGIME_STREAM   # past the table: the heuristic
    finally:
        s.ws.destroy()


def test_rule_slot_size_and_producers_reach_the_plan(dsv3):
    """A rule's slot size and producer-warp cap give the same plan as the
    workspace-wide tuning controls with those values."""
    arf.ar_workspace_set_regime_table(dsv3.ws, [(64, arf.AR_REGIME_CLUSTER, 4, 24576, 2)])
    with_rule = dsv3.plan(48)
    arf.ar_workspace_set_regime_table(dsv3.ws, [])
    arf.ar_workspace_set_regime(dsv3.ws, arf.AR_REGIME_CLUSTER)
    arf.ar_workspace_set_cluster_size(dsv3.ws, 4)
    arf.ar_workspace_set_stage_bytes(dsv3.ws, 24576)
    arf.ar_workspace_set_producer_warps(dsv3.ws, 2)
    assert dsv3.plan(48) == with_rule == (arf.AR_REGIME_CLUSTER, 4)


@pytest.mark.parametrize("shape", [(8, 8, 7168), (4, 8, 7168), (8, 8, 6144), (8, 10, 8192), (16, 10, 8192),
                                   (2, 0, 7168), (8, 0, 7168)])
def test_every_builtin_rule_has_its_own_plan(shape):
    """Every rule of every built-in table plans its own regime (and cluster
    size, where it names one) at both ends of its token range on a GB300-sized
    dry-run workspace -- no rule silently falls back to the heuristic."""
    s = Shape(*shape, max_tokens=256)
    try:
        rules = arf.ar_workspace_get_regime_table(s.ws)
        assert rules, "a built-in table is expected for this shape"
        lo = 1
        for max_tokens, regime, ctas, _stage, _producers in rules:
            for T in (lo, max_tokens):
                got_regime, got_ctas = s.plan(T)
                assert got_regime == regime, (shape, T, rules)
                if ctas and regime != arf.AR_REGIME_STREAM:
                    assert got_ctas == ctas, (shape, T, rules)
            lo = max_tokens + 1
    finally:
        s.ws.destroy()


def test_last_grid_reports_the_planned_ctas(dsv3):
    """ar_workspace_last_grid: the CTAs of the last planned call -- T x C for
    the split and one-shot kernels, the persistent grid for streaming."""
    assert arf.ar_workspace_last_grid(dsv3.ws) == 0
    arf.ar_workspace_set_regime(dsv3.ws, arf.AR_REGIME_SPLIT)
    arf.ar_workspace_set_cluster_size(dsv3.ws, 16)
    assert dsv3.plan(4) == (arf.AR_REGIME_SPLIT, 16)
    assert arf.ar_workspace_last_grid(dsv3.ws) == 64
    arf.ar_workspace_set_regime(dsv3.ws, arf.AR_REGIME_STREAM)
    assert dsv3.plan(300) == (arf.AR_REGIME_STREAM, 152)
    assert arf.ar_workspace_last_grid(dsv3.ws) == 152
    arf.ar_workspace_set_regime(dsv3.ws, arf.AR_REGIME_CLUSTER)
    arf.ar_workspace_set_cluster_size(dsv3.ws, 4)
    regime, ctas = dsv3.plan(24)
    assert (regime, ctas) == (arf.AR_REGIME_CLUSTER, 4)
    assert arf.ar_workspace_last_grid(dsv3.ws) == 24 * 4      # one cluster per row when that fits


def test_last_plan_reports_the_launch_shape():
    """ar_workspace_last_plan: the plan of the last validated call -- split
    column groups and copy rounds, streaming ring slots and producer warps,
    one-shot loads per thread -- all zero before the first call."""
    d = Shape(8, 8, 7168)
    heavy = Shape(16, 10, 8192)
    k0 = Shape(2, 0, 7168)
    try:
        assert set(arf.ar_workspace_last_plan(d.ws).values()) == {0}
        d.plan(4)                                    # table: split, 16 CTAs, four groups
        p = arf.ar_workspace_last_plan(d.ws)
        assert (p["regime"], p["ctas_per_row"], p["grid"]) == (arf.AR_REGIME_SPLIT, 16, 64)
        assert (p["column_groups"], p["copy_rounds"], p["producer_warps"]) == (4, 1, 1)
        assert p["ring_slots"] == 0 and p["loads_per_thread"] == 0 and p["smem_bytes"] > 0
        d.plan(64)                                   # table: four-CTA tiles
        p = arf.ar_workspace_last_plan(d.ws)
        assert (p["regime"], p["ctas_per_row"], p["grid"]) == (arf.AR_REGIME_CLUSTER, 4, 256)
        assert p["ring_slots"] >= 2 and p["ring_slot_bytes"] > 0 and p["producer_warps"] >= 1
        assert p["column_groups"] == 0 and p["copy_rounds"] == 0
        assert p["grid"] == arf.ar_workspace_last_grid(d.ws)
        k0.plan(16)                                  # one-shot, two loads per thread
        p = arf.ar_workspace_last_plan(k0.ws)
        assert p["regime"] == arf.AR_REGIME_ONESHOT and p["loads_per_thread"] == 2
        assert p["block"] * p["ctas_per_row"] >= 7168 // 8
        # heavy rows: one round in two column groups, two rounds in four
        arf.ar_workspace_set_regime(heavy.ws, arf.AR_REGIME_SPLIT)
        arf.ar_workspace_set_cluster_size(heavy.ws, 16)
        heavy.plan(1)
        one = arf.ar_workspace_last_plan(heavy.ws)
        arf.ar_workspace_set_split_column_groups(heavy.ws, 4)
        heavy.plan(1)
        two = arf.ar_workspace_last_plan(heavy.ws)
        assert (one["column_groups"], one["copy_rounds"]) == (2, 1)
        assert (two["column_groups"], two["copy_rounds"]) == (4, 2)
        assert 2 * (two["smem_bytes"] + 1024) <= 233472 < 2 * (one["smem_bytes"] + 1024)  # two CTAs per SM
    finally:
        for x in (d, heavy, k0):
            x.ws.destroy()

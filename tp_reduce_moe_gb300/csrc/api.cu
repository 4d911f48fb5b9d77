// api.cu -- the C ABI of libarfuse (declared in include/arfuse.h): argument
// validation, the workspace, and the choice of kernel regime per call.
//
// Validation follows the pages' contract for the fused boundary: a residual is
// required and any decline must leave the caller free to run its own split
// path (sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with final
// RMSNorm", Changes); one workspace serves all layers of a model and is fixed
// per hidden / top_k / eps (sglang PR #37196 "[Comm] Share the CuTe DSL AR
// fusion core and wire it for DeepSeek-V3 / GLM-5.x", Modifications section
// 2).  Nothing here allocates or synchronises on the call path, so a call can
// be captured in a CUDA graph.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "arf_host.h"
#include "arfuse.h"

struct ar_workspace {
    int device;
    int R, K, H;
    int64_t max_tokens;
    float eps;
    unsigned flags;
    unsigned* d_err;  // device error word (AR_DEVERR_* bits)
    unsigned* d_part;  // split-row counters [num_sms] (zero between calls), then fp32 scratch [num_sms, H]
    bool split_ok;     // plans may split rows (the scratch exists, or a dry run plans as if it did)
    int max_tail_parts;  // cap on the segment intervals of a split row (0 / 1: never split)
    int num_sms;
    int smem_optin;
    int max_cluster;  // largest co-schedulable cluster for the cluster kernel
    int max_cluster_stream;  // largest cluster for the clustered streaming kernel
    int max_cluster_split;   // largest cluster for the split kernel
    int regime_force;
    int force_ctas_per_row;  // 0: automatic
    int stage_bytes;         // 0: automatic
    int producer_warps;      // 0: automatic
    int split_groups;        // column groups per row of the split kernel; 0: automatic
    int last_regime;
    int last_ctas;
    int last_grid;
    ar_plan_info last_plan;
    unsigned long long stall_wait_ns;  // failure injection (whole-row streaming), 0 = off
    int table_n;  // rules in `table` (0: heuristic only)
    ar_regime_rule table[AR_MAX_REGIME_RULES];
};

namespace {

constexpr int64_t kMaxTokensLimit = int64_t(1) << 26;
constexpr int kDryRunSms = 152;          // GB300
constexpr int kDryRunSmemOptin = 232448;  // 227 KB

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Split-row workspace: num_sms counters (rounded up to 256 bytes), then
// num_sms fp32 rows of H.
size_t part_counter_words(int num_sms) { return ((size_t)num_sms * 4 + 255) / 256 * 64; }
size_t part_bytes(int num_sms, int H) {
    return part_counter_words(num_sms) * 4 + (size_t)num_sms * H * 4;
}

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const void* p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// Regime tables measured on GB300 (tp_reduce_moe_gb300.tune: every regime,
// cluster size and ring variant, L2-cold, at 28 token counts from 1 to 256; a
// faster plan replaces the running rule only when it is more than 1.5 %
// ahead), installed for these shapes at create.
struct BuiltinTable {
    int R, K, H, n;
    ar_regime_rule rules[16];
};
// Rules: {max_tokens, regime, ctas_per_row, stage_bytes, producer_warps}.
// Clustered rules with smaller ring slots (24 KB and two producer warps,
// 32 KB and two, 48 KB and three) hold more CTAs per SM than the default plan
// (64 KB slots) and win where that plan would run more rows per cluster than
// needed (dsv3 T = 96 22.9 -> 20.5 us with eight-CTA tiles; H = 8192 K = 10
// T = 64 20.4 -> 18.8 us with four-CTA tiles and 48 KB slots).  Twelve-CTA
// split clusters (four groups of three CTAs) win where sixteen-CTA ones would
// leave most SMs with two CTAs.  The crossovers fall between powers of two:
// four-CTA tiles at T = 72 are 11-15 % ahead of the plan that wins at T = 96.
const BuiltinTable kBuiltinTables[] = {
    // DeepSeek-V3 decode, TP8 (H = 7168, top-8)
    {8, 8, 7168, 10,
     {{14, AR_REGIME_SPLIT, 16, 0, 0}, {20, AR_REGIME_SPLIT, 12, 0, 0}, {36, AR_REGIME_CLUSTER, 8, 0, 0},
      {48, AR_REGIME_CLUSTER, 8, 24576, 2}, {72, AR_REGIME_CLUSTER, 4, 0, 0}, {96, AR_REGIME_CLUSTER, 8, 24576, 2},
      {128, AR_REGIME_STREAM, 0, 0, 2}, {160, AR_REGIME_CLUSTER, 4, 24576, 2},
      {224, AR_REGIME_CLUSTER, 8, 24576, 2}, {256, AR_REGIME_STREAM, 0, 0, 2}}},
    // DeepSeek-V3 decode, TP4
    {4, 8, 7168, 9,
     {{6, AR_REGIME_SPLIT, 16, 0, 0}, {28, AR_REGIME_SPLIT, 8, 0, 0}, {48, AR_REGIME_CLUSTER, 8, 49152, 3},
      {72, AR_REGIME_CLUSTER, 4, 0, 0}, {96, AR_REGIME_CLUSTER, 4, 32768, 2}, {128, AR_REGIME_STREAM, 0, 0, 0},
      {192, AR_REGIME_CLUSTER, 4, 32768, 2}, {224, AR_REGIME_CLUSTER, 8, 24576, 2},
      {256, AR_REGIME_CLUSTER, 4, 0, 0}}},
    // GLM-style decode, TP8 (H = 6144, top-8)
    {8, 8, 6144, 11,
     {{20, AR_REGIME_SPLIT, 16, 0, 0}, {36, AR_REGIME_CLUSTER, 8, 0, 0}, {44, AR_REGIME_CLUSTER, 8, 24576, 2},
      {48, AR_REGIME_CLUSTER, 8, 32768, 2}, {72, AR_REGIME_CLUSTER, 4, 0, 0}, {80, AR_REGIME_CLUSTER, 4, 24576, 2},
      {96, AR_REGIME_CLUSTER, 8, 32768, 2}, {128, AR_REGIME_STREAM, 0, 0, 2},
      {160, AR_REGIME_CLUSTER, 4, 24576, 2}, {224, AR_REGIME_CLUSTER, 8, 24576, 2},
      {256, AR_REGIME_STREAM, 0, 0, 2}}},
    // H = 8192, top-10, TP8
    {8, 10, 8192, 13,
     {{6, AR_REGIME_SPLIT, 16, 0, 0}, {8, AR_REGIME_SPLIT, 12, 0, 0}, {14, AR_REGIME_SPLIT, 16, 0, 0},
      {20, AR_REGIME_CLUSTER, 16, 24576, 2}, {36, AR_REGIME_CLUSTER, 8, 0, 0},
      {48, AR_REGIME_CLUSTER, 8, 24576, 2}, {72, AR_REGIME_CLUSTER, 4, 49152, 3},
      {80, AR_REGIME_CLUSTER, 8, 24576, 2}, {96, AR_REGIME_CLUSTER, 8, 32768, 2},
      {128, AR_REGIME_CLUSTER, 4, 49152, 3}, {160, AR_REGIME_CLUSTER, 16, 0, 0},
      {224, AR_REGIME_CLUSTER, 8, 24576, 2}, {256, AR_REGIME_CLUSTER, 4, 49152, 3}}},
    // H = 8192, top-10, TP16 (with TP8 above, the GB300 routing profiles of sglang PR
    // #37196, Known gaps); from T = 8 the split kernel runs in two copy rounds
    {16, 10, 8192, 10,
     {{12, AR_REGIME_SPLIT, 16, 0, 0}, {20, AR_REGIME_CLUSTER, 16, 0, 0}, {36, AR_REGIME_CLUSTER, 8, 49152, 3},
      {48, AR_REGIME_CLUSTER, 8, 24576, 2}, {72, AR_REGIME_CLUSTER, 4, 24576, 2},
      {96, AR_REGIME_CLUSTER, 8, 24576, 2}, {128, AR_REGIME_STREAM, 0, 0, 0},
      {160, AR_REGIME_CLUSTER, 8, 49152, 3}, {224, AR_REGIME_CLUSTER, 8, 24576, 2},
      {256, AR_REGIME_STREAM, 0, 0, 0}}},
    // trailing all-reduce + RMSNorm, two partials (K = 0): the one-shot kernel in
    // smaller clusters than its plan's coverage rule picks (T = 160-256: wave
    // quantisation of the grid decides between four- and two-CTA clusters)
    {2, 0, 7168, 4,
     {{128, AR_REGIME_ONESHOT, 8, 0, 0}, {192, AR_REGIME_ONESHOT, 4, 0, 0}, {224, AR_REGIME_ONESHOT, 2, 0, 0},
      {256, AR_REGIME_ONESHOT, 4, 0, 0}}},
    // trailing all-reduce + RMSNorm, eight partials (K = 0, TP8): the one-shot
    // kernel in eight-CTA clusters, its 64-register form once a launch no longer
    // fits one wave of the 80-register form (T = 128 6.6 us, T = 256 10.8 us
    // against 8.1 and 11.0 us for the best streaming plans)
    {8, 0, 7168, 3,
     {{96, AR_REGIME_ONESHOT, 8, 0, 0}, {112, AR_REGIME_ONESHOT, 2, 0, 0}, {256, AR_REGIME_ONESHOT, 8, 0, 0}}},
};

bool valid_regime(int r) {
    return r == AR_REGIME_AUTO || r == AR_REGIME_CLUSTER || r == AR_REGIME_STREAM ||
           r == AR_REGIME_ONESHOT || r == AR_REGIME_SPLIT;
}

bool valid_table(const ar_regime_rule* rules, int n) {
    if (n < 0 || n > AR_MAX_REGIME_RULES || (n > 0 && !rules)) return false;
    for (int i = 0; i < n; ++i) {
        const ar_regime_rule& r = rules[i];
        if (r.max_tokens < 1 || (i > 0 && r.max_tokens <= rules[i - 1].max_tokens)) return false;
        if (!valid_regime(r.regime)) return false;
        if (r.ctas_per_row != 0) {
            if (r.regime != AR_REGIME_CLUSTER && r.regime != AR_REGIME_SPLIT && r.regime != AR_REGIME_ONESHOT)
                return false;
            if (r.ctas_per_row < 2 || r.ctas_per_row > 16) return false;
        }
        if (r.stage_bytes != 0 || r.producer_warps != 0) {
            if (r.regime != AR_REGIME_CLUSTER && r.regime != AR_REGIME_STREAM) return false;
            if (r.stage_bytes != 0 && (r.stage_bytes < 1024 || r.stage_bytes > 131072)) return false;
            if (r.producer_warps < 0 || r.producer_warps > 4) return false;
        }
    }
    return true;
}

// The built-in table for the workspace's shape, if the library has one.
void install_builtin_table(ar_workspace* ws) {
    ws->table_n = 0;
    for (const BuiltinTable& b : kBuiltinTables)
        if (b.R == ws->R && b.K == ws->K && b.H == ws->H) {
            ws->table_n = b.n;
            for (int i = 0; i < b.n; ++i) ws->table[i] = b.rules[i];
        }
}

struct Plans {
    arf::ClusterPlan c{};
    arf::StreamPlan s{};
    arf::SplitPlan x{};
};

// Host-side occupancy queries, cached per (device, query kind, kernel
// instantiation, block, shared memory, cluster) in a fixed-size table (no
// allocation): resident blocks per SM of a one-shot plan (kind 0) and
// co-resident clusters of a clustered streaming plan (kind 1) or of a split
// plan (kind 2).
struct OccEntry {
    int key[7];  // device + 1, kind, then the kind's fields; key[0] == 0: empty
    int n;
};
OccEntry g_occ[64];
int g_occ_next = 0;
std::mutex g_occ_mu;

template <class Query>
int occ_cached(const int (&key)[7], Query query) {
    std::lock_guard<std::mutex> lock(g_occ_mu);
    for (const OccEntry& e : g_occ)
        if (std::memcmp(e.key, key, sizeof key) == 0) return e.n;
    const int n = query();
    OccEntry& e = g_occ[g_occ_next];
    std::memcpy(e.key, key, sizeof key);
    e.n = n;
    g_occ_next = (g_occ_next + 1) % 64;
    return n;
}

int oneshot_blocks_per_sm(int device, const arf::ClusterPlan& p, bool res_f32) {
    const int key[7] = {device + 1, 0, p.maxt, res_f32 ? 1 : 0, p.threads, p.smem, 0};
    return occ_cached(key, [&] { return arf::cluster_rows_blocks_per_sm(p, res_f32); });
}

int stream_active_clusters(int device, const arf::StreamPlan& p, bool res_f32) {
    const int key[7] = {device + 1, 1, p.cpt, res_f32 ? 1 : 0, p.threads, p.smem, p.geo.C};
    return occ_cached(key, [&] { return arf::stream_rows_active_clusters(p, res_f32); });
}

int split_active_clusters(int device, const arf::SplitPlan& p, bool res_f32) {
    const int key[7] = {device + 1, 2, p.cpt, res_f32 ? 1 : 0, p.threads, p.smem, p.geo.C};
    return occ_cached(key, [&] { return arf::split_rows_active_clusters(p, res_f32); });
}

// A clustered streaming plan sizes its grid from shared memory per SM; the
// device may co-schedule fewer clusters (a cluster lives in one GPC, and the
// GPCs' SM counts need not be multiples of the cluster size).  The rows go
// round-robin over the clusters, so clusters beyond the co-resident ones
// would only start once others finish (measured: dsv3 T = 192, four-CTA
// tiles with 24 KB slots, 114 planned clusters, the last ones starting
// 19 us into the launch); the grid is capped at the co-resident count.
// Returns whether the grid fills every co-resident cluster slot.
bool stream_wave_fit(const ar_workspace* ws, arf::StreamPlan* p, bool res_f32) {
    if ((ws->flags & AR_WS_DRY_RUN) || p->geo.C < 2) return false;
    const int n = stream_active_clusters(ws->device, *p, res_f32);
    if (n < 1) return false;
    if ((int64_t)n * p->geo.C < p->grid) p->grid = n * p->geo.C;
    return p->grid / p->geo.C >= n;
}

// A one-shot launch of eight loads per thread that does not fit one wave of
// the 80-register form runs the 64-register form when that holds more CTAs
// (measured for eight partials, K = 0, H = 7168: T = 128 9.1 -> 7.0 us,
// T = 256 17.2 -> 12.9 us; within one wave the 80-register form is 0.2-0.4 us
// faster).
void oneshot_wave_fit(const ar_workspace* ws, arf::ClusterPlan* p, int64_t T, bool res_f32) {
    if ((ws->flags & AR_WS_DRY_RUN) || p->maxt != 8 || p->threads > 512) return;
    const int b80 = oneshot_blocks_per_sm(ws->device, *p, res_f32);
    if (T * p->C <= (int64_t)b80 * ws->num_sms) return;
    arf::ClusterPlan q = *p;
    q.maxt = arf::kClusterMaxTerms64;
    if (arf::oneshot_prefer_64(*p, T, ws->num_sms, b80, oneshot_blocks_per_sm(ws->device, q, res_f32))) *p = q;
}


// Column groups of a split plan (0: the planner's choice).
int split_groups(const ar_workspace* ws) { return ws->split_groups; }

// A split plan of one round buffers all of a CTA's segments; for heavy rows
// that can leave one CTA per SM and fewer co-resident clusters than rows, so
// the last rows would run in a second wave.  Then the same cluster size with
// two copy rounds (half the buffers) runs instead when the device holds more
// of its clusters (measured at R = 16, K = 10, H = 8192).
void split_wave_fit(const ar_workspace* ws, arf::SplitPlan* p, int R, int K, int H, bool shared, int64_t T,
                    bool res_f32) {
    if ((ws->flags & AR_WS_DRY_RUN) || p->geo.rounds != 1) return;
    const int n1 = split_active_clusters(ws->device, *p, res_f32);
    if (n1 < 1 || n1 >= T) return;
    arf::SplitPlan q{};
    if (!arf::plan_split_rows(R, K, H, shared, T, ws->num_sms, ws->smem_optin, ws->max_cluster_split,
                              p->geo.C, &q, split_groups(ws), 2))
        return;
    if (arf::split_prefer_two_rounds(T, n1, split_active_clusters(ws->device, q, res_f32))) *p = q;
}

// Plan `regime` with `ctas` CTAs per row (0: the regime's own choice).
// Returns the regime that will run (a streaming plan reports CLUSTER when its
// rows are split over a cluster, STREAM otherwise), 0 when there is no plan.
int plan_regime(const ar_workspace* ws, int regime, int ctas, int R, int K, int H, bool shared,
                int64_t T, Plans* p, int stage_bytes = 0, int producer_warps = 0) {
    const int sb = stage_bytes ? stage_bytes : ws->stage_bytes;
    const int pw = producer_warps ? producer_warps : ws->producer_warps;
    switch (regime) {
        case AR_REGIME_ONESHOT:
            return arf::plan_cluster_rows(R, K, H, shared, ws->max_cluster, T, ws->num_sms, &p->c, ctas)
                       ? AR_REGIME_ONESHOT
                       : 0;
        case AR_REGIME_SPLIT:
            // the given cluster size, else the largest that fits; with every
            // segment buffered at once, else in two copy rounds
            for (int rounds = 1; rounds <= 2; ++rounds)
                for (int c = ctas ? ctas : 16; c >= 2; c = ctas ? 0 : c >> 1)
                    if (arf::plan_split_rows(R, K, H, shared, T, ws->num_sms, ws->smem_optin,
                                             ws->max_cluster_split, c, &p->x, split_groups(ws), rounds))
                        return AR_REGIME_SPLIT;
            return 0;
        case AR_REGIME_STREAM:
        case AR_REGIME_CLUSTER: {
            int C = regime == AR_REGIME_STREAM ? 1 : ctas;
            if (C == 0) {
                arf::StreamPlan probe{};
                if (!arf::plan_stream_rows(R, K, H, shared, T, ws->num_sms, ws->smem_optin,
                                           ws->max_cluster_stream, 0, sb, &probe, pw))
                    return 0;
                C = probe.geo.C > 1 ? probe.geo.C : 2;
            }
            if (!arf::plan_stream_rows(R, K, H, shared, T, ws->num_sms, ws->smem_optin,
                                       ws->max_cluster_stream, C, sb, &p->s, pw,
                                       ws->split_ok ? ws->max_tail_parts : 0))
                return 0;
            return p->s.geo.C > 1 ? AR_REGIME_CLUSTER : AR_REGIME_STREAM;
        }
    }
    return 0;
}

// The built-in choice (measured on GB300 with the tuner):
//  - light rows (at most 8 summands per 16-byte chunk, one load wave per
//    thread) up to 5/3 rows per SM: the one-shot kernel (two and eight
//    partials, K = 0, H = 7168: ahead of whole-row streaming to T = 256 with
//    the 40-register and the 64-register forms);
//  - heavy rows at small T (one cluster per row in three quarters of the
//    SMs): the split kernel, fewest bulk copies per CTA;
//  - otherwise the streaming kernel (tiles over a cluster for small T, whole
//    rows for large T).
int plan_heuristic(const ar_workspace* ws, int R, int K, int H, bool shared, int64_t T, Plans* p) {
    const int summands = (shared ? R : 0) + R * K;
    const bool light = summands <= 8 && 3 * T <= 5 * (int64_t)ws->num_sms;
    if (light && arf::plan_cluster_rows(R, K, H, shared, ws->max_cluster, T, ws->num_sms, &p->c))
        return AR_REGIME_ONESHOT;
    if (summands > 8 && arf::plan_split_rows(R, K, H, shared, T, ws->num_sms, ws->smem_optin,
                                             ws->max_cluster_split, 0, &p->x, split_groups(ws)))
        return AR_REGIME_SPLIT;
    if (!arf::plan_stream_rows(R, K, H, shared, T, ws->num_sms, ws->smem_optin,
                               ws->max_cluster_stream, 0, ws->stage_bytes, &p->s, ws->producer_warps,
                               ws->split_ok ? ws->max_tail_parts : 0))
        return 0;
    return p->s.geo.C > 1 ? AR_REGIME_CLUSTER : AR_REGIME_STREAM;
}

// Largest clusters the device co-schedules for the block shapes of one model
// shape (R, K, H): the one-shot kernel, the clustered streaming kernel (16
// tiles of one row) and the split kernel.
void cluster_limits(int R, int K, int H, int num_sms, int smem_optin, int* max_cluster,
                    int* max_cluster_stream, int* max_cluster_split) {
    arf::ClusterPlan p{};
    *max_cluster = 16;
    if (arf::plan_cluster_rows(R, K, H, true, 16, 1, num_sms, &p))
        *max_cluster = arf::cluster_rows_max_cluster(p.threads, p.smem, false);
    if (*max_cluster < 1) *max_cluster = 1;
    arf::StreamPlan sp{};
    *max_cluster_stream = 1;
    for (int c = 16; c >= 2 && *max_cluster_stream == 1; c >>= 1)
        if (arf::plan_stream_rows(R, K, H, true, 1, num_sms, smem_optin, 16, c, 0, &sp))
            *max_cluster_stream = arf::stream_rows_max_cluster(sp.threads, sp.smem, sp.cpt);
    arf::SplitPlan xp{};
    *max_cluster_split = 1;
    for (int c = 16; c >= 2 && *max_cluster_split == 1; c >>= 1)
        if (arf::plan_split_rows(R, K, H, true, 1, num_sms, smem_optin, 16, c, &xp))
            *max_cluster_split = arf::split_rows_max_cluster(xp.threads, xp.smem, xp.cpt);
}

// What the last call launched (or, on a dry-run workspace, planned).
void record_plan(ar_workspace* ws, int regime, int ctas, int grid, const Plans& pl) {
    ws->last_regime = regime;
    ws->last_ctas = ctas;
    ws->last_grid = grid;
    ar_plan_info& i = ws->last_plan;
    std::memset(&i, 0, sizeof i);
    i.regime = regime;
    i.ctas_per_row = ctas;
    i.grid = grid;
    if (regime == AR_REGIME_ONESHOT) {
        i.block = pl.c.threads;
        i.smem_bytes = pl.c.smem;
        i.loads_per_thread = pl.c.maxt == arf::kClusterMaxTerms64 ? 8 : pl.c.maxt;
    } else if (regime == AR_REGIME_SPLIT) {
        i.block = pl.x.threads;
        i.smem_bytes = pl.x.smem;
        i.column_groups = pl.x.geo.C / pl.x.geo.Cs;
        i.copy_rounds = pl.x.geo.rounds;
        i.producer_warps = 1;
    } else {
        i.block = pl.s.threads;
        i.smem_bytes = pl.s.smem;
        i.ring_slots = pl.s.geo.nstages;
        i.ring_slot_bytes = pl.s.geo.slot_bytes;
        i.producer_warps = pl.s.geo.producers;
    }
}

ar_status run(ar_workspace* ws, const void* const* E, int64_t rows_e, const int32_t* perm,
              const float* w, const void* const* S, const void* residual, const void* gamma,
              float weight_bias, float eps, int64_t T, int R, int K, int H, void* out,
              void* residual_out, int res_f32, void* stream, bool routed_call,
              const float* gate = nullptr,
              bool (*plan_fits)(void* ctx, int regime, const Plans& p, bool res_f32) = nullptr,
              void* fits_ctx = nullptr) {
    if (!ws) return AR_ERR_INVALID_ARG;
    if (R != ws->R || H != ws->H) return AR_ERR_INVALID_ARG;
    if (routed_call && K != ws->K) return AR_ERR_INVALID_ARG;
    if (!(eps == ws->eps)) return AR_ERR_INVALID_ARG;
    if (T < 0) return AR_ERR_INVALID_ARG;
    if (T > ws->max_tokens) return AR_ERR_CAPACITY;
    if (res_f32 != 0 && res_f32 != 1) return AR_ERR_INVALID_ARG;
    if (T == 0) return AR_OK;
    if (!residual || !gamma || !out || !residual_out) return AR_ERR_INVALID_ARG;
    if (K > 0) {
        if (!E || !perm || !w || rows_e < 1) return AR_ERR_INVALID_ARG;
        if (rows_e > (INT64_MAX / 4) / H) return AR_ERR_INVALID_ARG;
        for (int r = 0; r < R; ++r)
            if (!E[r]) return AR_ERR_INVALID_ARG;
    }
    if (K == 0 && !S) return AR_ERR_INVALID_ARG;  // nothing to reduce
    if (S)
        for (int r = 0; r < R; ++r)
            if (!S[r]) return AR_ERR_INVALID_ARG;

    // Alignment: 16-byte vectors and bulk copies everywhere.
    if (!aligned(residual, 16) || !aligned(gamma, 16) || !aligned(out, 16) ||
        !aligned(residual_out, 16))
        return AR_ERR_ALIGNMENT;
    if (K > 0) {
        if (!aligned(perm, 4) || !aligned(w, 4)) return AR_ERR_ALIGNMENT;
        for (int r = 0; r < R; ++r)
            if (!aligned(E[r], 16)) return AR_ERR_ALIGNMENT;
    }
    if (S)
        for (int r = 0; r < R; ++r)
            if (!aligned(S[r], 16)) return AR_ERR_ALIGNMENT;
    if (gate && !aligned(gate, 4)) return AR_ERR_ALIGNMENT;

    // Outputs must not overlap each other or an input (the exact bf16 in-place
    // residual alias excepted).
    const int64_t row2 = T * H * 2;
    const Range r_out = range_of(out, row2);
    const Range r_rout = range_of(residual_out, res_f32 ? 2 * row2 : row2);
    const bool inplace = (residual_out == residual) && !res_f32;
    if (overlap(r_out, r_rout)) return AR_ERR_INVALID_ARG;
    Range ins[2 * AR_MAX_RANKS + 5];
    int n_in = 0;
    ins[n_in++] = range_of(gamma, (int64_t)H * 2);
    if (K > 0) {
        ins[n_in++] = range_of(perm, T * K * 4);
        ins[n_in++] = range_of(w, T * K * 4);
        for (int r = 0; r < R; ++r) ins[n_in++] = range_of(E[r], rows_e * H * 2);
    }
    if (S)
        for (int r = 0; r < R; ++r) ins[n_in++] = range_of(S[r], row2);
    if (gate) ins[n_in++] = range_of(gate, T * 4);
    for (int i = 0; i < n_in; ++i)
        if (overlap(r_out, ins[i]) || overlap(r_rout, ins[i])) return AR_ERR_INVALID_ARG;
    const Range r_res = range_of(residual, row2);
    if (overlap(r_out, r_res)) return AR_ERR_INVALID_ARG;
    if (!inplace && overlap(r_rout, r_res)) return AR_ERR_INVALID_ARG;

    // Regime and launch plan: a forced regime, else the table's rule for T,
    // else (no rule, or no plan for it) the heuristic.
    const bool shared = S != nullptr;
    Plans pl;
    int regime = 0;
    if (ws->regime_force != AR_REGIME_AUTO) {
        regime = plan_regime(ws, ws->regime_force, ws->force_ctas_per_row, R, K, H, shared, T, &pl);
        if (!regime) return AR_ERR_UNSUPPORTED;
    } else {
        for (int i = 0; i < ws->table_n; ++i)
            if (T <= ws->table[i].max_tokens) {
                if (ws->table[i].regime != AR_REGIME_AUTO)
                    regime = plan_regime(ws, ws->table[i].regime, ws->table[i].ctas_per_row, R, K, H,
                                         shared, T, &pl, ws->table[i].stage_bytes,
                                         ws->table[i].producer_warps);
                break;
            }
        if (!regime) regime = plan_heuristic(ws, R, K, H, shared, T, &pl);
        if (!regime) return AR_ERR_UNSUPPORTED;
    }
    // The injected wait exists only in whole-row streaming.
    if (ws->stall_wait_ns && regime != AR_REGIME_STREAM) return AR_ERR_UNSUPPORTED;
    // A caller-supplied check of the exact launch (block, shared memory,
    // cluster): a plan the device cannot co-schedule is declined here, before
    // anything is launched.
    if (plan_fits && !plan_fits(fits_ctx, regime, pl, res_f32 != 0)) return AR_ERR_UNSUPPORTED;
    // The occupancy queries below run on the current device and are cached
    // under the workspace's: the two must be the same device.
    if (!(ws->flags & AR_WS_DRY_RUN)) {
        int cur = -1;
        if (cudaGetDevice(&cur) != cudaSuccess) return AR_ERR_CUDA;
        if (cur != ws->device) return AR_ERR_INVALID_ARG;
    }
    if (regime == AR_REGIME_ONESHOT) oneshot_wave_fit(ws, &pl.c, T, res_f32 != 0);
    if (regime == AR_REGIME_SPLIT) split_wave_fit(ws, &pl.x, R, K, H, shared, T, res_f32 != 0);
    const bool fills_device = regime == AR_REGIME_CLUSTER && stream_wave_fit(ws, &pl.s, res_f32 != 0);
    const int ctas = regime == AR_REGIME_ONESHOT ? pl.c.C
                     : regime == AR_REGIME_SPLIT ? pl.x.geo.C
                     : regime == AR_REGIME_CLUSTER ? pl.s.geo.C
                                                   : pl.s.grid;
    const int grid = regime == AR_REGIME_ONESHOT ? (int)(T * pl.c.C)
                     : regime == AR_REGIME_SPLIT ? pl.x.grid
                                                 : pl.s.grid;

    if (ws->flags & AR_WS_DRY_RUN) {
        record_plan(ws, regime, ctas, grid, pl);
        return AR_VALIDATED;
    }

    arf::RowArgs a;
    std::memset(&a, 0, sizeof a);
    for (int r = 0; r < R; ++r) {
        if (K > 0) a.E[r] = static_cast<const uint16_t*>(E[r]);
        if (S) a.S[r] = static_cast<const uint16_t*>(S[r]);
    }
    a.perm = perm;
    a.w = w;
    a.residual = static_cast<const uint16_t*>(residual);
    a.gamma = static_cast<const uint16_t*>(gamma);
    a.out = out;
    a.residual_out = residual_out;
    a.err = ws->d_err;
    if (ws->d_part) {
        a.part_count = ws->d_part;
        a.part_scratch = reinterpret_cast<float*>(ws->d_part + part_counter_words(ws->num_sms));
    }
    a.T = T;
    a.rows_e = K > 0 ? rows_e : 0;
    a.R = R;
    a.K = K;
    a.H = H;
    a.has_shared = S ? 1 : 0;
    a.shared_gate = gate;
    a.norm_bf16_h = (ws->flags & AR_WS_NORM_BF16_H) ? 1 : 0;
    a.weight_bias = weight_bias;
    a.eps = eps;
    a.stall_wait_ns = ws->stall_wait_ns;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    // A clustered streaming launch that fills every co-resident cluster slot
    // runs without programmatic dependent launch: the next call's clusters
    // cannot be placed before it drains anyway, and placed early they left
    // an eight-CTA cluster waiting (measured, dsv3 T = 36, 36 clusters of 8
    // on 36 slots: +1.7-2.0 us per call with the attribute, none without).
    const bool pdl = (ws->flags & AR_WS_PDL) != 0 && !fills_device;
    if (regime == AR_REGIME_ONESHOT)
        e = arf::launch_cluster_rows(a, pl.c, res_f32 != 0, s, pdl);
    else if (regime == AR_REGIME_SPLIT)
        e = arf::launch_split_rows(a, pl.x, res_f32 != 0, s, pdl);
    else
        e = arf::launch_stream_rows(a, pl.s, res_f32 != 0, s, pdl);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ERR_CUDA;
    }
    record_plan(ws, regime, ctas, grid, pl);
    return AR_OK;
}

}  // namespace

extern "C" {

ar_status ar_workspace_create(int device, int ranks, int top_k, int hidden, int64_t max_tokens,
                              float eps, unsigned flags, ar_workspace** out) {
    if (!out) return AR_ERR_INVALID_ARG;
    *out = nullptr;
    if (max_tokens < 1 || !(eps >= 0.0f) || eps > 3.0e38f) return AR_ERR_INVALID_ARG;
    if ((flags & ~(AR_WS_DRY_RUN | AR_WS_NORM_BF16_H | AR_WS_PDL)) != 0) return AR_ERR_INVALID_ARG;
    if (hidden < 8 || hidden % 8 != 0) return hidden < 8 ? AR_ERR_UNSUPPORTED : AR_ERR_ALIGNMENT;
    if (ranks < 1 || ranks > AR_MAX_RANKS || top_k < 0 || top_k > AR_MAX_TOP_K ||
        hidden > AR_MAX_HIDDEN || max_tokens > kMaxTokensLimit)
        return AR_ERR_UNSUPPORTED;

    ar_workspace* ws = new (std::nothrow) ar_workspace();
    if (!ws) return AR_ERR_CUDA;
    ws->device = device;
    ws->R = ranks;
    ws->K = top_k;
    ws->H = hidden;
    ws->max_tokens = max_tokens;
    ws->eps = eps;
    ws->flags = flags;
    ws->d_err = nullptr;
    ws->d_part = nullptr;
    ws->split_ok = (flags & AR_WS_DRY_RUN) != 0;
    ws->max_tail_parts = arf::kMaxTailParts;
    ws->regime_force = AR_REGIME_AUTO;
    ws->force_ctas_per_row = 0;
    ws->stage_bytes = 0;
    ws->producer_warps = 0;
    ws->last_regime = 0;
    ws->last_ctas = 0;
    ws->last_grid = 0;
    std::memset(&ws->last_plan, 0, sizeof ws->last_plan);
    install_builtin_table(ws);

    if (flags & AR_WS_DRY_RUN) {
        ws->num_sms = kDryRunSms;
        ws->smem_optin = kDryRunSmemOptin;
        ws->max_cluster = 16;
        ws->max_cluster_stream = 16;
        ws->max_cluster_split = 16;
        *out = ws;
        return AR_OK;
    }

    int prev = -1;
    ar_status st = AR_OK;
    cudaDeviceProp prop;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess ||
        cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
        st = AR_ERR_CUDA;
        goto fail;
    }
    if (prop.major < 10) {
        st = AR_ERR_UNSUPPORTED;
        goto fail;
    }
    ws->num_sms = prop.multiProcessorCount;
    ws->smem_optin = (int)prop.sharedMemPerBlockOptin;
    if (arf::stream_rows_set_attributes(ws->smem_optin) != cudaSuccess) {
        st = AR_ERR_CUDA;
        goto fail;
    }
    if (arf::cluster_rows_set_attributes() != cudaSuccess ||
        arf::split_rows_set_attributes(ws->smem_optin) != cudaSuccess) {
        st = AR_ERR_CUDA;
        goto fail;
    }
    cluster_limits(ranks, top_k, hidden, ws->num_sms, ws->smem_optin, &ws->max_cluster,
                   &ws->max_cluster_stream, &ws->max_cluster_split);
    if (cudaMalloc(&ws->d_err, 256) != cudaSuccess || cudaMemset(ws->d_err, 0, 256) != cudaSuccess) {
        st = AR_ERR_CUDA;
        goto fail;
    }
    {
        // Split rows: one counter and one fp32 partial row per CTA of a whole-row grid.
        const size_t bytes = part_bytes(ws->num_sms, hidden);
        if (cudaMalloc(&ws->d_part, bytes) != cudaSuccess || cudaMemset(ws->d_part, 0, bytes) != cudaSuccess) {
            st = AR_ERR_CUDA;
            goto fail;
        }
        ws->split_ok = true;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        st = AR_ERR_CUDA;
        goto fail;
    }
    (void)cudaSetDevice(prev);
    *out = ws;
    return AR_OK;

fail:
    (void)cudaGetLastError();
    if (ws->d_err) (void)cudaFree(ws->d_err);
    if (ws->d_part) (void)cudaFree(ws->d_part);
    if (prev >= 0) (void)cudaSetDevice(prev);
    delete ws;
    return st;
}

ar_status ar_workspace_destroy(ar_workspace* ws) {
    if (!ws) return AR_OK;
    ar_status st = AR_OK;
    if (ws->d_err) {
        int prev = -1;
        (void)cudaGetDevice(&prev);
        if (cudaSetDevice(ws->device) != cudaSuccess || cudaFree(ws->d_err) != cudaSuccess ||
            (ws->d_part && cudaFree(ws->d_part) != cudaSuccess))
            st = AR_ERR_CUDA;
        if (prev >= 0) (void)cudaSetDevice(prev);
    }
    delete ws;
    return st;
}

ar_status ar_finalize_rmsnorm(ar_workspace* ws, const void* const* expert_out, int64_t rows_e,
                              const int32_t* perm, const float* topk_w,
                              const void* const* shared_out, const void* residual,
                              const void* gamma, float weight_bias, float eps, int64_t T, int R,
                              int K, int H, void* out, void* residual_out,
                              int residual_out_is_fp32, void* stream) {
    if (K < 0 || K > AR_MAX_TOP_K || R < 1 || R > AR_MAX_RANKS) return AR_ERR_INVALID_ARG;
    return run(ws, expert_out, rows_e, perm, topk_w, shared_out, residual, gamma, weight_bias, eps,
               T, R, K, H, out, residual_out, residual_out_is_fp32, stream, true);
}

ar_status ar_finalize_rmsnorm_gated(ar_workspace* ws, const void* const* expert_out,
                                    int64_t rows_e, const int32_t* perm, const float* topk_w,
                                    const void* const* shared_out, const float* shared_gate,
                                    const void* residual, const void* gamma, float weight_bias,
                                    float eps, int64_t T, int R, int K, int H, void* out,
                                    void* residual_out, int residual_out_is_fp32, void* stream) {
    if (K < 0 || K > AR_MAX_TOP_K || R < 1 || R > AR_MAX_RANKS) return AR_ERR_INVALID_ARG;
    if (!ws) return AR_ERR_INVALID_ARG;
    if (T > 0 && (!shared_gate || !shared_out)) return AR_ERR_INVALID_ARG;
    return run(ws, expert_out, rows_e, perm, topk_w, shared_out, residual, gamma, weight_bias, eps,
               T, R, K, H, out, residual_out, residual_out_is_fp32, stream, true, shared_gate);
}

ar_status ar_rmsnorm(ar_workspace* ws, const void* const* partials, int R, const void* residual,
                     const void* gamma, float weight_bias, float eps, int64_t T, int H, void* out,
                     void* residual_out, int residual_out_is_fp32, void* stream) {
    if (R < 1 || R > AR_MAX_RANKS) return AR_ERR_INVALID_ARG;
    if (!partials) return AR_ERR_INVALID_ARG;
    return run(ws, nullptr, 0, nullptr, nullptr, partials, residual, gamma, weight_bias, eps, T, R,
               0, H, out, residual_out, residual_out_is_fp32, stream, false);
}

ar_status ar_mhc_post(ar_workspace* ws, const void* const* partials, int R, const void* streams,
                      const float* post, const float* comb, int64_t T, int H, int hc,
                      void* streams_out, void* stream) {
    if (!ws || !partials) return AR_ERR_INVALID_ARG;
    if (R < 1 || R > AR_MAX_RANKS || R != ws->R || H != ws->H) return AR_ERR_INVALID_ARG;
    if (hc < 1 || hc > AR_MAX_HC_STREAMS) return AR_ERR_INVALID_ARG;
    if (T < 0) return AR_ERR_INVALID_ARG;
    if (T > ws->max_tokens) return AR_ERR_CAPACITY;
    if (T == 0) return AR_OK;
    if (!streams || !post || !comb || !streams_out) return AR_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r)
        if (!partials[r]) return AR_ERR_INVALID_ARG;
    if (!aligned(streams, 16) || !aligned(streams_out, 16) || !aligned(post, 4) || !aligned(comb, 4))
        return AR_ERR_ALIGNMENT;
    for (int r = 0; r < R; ++r)
        if (!aligned(partials[r], 16)) return AR_ERR_ALIGNMENT;
    // The output may be the incoming streams exactly; otherwise it overlaps no input.
    const Range r_out = range_of(streams_out, T * hc * H * 2);
    const Range r_x = range_of(streams, T * hc * H * 2);
    if (streams_out != streams && overlap(r_out, r_x)) return AR_ERR_INVALID_ARG;
    if (overlap(r_out, range_of(post, T * hc * 4)) || overlap(r_out, range_of(comb, T * hc * hc * 4)))
        return AR_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r)
        if (overlap(r_out, range_of(partials[r], T * H * 2))) return AR_ERR_INVALID_ARG;
    if (ws->flags & AR_WS_DRY_RUN) return AR_VALIDATED;

    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return AR_ERR_CUDA;
    if (cur != ws->device) return AR_ERR_INVALID_ARG;
    arf::MhcArgs a;
    std::memset(&a, 0, sizeof a);
    for (int r = 0; r < R; ++r) a.P[r] = static_cast<const uint16_t*>(partials[r]);
    a.x = static_cast<const uint16_t*>(streams);
    a.post = post;
    a.comb = comb;
    a.out = static_cast<uint16_t*>(streams_out);
    a.T = T;
    a.R = R;
    a.H = H;
    a.hc = hc;
    if (arf::launch_mhc_post(a, static_cast<cudaStream_t>(stream), (ws->flags & AR_WS_PDL) != 0) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ERR_CUDA;
    }
    return AR_OK;
}

ar_status ar_workspace_device_error(ar_workspace* ws, int* code) {
    if (!ws || !code) return AR_ERR_INVALID_ARG;
    *code = 0;
    if (ws->flags & AR_WS_DRY_RUN) return AR_OK;
    int prev = -1;
    (void)cudaGetDevice(&prev);
    unsigned v = 0;
    ar_status st = AR_OK;
    if (cudaSetDevice(ws->device) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&v, ws->d_err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(ws->d_err, 0, sizeof v) != cudaSuccess ||
        // a call cut short may have left split-row counters part-way: restart them
        (v && ws->d_part &&
         cudaMemset(ws->d_part, 0, part_counter_words(ws->num_sms) * sizeof(unsigned)) != cudaSuccess) ||
        cudaDeviceSynchronize() != cudaSuccess) {
        (void)cudaGetLastError();
        st = AR_ERR_CUDA;
    }
    if (prev >= 0) (void)cudaSetDevice(prev);
    if (st != AR_OK) return st;
    *code = (int)v;
    return v ? AR_ERR_DEVICE_CHECK : AR_OK;
}

ar_status ar_workspace_set_regime(ar_workspace* ws, int regime) {
    if (!ws) return AR_ERR_INVALID_ARG;
    if (regime != AR_REGIME_AUTO && regime != AR_REGIME_CLUSTER && regime != AR_REGIME_STREAM &&
        regime != AR_REGIME_ONESHOT && regime != AR_REGIME_SPLIT)
        return AR_ERR_INVALID_ARG;
    ws->regime_force = regime;
    return AR_OK;
}

ar_status ar_workspace_set_cluster_size(ar_workspace* ws, int ctas_per_row) {
    if (!ws) return AR_ERR_INVALID_ARG;
    if (ctas_per_row != 0 && (ctas_per_row < 2 || ctas_per_row > 16)) return AR_ERR_INVALID_ARG;
    ws->force_ctas_per_row = ctas_per_row;
    return AR_OK;
}

ar_status ar_workspace_set_stage_bytes(ar_workspace* ws, int bytes) {
    if (!ws) return AR_ERR_INVALID_ARG;
    if (bytes != 0 && (bytes < 1024 || bytes > 131072)) return AR_ERR_INVALID_ARG;
    ws->stage_bytes = bytes;
    return AR_OK;
}

ar_status ar_workspace_set_regime_table(ar_workspace* ws, const ar_regime_rule* rules, int n) {
    if (!ws || !valid_table(rules, n)) return AR_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) ws->table[i] = rules[i];
    ws->table_n = n;
    return AR_OK;
}

ar_status ar_workspace_get_regime_table(const ar_workspace* ws, ar_regime_rule* rules, int cap,
                                        int* n) {
    if (!ws || !n || cap < 0 || (cap > 0 && !rules)) return AR_ERR_INVALID_ARG;
    for (int i = 0; i < ws->table_n && i < cap; ++i) rules[i] = ws->table[i];
    *n = ws->table_n;
    return AR_OK;
}

ar_status ar_workspace_set_split_rows(ar_workspace* ws, int max_parts) {
    if (!ws) return AR_ERR_INVALID_ARG;
    if (max_parts < 0 || max_parts > arf::kMaxTailParts) return AR_ERR_INVALID_ARG;
    ws->max_tail_parts = max_parts;
    return AR_OK;
}

ar_status ar_workspace_set_split_column_groups(ar_workspace* ws, int groups) {
    if (!ws) return AR_ERR_INVALID_ARG;
    if (groups < 0 || groups > 8) return AR_ERR_INVALID_ARG;
    ws->split_groups = groups;
    return AR_OK;
}

ar_status ar_workspace_inject_wait_timeout(ar_workspace* ws, int64_t limit_ns) {
    if (!ws) return AR_ERR_INVALID_ARG;
    if (limit_ns < 0 || limit_ns > (int64_t)arf::kWaitLimitNs) return AR_ERR_INVALID_ARG;
    ws->stall_wait_ns = (unsigned long long)limit_ns;
    return AR_OK;
}

ar_status ar_workspace_set_producer_warps(ar_workspace* ws, int warps) {
    if (!ws) return AR_ERR_INVALID_ARG;
    if (warps < 0 || warps > 4) return AR_ERR_INVALID_ARG;
    ws->producer_warps = warps;
    return AR_OK;
}

int ar_workspace_last_grid(const ar_workspace* ws) { return ws ? ws->last_grid : 0; }

ar_status ar_workspace_last_plan(const ar_workspace* ws, ar_plan_info* info) {
    if (!ws || !info) return AR_ERR_INVALID_ARG;
    *info = ws->last_plan;
    return AR_OK;
}

int ar_workspace_last_regime(const ar_workspace* ws, int* ctas) {
    if (!ws) return 0;
    if (ctas) *ctas = ws->last_ctas;
    return ws->last_regime;
}

const char* ar_status_string(ar_status s) {
    switch (s) {
        case AR_OK: return "ok";
        case AR_ERR_INVALID_ARG: return "invalid argument";
        case AR_ERR_ALIGNMENT: return "misaligned pointer or hidden size not a multiple of 8";
        case AR_ERR_UNSUPPORTED: return "outside the library's limits";
        case AR_ERR_CAPACITY: return "more tokens than the workspace's max_tokens";
        case AR_ERR_CUDA: return "CUDA runtime error";
        case AR_ERR_DEVICE_CHECK: return "a device-side check fired";
        case AR_VALIDATED: return "validated (dry-run workspace, nothing launched)";
    }
    return "unknown status";
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc: code that runs while a serving
// framework captures a CUDA graph (allocation is illegal inside a capture),
// plugins living under an engine whose memory pool owns all device memory and
// rejects allocations it did not make, or deployments with a fixed device
// memory budget checked at start-up.  ar_workspace_create() allocates a small
// device block for the kernels' status word (and a split-row scratch), so
// those callers cannot use it.  ar_finalize_rmsnorm_noalloc() needs no
// workspace: the only global memory the kernels use beyond the caller's
// inputs and outputs -- the status word that device-side checks write -- lives
// in the fixed array below, which every GPU that loads this library holds
// until the process exits.  Without a split-row scratch, its plans never split
// the rows of whole-row streaming's last partial wave.
namespace {

constexpr int kNoAllocScratchBytes = 256;  // stated maximum; a call uses 4 bytes
static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoAllocScratchBytes / 4];

// Host-side caches (fixed size, no allocation): cluster limits per model
// shape, and whether an exact launch fits the device.
constexpr int kNoAllocMaxDevices = 64;
constexpr int kShapeCache = 32;
constexpr int kFitCache = 64;
struct ShapeLimits {
    int R, K, H;  // R == 0: empty entry
    int max_cluster, max_cluster_stream, max_cluster_split;
};
struct LaunchFit {
    int key[6];  // regime, instantiation, res_f32, threads, smem, cluster size; key[0] == 0: empty
    bool fits;
};
struct NoAllocDevice {
    bool ready;
    unsigned* scratch;  // device address of g_noalloc_scratch on this device
    int num_sms;
    int smem_optin;
    ShapeLimits shapes[kShapeCache];
    int next_shape;
    LaunchFit fit[kFitCache];
    int next_fit;
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// One-time set-up for the current device: kernel attributes and the device
// address of the scratch array.  Allocates nothing.
ar_status noalloc_setup(int device, NoAllocDevice** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocDevice& d = g_noalloc_dev[device];
    if (d.ready) {
        *out = &d;
        return AR_OK;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return AR_ERR_CUDA;
    if (prop.major < 10) return AR_ERR_UNSUPPORTED;
    if (arf::stream_rows_set_attributes((int)prop.sharedMemPerBlockOptin) != cudaSuccess ||
        arf::cluster_rows_set_attributes() != cudaSuccess ||
        arf::split_rows_set_attributes((int)prop.sharedMemPerBlockOptin) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ERR_CUDA;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return AR_ERR_CUDA;
    }
    d.scratch = static_cast<unsigned*>(p);
    d.num_sms = prop.multiProcessorCount;
    d.smem_optin = (int)prop.sharedMemPerBlockOptin;
    d.ready = true;
    *out = &d;
    return AR_OK;
}

// Cluster limits of a model shape, computed as ar_workspace_create() does
// (so the plans match the workspace entry point's) and cached.
ShapeLimits noalloc_limits(NoAllocDevice* d, int R, int K, int H) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (const ShapeLimits& e : d->shapes)
        if (e.R == R && e.K == K && e.H == H) return e;
    ShapeLimits e{R, K, H, 1, 1, 1};
    cluster_limits(R, K, H, d->num_sms, d->smem_optin, &e.max_cluster, &e.max_cluster_stream,
                   &e.max_cluster_split);
    d->shapes[d->next_shape] = e;
    d->next_shape = (d->next_shape + 1) % kShapeCache;
    return e;
}

// Whether the device can run the exact launch of a plan (cached).
bool noalloc_plan_fits(void* ctx, int regime, const Plans& p, bool res_f32) {
    NoAllocDevice* d = static_cast<NoAllocDevice*>(ctx);
    int key[6] = {regime, 0, res_f32 ? 1 : 0, 0, 0, 0};
    if (regime == AR_REGIME_ONESHOT) {
        key[1] = p.c.maxt; key[3] = p.c.threads; key[4] = p.c.smem; key[5] = p.c.C;
    } else if (regime == AR_REGIME_SPLIT) {
        key[1] = p.x.cpt; key[3] = p.x.threads; key[4] = p.x.smem; key[5] = p.x.geo.C;
    } else {
        key[1] = p.s.cpt; key[3] = p.s.threads; key[4] = p.s.smem; key[5] = p.s.geo.C;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (const LaunchFit& f : d->fit)
        if (f.key[0] != 0 && std::memcmp(f.key, key, sizeof key) == 0) return f.fits;
    const bool fits = regime == AR_REGIME_ONESHOT ? arf::cluster_rows_plan_fits(p.c, res_f32)
                      : regime == AR_REGIME_SPLIT ? arf::split_rows_plan_fits(p.x, res_f32)
                                                  : arf::stream_rows_plan_fits(p.s, res_f32);
    LaunchFit& f = d->fit[d->next_fit];
    std::memcpy(f.key, key, sizeof key);
    f.fits = fits;
    d->next_fit = (d->next_fit + 1) % kFitCache;
    return fits;
}

}  // namespace

extern "C" {

ar_status ar_finalize_rmsnorm_noalloc(const void* const* expert_out, int64_t rows_e,
                                      const int32_t* perm, const float* topk_w,
                                      const void* const* shared_out, const void* residual,
                                      const void* gamma, float weight_bias, float eps, int64_t T,
                                      int R, int K, int H, void* out, void* residual_out,
                                      int residual_out_is_fp32, void* stream) {
    if (K < 0 || K > AR_MAX_TOP_K || R < 1 || R > AR_MAX_RANKS) return AR_ERR_INVALID_ARG;
    if (H < 8 || H > AR_MAX_HIDDEN) return AR_ERR_UNSUPPORTED;
    if (H % 8 != 0) return AR_ERR_ALIGNMENT;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return AR_ERR_INVALID_ARG;
    if (T > kMaxTokensLimit) return AR_ERR_CAPACITY;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return AR_ERR_CUDA;
    if (device < 0 || device >= kNoAllocMaxDevices) return AR_ERR_UNSUPPORTED;
    NoAllocDevice* d = nullptr;
    const ar_status st = noalloc_setup(device, &d);
    if (st != AR_OK) return st;
    const ShapeLimits lim = noalloc_limits(d, R, K, H);

    // A workspace on the stack: the same validation, plans and kernels as
    // ar_finalize_rmsnorm(), with the scratch array as the status word and no
    // split-row scratch.
    ar_workspace ws;
    std::memset(&ws, 0, sizeof ws);
    ws.device = device;
    ws.R = R;
    ws.K = K;
    ws.H = H;
    ws.max_tokens = kMaxTokensLimit;
    ws.eps = eps;
    ws.flags = 0;
    ws.d_err = d->scratch;
    ws.num_sms = d->num_sms;
    ws.smem_optin = d->smem_optin;
    ws.max_cluster = lim.max_cluster;
    ws.max_cluster_stream = lim.max_cluster_stream;
    ws.max_cluster_split = lim.max_cluster_split;
    ws.regime_force = AR_REGIME_AUTO;
    install_builtin_table(&ws);
    // The status word is only ever OR-ed into by the kernels and read by
    // nobody here, so it is not cleared between calls.
    return run(&ws, expert_out, rows_e, perm, topk_w, shared_out, residual, gamma, weight_bias,
               eps, T, R, K, H, out, residual_out, residual_out_is_fp32, stream, true, nullptr,
               noalloc_plan_fits, d);
}

}  // extern "C"

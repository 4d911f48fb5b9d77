// Host-only check of the streaming kernel's launch planner and of the address
// arithmetic its kernel derives from a plan (compiled and run by
// tests/test_plans.py; no GPU needed).  For every shape it checks that the
// plan fits shared memory, that every CTA of a row owns at least one column
// chunk, that consumer threads cover every chunk, that a slot holds its
// segments and their coefficient header, and that a slot's bytes fit an
// mbarrier transaction count.  The automatic plan must exist for every shape.
#include "stream_rows.cu"
#include "split_rows.cu"
#include "cluster_rows.cu"
#include <cstdio>
#include <cstdlib>
using namespace arf;
int main() {
  long checks = 0, fails = 0, n64 = 0;
  int Hs[] = {8, 56, 256, 264, 2048, 6144, 7168, 8192, 12296, 16384};
  int Rs[] = {1, 2, 3, 8, 16};
  int Ks[] = {0, 1, 2, 5, 8, 10, 16};
  long Ts[] = {1, 2, 3, 4, 7, 16, 37, 64, 128, 151, 152, 153, 333, 512, 2048, 8192};
  for (int H : Hs) for (int R : Rs) for (int K : Ks) for (int sh = 0; sh < 2; ++sh) for (long T : Ts) {
    if (K == 0 && !sh) continue;
    for (int sb : {0, 1024, 4096, 16384, 65536, 131072})
    for (int Cf = 0; Cf <= 16; ++Cf) {
      StreamPlan p;
      const int split = (sb == 0 || sb == 65536) ? 8 : 0;  // split rows of the last wave
      if (!plan_stream_rows(R, K, H, sh, T, 152, 232448, 16, Cf, sb, &p, 0, split)) {
        if (Cf == 0 || Cf == 1) { ++fails; printf("auto/stream plan failed H=%d R=%d K=%d T=%ld Cf=%d\n", H, R, K, T, Cf); }
        continue;
      }
      const auto& g = p.geo;
      int C = g.C; int chunks = H / 8;
      int nS = sh ? R : 0, nseg = nS + 1 + R * K;
      ++checks;
      bool bad = false;
      if (p.smem > 232448) bad = true;
      if (stream_ring_offset(g.nstages) + g.nstages * g.slot_bytes > p.smem) bad = true;
      if (p.grid % C) bad = true;
      if (p.threads > 640 || p.threads % 32) bad = true;
      if (g.nstages < 2) bad = true;
      // split rows: whole rows fill complete waves, each split row's parts
      // have a CTA each and at least one segment each
      if (g.tail_parts < 1 || g.tail_parts > 8 || g.main_rows < 0 || g.main_rows > T) bad = true;
      if (g.tail_parts > 1) {
        if (C != 1 || !split) bad = true;
        if (g.main_rows % p.grid) bad = true;
        if ((T - g.main_rows) * g.tail_parts > p.grid) bad = true;
        if (g.tail_parts > nseg / 8) bad = true;
        if (T < 152 && (g.main_rows != 0 || p.grid != T * g.tail_parts)) bad = true;
        if (p.grid > 152) bad = true;
        for (int q = 0; q < g.tail_parts; ++q)
          if ((long)(q + 1) * nseg / g.tail_parts - (long)q * nseg / g.tail_parts < 1) bad = true;
      } else if (g.main_rows != T) bad = true;
      // every producer warp owns at least one slot
      if (g.producers < 1 || g.producers > 4 || g.producers > g.nstages) bad = true;
      if (g.seg_per_stage < 1 || g.seg_per_stage > 32 || g.seg_per_stage > nseg) bad = true;
      if (g.slot_bytes != kSlotHeader + g.seg_per_stage * g.seg_stride) bad = true;
      if (g.seg_per_stage * 4 > kSlotHeader) bad = true;
      // the tx bytes of one slot fit an mbarrier's transaction count
      if ((long)g.seg_per_stage * g.seg_stride >= (1 << 20)) bad = true;
      int ncw = p.threads / 32 - g.producers, nct = ncw * 32;
      if (ncw < 1) bad = true;
      for (int c = 0; c < C; ++c) {
        int chunk0 = c * g.tile_chunks;
        int nchunk = std::min(g.tile_chunks, chunks - chunk0);
        if (nchunk < 1) bad = true;
        if (nchunk * 16 > g.seg_stride) bad = true;
        if (g.seg_stride % 128) bad = true;
        // consumers cover every chunk of the tile exactly once
        if ((long)nct * p.cpt < nchunk) bad = true;
        // the last element written
        if ((long)(chunk0 + nchunk) * 8 > H) bad = true;
      }
      // header: rec[] ends before the ring
      int hdr = g.nstages * 16 + 16 + 2 * 16 * 4 + 64 * 4 + 16 + g.nstages;
      if (hdr > stream_ring_offset(g.nstages)) bad = true;
      if (nseg < 1) bad = true;
      // ring positions: q in [0, 2n) maps to a slot < n
      for (int q = 0; q < 2 * g.nstages; ++q) { int sl = q >= g.nstages ? q - g.nstages : q; if (sl < 0 || sl >= g.nstages) bad = true; }
      if (bad) { ++fails; if (fails < 20) printf("BAD H=%d R=%d K=%d sh=%d T=%ld Cf=%d -> C=%d tile=%d nst=%d slot=%d thr=%d smem=%d grid=%d\n", H,R,K,sh,T,Cf,C,g.tile_chunks,g.nstages,g.slot_bytes,p.threads,p.smem,p.grid); }
    }
  }
  // split plans (one row per cluster, segments dealt round-robin within a
  // column group)
  for (int H : Hs) for (int R : Rs) for (int K : Ks) for (int sh = 0; sh < 2; ++sh) for (long T : Ts)
  for (int G = 1; G <= 8; ++G) for (int rounds = 1; rounds <= 2; ++rounds) {
    if (K == 0 && !sh) continue;
    for (int Cf = 0; Cf <= 16; Cf = Cf ? Cf + 1 : 2) {
      SplitPlan p;
      if (!plan_split_rows(R, K, H, sh, T, 152, 232448, 16, Cf, &p, G, rounds)) continue;
      ++checks;
      const auto& g = p.geo;
      const int chunks = H / 8, nseg = (sh ? R : 0) + 1 + R * K, C = g.C, Cs = g.Cs;
      bool bad = false;
      if (p.smem > 232448 || p.grid != T * C || p.threads > 544 || p.threads % 32) bad = true;
      if (Cs < 2 || C != Cs * G || g.group_chunks * G < chunks || (G - 1) * g.group_chunks >= chunks) bad = true;
      const int consumers = p.threads - 32;
      if ((long)consumers * p.cpt < g.group_chunks) bad = true;  // partial row of a group fully covered
      if (2 * g.tile_chunks > p.cpt * consumers) bad = true;     // <= CPT float4 items per thread
      if (g.seg_stride < g.group_chunks * 16 || g.seg_stride % 128 || g.part_bytes < Cs * g.tile_chunks * 32) bad = true;
      if (g.row_f32_bytes < g.group_chunks * 32) bad = true;
      if (g.rounds != rounds) bad = true;
      const int nsr = (sh ? R : 0) + 1;
      bool second = false;
      long covered = 0;
      for (int c = 0; c < C; ++c) {
        const int grp = c / Cs, cs = c % Cs;
        const int g0 = grp * g.group_chunks, gchunks = std::min(g.group_chunks, chunks - g0);
        const int ns = (nseg - cs + Cs - 1) / Cs;
        // the kernel's own split of the CTA's segments: [0, nsr_c) shared
        // partials and residual, [nsr_c, nmid) the first routed half
        const int nsr_c = nsr > cs ? (nsr - 1 - cs) / Cs + 1 : 0;
        const int nmid = nsr_c + (ns - nsr_c + 1) / 2;
        if (gchunks < 1 || ns < 1 || ns > 64) bad = true;       // coefficient table of 64
        // buffers the CTA touches: every segment's, or with two rounds the
        // first nmid (segment i >= nmid lands in buffer i - nmid < ns - nmid)
        const int nbuf = rounds == 1 ? ns : nmid;
        if (rounds == 1 && ns > 32) bad = true;                 // one producer lane per segment
        if (rounds == 2 && (nmid > 32 || ns - nmid > 32 || ns - nmid > nmid)) bad = true;
        if (rounds == 2 && ns > nmid) second = true;
        if (1024 + g.part_bytes + std::max<long>(g.row_f32_bytes, (long)nbuf * g.seg_stride) > p.smem) bad = true;
        if ((long)ns * gchunks * 16 >= (1 << 20)) bad = true;   // mbarrier transaction count
        const int ntile = std::min(g.tile_chunks, gchunks - cs * g.tile_chunks);
        if (ntile < 1) bad = true;                               // every CTA owns a tile
        if ((long)Cs * ntile * 32 > g.part_bytes) bad = true;
        covered += ntile;
      }
      if (covered != chunks) bad = true;                         // tiles partition the row
      if (rounds == 2 && !second) bad = true;                    // a second round exists
      if (bad) { ++fails; if (fails < 20) printf("BAD split H=%d R=%d K=%d sh=%d T=%ld Cf=%d G=%d rounds=%d\n", H, R, K, sh, T, Cf, G, rounds); }
    }
  }
  // one-shot plans (one cluster per row, every load of a thread in flight)
  for (int H : Hs) for (int R : Rs) for (int K : Ks) for (int sh = 0; sh < 2; ++sh) for (long T : Ts)
  for (int mc = 1; mc <= 16; mc *= 2) for (int fc = 0; fc <= 16; fc = fc ? fc * 2 : 1) {
    if (K == 0 && !sh) continue;
    ClusterPlan p;
    if (!plan_cluster_rows(R, K, H, sh, mc, T, 152, &p, fc)) continue;
    ++checks;
    if (fc && p.C != fc) { ++fails; if (fails < 20) printf("BAD one-shot forced C=%d got %d\n", fc, p.C); }
    const int chunks = H / 8, NT = (sh ? R : 0) + R * K;
    bool bad = false;
    if (p.C < 1 || p.C > mc || p.threads != p.nch * p.G || p.threads > 768) bad = true;
    if ((long)p.nch * p.C < chunks || p.nch > chunks) bad = true;                // every chunk has a CTA
    if ((long)p.G * p.maxt < NT || (p.maxt != 2 && p.maxt != 8)) bad = true;     // every term has a load slot
    if (p.smem != (p.G - 1) * 2 * p.nch * 16) bad = true;
    // the 64-register form: chosen only for eight-load plans of at most 512
    // threads that do not fit one wave of the 80-register form (register
    // counts 80 and 64, 65536 registers and 2048 threads per SM)
    {
      auto blocks = [&](int regs) {
        const int warps = (p.threads + 31) / 32;
        const int by_regs = 65536 / (warps * ((regs * 32 + 255) / 256 * 256));
        return std::min(by_regs, 2048 / p.threads);
      };
      const int b80 = blocks(80), b64 = blocks(64);
      const bool use64 = oneshot_prefer_64(p, T, 152, b80, b64);
      if (use64 && (p.maxt != 8 || p.threads > 512 || T * p.C <= (long)b80 * 152 || b64 <= b80)) bad = true;
      if (!use64 && p.maxt == 8 && p.threads <= 512 && T * p.C > (long)b80 * 152 && b64 > b80) bad = true;
      if (use64) ++n64;
    }
    if (bad) { ++fails; if (fails < 20) printf("BAD oneshot H=%d R=%d K=%d sh=%d T=%ld mc=%d\n", H, R, K, sh, T, mc); }
  }
  // show the automatic plans for the workloads
  struct W { const char* n; int R, K, H; bool sh; long T[8]; } ws[] = {
    {"ar_only", 2, 0, 7168, true, {1, 2, 4, 8, 16, 32, 64, 128}},
    {"dsv3", 8, 8, 7168, true, {1, 4, 16, 64, 128, 0}},
    {"glm", 8, 8, 6144, true, {1, 2, 4, 8, 16, 0}},
    {"prefill", 8, 10, 8192, true, {512, 2048, 8192, 0}}};
  for (auto& w : ws) for (long T : w.T) { if (!T) break; StreamPlan p; bool ok = plan_stream_rows(w.R, w.K, w.H, w.sh, T, 152, 232448, 16, 0, 0, &p);
      printf("%-8s T=%5ld ok=%d C=%2d tile=%4d cpt=%d thr=%3d nst=%3d P=%2d slot=%5d smem=%6d grid=%4d\n", w.n, T, ok, p.geo.C, p.geo.tile_chunks, p.cpt, p.threads, p.geo.nstages, p.geo.seg_per_stage, p.geo.slot_bytes, p.smem, p.grid); }
  if (n64 == 0) { ++fails; printf("the 64-register one-shot form is never chosen\n"); }
  {
    // eight partials, K = 0, H = 7168: the 80-register form up to one wave,
    // the 64-register form at T = 128 and 256
    ClusterPlan p;
    for (long T : {16L, 128L, 256L}) {
      if (!plan_cluster_rows(8, 0, 7168, true, 16, T, 152, &p)) { ++fails; continue; }
      const int warps = (p.threads + 31) / 32;
      const int b80 = std::min(65536 / (warps * 2560), 2048 / p.threads), b64 = std::min(65536 / (warps * 2048), 2048 / p.threads);
      const bool use64 = oneshot_prefer_64(p, T, 152, b80, b64);
      printf("oneshot R=8 K=0 H=7168 T=%ld C=%d threads=%d -> %s\n", T, p.C, p.threads, use64 ? "64-register form" : "80-register form");
      if (use64 != (T >= 128)) { ++fails; printf("unexpected form at T=%ld\n", T); }
    }
  }
  // the two-round switch: only when one-round clusters are fewer than the
  // rows and the two-round form holds more
  {
    struct Case { long T; int n1, n2; bool want; };
    const Case cases[] = {{8, 7, 14, true}, {7, 7, 14, false}, {8, 7, 7, false}, {8, 7, 6, false},
                          {16, 7, 14, true}, {1, 7, 14, false}, {8, 0, 14, false}};
    for (const Case& c : cases)
      if (split_prefer_two_rounds(c.T, c.n1, c.n2) != c.want) {
        ++fails;
        printf("two-round switch T=%ld n1=%d n2=%d: expected %d\n", c.T, c.n1, c.n2, (int)c.want);
      }
    // the heavy-row shape that needs it: R = 16, K = 10, H = 8192
    SplitPlan p1, p2;
    const bool ok1 = plan_split_rows(16, 10, 8192, true, 8, 152, 232448, 16, 16, &p1, 0, 1);
    const bool ok2 = plan_split_rows(16, 10, 8192, true, 8, 152, 232448, 16, 16, &p2, 0, 2);
    printf("split R=16 K=10 H=8192 C=16: one round %s (groups %d, %d B), two rounds %s (groups %d, %d B)\n",
           ok1 ? "ok" : "none", ok1 ? p1.geo.C / p1.geo.Cs : 0, ok1 ? p1.smem : 0, ok2 ? "ok" : "none",
           ok2 ? p2.geo.C / p2.geo.Cs : 0, ok2 ? p2.smem : 0);
    // two rounds must fit two CTAs per SM there (1 KB reserved per CTA)
    if (!ok1 || !ok2 || 2 * (p2.smem + 1024) > 233472) { ++fails; printf("unexpected heavy-row split plans\n"); }
  }
  printf("checked %ld plans, %ld bad\n", checks, fails);
  return fails != 0;
}

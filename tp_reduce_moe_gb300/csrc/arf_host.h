// arf_host.h -- host side of the kernel family: launch plans, planners,
// launchers and occupancy queries (no device code; the kernels' own
// parameters are in arf_common.cuh).
#pragma once

#include "arf_common.cuh"

namespace arf {

struct ClusterPlan {
    int C;    // CTAs per row (cluster size)
    int nch;  // 16-byte column chunks per CTA
    int G;    // thread groups splitting the term list
    int threads;
    int smem;  // dynamic shared memory bytes
    int maxt;  // loads per thread the kernel instantiation holds: 2, 8, or
               // kClusterMaxTerms64 (eight in a 64-register form)
};
constexpr int kClusterMaxTerms64 = 9;

// Kernel plan for the small-T regime; returns false if (R, K, H, shared) has
// no launchable plan with a cluster of at most max_c CTAs.  T and the SM count
// set how many CTAs per row are worth using.
// force_c > 0: exactly that cluster size (a power of two up to 16), else no plan.
bool plan_cluster_rows(int R, int K, int H, bool shared, int max_c, int64_t T, int num_sms,
                       ClusterPlan* p, int force_c = 0);
int cluster_rows_max_cluster(int threads, int smem, bool res_f32);
cudaError_t launch_cluster_rows(const RowArgs& a, const ClusterPlan& p, bool res_f32,
                                cudaStream_t stream, bool pdl = false);
cudaError_t cluster_rows_set_attributes();
bool cluster_rows_plan_fits(const ClusterPlan& p, bool res_f32);
int cluster_rows_blocks_per_sm(const ClusterPlan& p, bool res_f32);
bool oneshot_prefer_64(const ClusterPlan& p, int64_t T, int num_sms, int blocks80, int blocks64);

// The all-reduce + mHC write-back (mhc_post.cu).
cudaError_t launch_mhc_post(const MhcArgs& a, cudaStream_t stream, bool pdl = false);

struct StreamPlan {
    StreamGeom geo;
    int cpt;          // 16-byte chunks per consumer thread
    int threads;      // producer warps + consumer warps
    int smem;         // dynamic shared memory bytes
    int grid;         // CTAs (a multiple of C)
};

// Plan a stream_rows launch for T rows.  C = 0 picks the CTAs per row from T
// and the SM count; C >= 1 forces it.  stage_bytes = 0 picks the slot size,
// otherwise it is the target.  producers = 0 picks the producer warps (up to
// four), otherwise it is the cap.  max_tail_parts >= 2 lets whole-row plans
// (C = 1) split the rows of a last, partial wave over up to that many CTAs
// each (their partial rows meet in a workspace scratch of num_sms rows of H
// fp32 and num_sms counters); 0 or 1 never splits.  Returns false if no plan
// fits.
constexpr int kMaxTailParts = 8;
bool plan_stream_rows(int R, int K, int H, bool shared, int64_t T, int num_sms, int smem_optin,
                      int max_cluster, int C, int stage_bytes, StreamPlan* p, int producers = 0,
                      int max_tail_parts = 0);
cudaError_t launch_stream_rows(const RowArgs& a, const StreamPlan& p, bool res_f32,
                               cudaStream_t stream, bool pdl = false);
cudaError_t stream_rows_set_attributes(int smem_optin);
// Largest cluster (<= 16) co-schedulable for a clustered plan of this shape.
int stream_rows_max_cluster(int threads, int smem, int cpt);
bool stream_rows_plan_fits(const StreamPlan& p, bool res_f32);
// Clusters of a clustered plan the device co-schedules (0: query failed).
int stream_rows_active_clusters(const StreamPlan& p, bool res_f32);

struct SplitPlan {
    SplitGeom geo;
    int cpt;
    int threads;
    int smem;
    int grid;
};

// Plan a split_rows launch (one row per cluster); C = 0 picks the largest
// cluster that fits; `groups` column groups per row (they must divide C; 0
// picks the most that fit); `rounds` 1 buffers all of a CTA's segments at
// once, 2 fetches the second routed half into the first half's buffers once
// those are folded (half the shared memory, one more round trip).  Returns
// false if no plan fits.
bool plan_split_rows(int R, int K, int H, bool shared, int64_t T, int num_sms, int smem_optin,
                     int max_cluster, int C, SplitPlan* p, int groups = 1, int rounds = 1);
cudaError_t launch_split_rows(const RowArgs& a, const SplitPlan& p, bool res_f32,
                              cudaStream_t stream, bool pdl = false);
cudaError_t split_rows_set_attributes(int smem_optin);
int split_rows_max_cluster(int threads, int smem, int cpt);
bool split_rows_plan_fits(const SplitPlan& p, bool res_f32);
// Clusters of a split plan the device holds at once (0 if the query fails).
int split_rows_active_clusters(const SplitPlan& p, bool res_f32);
// Whether T rows should run the two-round form of a split plan, given the
// co-resident clusters of its one-round form (n1) and two-round form (n2):
// only when the one-round launch does not fit one wave and the two-round
// form holds more clusters.
bool split_prefer_two_rounds(int64_t T, int n1, int n2);

}  // namespace arf

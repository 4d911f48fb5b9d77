/*
 * arfuse.h -- C ABI of libarfuse: the fused decode-layer boundary op for one
 * GB300 (sm_103a) GPU.
 *
 * For every token row t (0 <= t < T) and column j (0 <= j < H) the library
 * computes, accumulating in fp32:
 *
 *   y[t,j]   = sum_{r<R} ( sum_{k<K} w[t,k] * E_r[perm[t,k], j]  +  S_r[t,j] )
 *   h[t,j]   = y[t,j] + residual[t,j]                       -> residual_out
 *   out[t,j] = h[t,j] * rsqrt( (1/H) sum_j h[t,j]^2 + eps ) * (gamma[j] + weight_bias)
 *
 * i.e. the MoE finalize (weighted gather of the permuted expert-output rows
 * back to token order), the shared-expert add, the arithmetic of the
 * post-experts tensor-parallel all-reduce over R rank partials that all sit
 * in this GPU's memory, the residual add and the next layer's input RMSNorm,
 * in one launch.
 *   - The fold of finalize + shared add + all-reduce into the next input norm:
 *     sglang PR #37196 "[Comm] Share the CuTe DSL AR fusion core and wire it
 *     for DeepSeek-V3 / GLM-5.x", Motivation.
 *   - The (gamma + weight_bias) scale, with weight_bias = 0 both for plain
 *     RMSNorm weights and for Gemma-style weights stored as checkpoint + 1:
 *     same page, Modifications section 1.
 *   - S_r added without a gate, once per rank partial (a replicated shared
 *     expert must not be passed as a partial): same page, Modifications
 *     section 2.
 *   - The K = 0 form (trailing all-reduce + residual RMSNorm), the mandatory
 *     residual and the clean decline that lets the caller run its own split
 *     path: sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with
 *     final RMSNorm", Changes.
 *   - One workspace per model, shared by its layers and fixed per
 *     hidden / top_k / eps; calls capturable in a CUDA graph: sglang PR
 *     #37196, Modifications section 2, and sglang PR #37104, Correctness.
 *
 * Conventions for every entry point below:
 *   - "device" pointers point into memory of the workspace's GPU; "host"
 *     pointers point into ordinary host memory and are read during the call
 *     only (the library keeps no reference to them after it returns).
 *   - The caller owns every tensor.  The library owns only the workspace.
 *   - Layouts are dense row-major with no padding; bf16 is IEEE bfloat16.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = the legacy default stream).  They never allocate, free or
 *     synchronise, so they can be captured in a CUDA graph.  The caller's
 *     current device must be the workspace's device.
 *   - The returned status covers host-side validation and the launch only.
 *     Any status other than AR_OK means nothing was launched: the caller can
 *     fall back to its own unfused path.
 *   - Device-side problems (a perm value outside [0, rows_e); a pipeline wait
 *     that ran past its time limit) never fault: the kernel clamps or gives
 *     up, records a bit in the workspace's error word and still returns;
 *     read it with ar_workspace_device_error() after synchronising.
 */
#ifndef ARFUSE_H
#define ARFUSE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ARFUSE_API __attribute__((visibility("default")))
#else
#define ARFUSE_API
#endif

/* Limits of the library. */
#define AR_MAX_RANKS 16      /* R: rank partials per call            */
#define AR_MAX_TOP_K 16      /* K: routed experts per token          */
#define AR_MAX_HIDDEN 16384  /* H: columns per row (multiple of 8)   */

typedef enum ar_status {
    AR_OK = 0,
    AR_ERR_INVALID_ARG = 1,  /* NULL / inconsistent / overlapping arguments   */
    AR_ERR_ALIGNMENT = 2,    /* a pointer not 16-byte aligned, or H % 8 != 0   */
    AR_ERR_UNSUPPORTED = 3,  /* outside the library's limits or launch plans  */
    AR_ERR_CAPACITY = 4,     /* T larger than the workspace's max_tokens       */
    AR_ERR_CUDA = 5,         /* a CUDA runtime call or the launch failed      */
    AR_ERR_DEVICE_CHECK = 6, /* a device-side check fired (see device_error)  */
    AR_VALIDATED = 7         /* dry-run workspace: arguments valid, no launch */
} ar_status;

/* ar_workspace_create() flags. */
#define AR_WS_DRY_RUN 0x1u      /* no GPU state: calls validate, then return AR_VALIDATED   */
#define AR_WS_NORM_BF16_H 0x2u  /* the norm reads h rounded to bf16, as a bf16 residual_out  */
                                /* stores it (default: the unrounded fp32 sum)              */
#define AR_WS_PDL 0x4u          /* launch with programmatic dependent launch (see below)      */

/* Bits of the device error word (ar_workspace_device_error). */
#define AR_DEVERR_PERM_RANGE 0x1   /* some perm value was outside [0, rows_e); clamped */
#define AR_DEVERR_TIMEOUT 0x2      /* a pipeline wait gave up after its time limit     */

/* Kernel regimes (ar_workspace_set_regime / ar_workspace_last_regime). */
#define AR_REGIME_AUTO 0     /* pick by (T, R, K, H) and the SM count                    */
#define AR_REGIME_CLUSTER 1  /* small T: each row split into column tiles over a cluster  */
                             /* of C CTAs, each streaming its tile through a bulk-copy    */
                             /* ring; sum of squares exchanged in distributed smem        */
#define AR_REGIME_STREAM 2   /* large T: persistent CTAs, whole rows through the ring     */
#define AR_REGIME_ONESHOT 3  /* one cluster per row, every load in flight at once from    */
                             /* registers, no pipeline (latency-optimal for tiny rows)    */
#define AR_REGIME_SPLIT 4    /* small T: one cluster per row, the row's segments dealt    */
                             /* to its C CTAs (in column groups), partial rows            */
                             /* reduce-scattered through distributed shared memory        */
                             /* (fewest copies per CTA); heavy rows in two copy rounds    */
                             /* through half the buffers when that fits more clusters     */

typedef struct ar_workspace ar_workspace;  /* opaque, library-owned */

/*
 * Create the workspace for one model: fixes ranks (R), top_k (K), hidden (H)
 * and eps, as the model's MoE layers share them.  Allocates its device memory
 * on `device` -- the error word, and a scratch of one fp32 row of H plus one
 * counter per SM for rows split over several CTAs (4.4 MB at H = 7168 on 152
 * SMs) -- and sets kernel attributes; call it once, outside any stream
 * capture.  A workspace serves one stream of calls at a time: calls that use
 * the same workspace must be ordered on the GPU (one stream, or event
 * ordering); concurrent callers need a workspace each.
 *   device      CUDA device ordinal (ignored with AR_WS_DRY_RUN)
 *   ranks       1 .. AR_MAX_RANKS
 *   top_k       0 .. AR_MAX_TOP_K (0: only ar_rmsnorm is meaningful)
 *   hidden      8 .. AR_MAX_HIDDEN, a multiple of 8
 *   max_tokens  largest T any call may pass (>= 1)
 *   eps         RMSNorm epsilon every call must repeat
 *   flags       0, or any of AR_WS_DRY_RUN, AR_WS_NORM_BF16_H, AR_WS_PDL.
 *               AR_WS_PDL launches the kernels with programmatic dependent
 *               launch (cudaLaunchAttributeProgrammaticStreamSerialization):
 *               the launch may begin while the previous kernel in the stream
 *               is still running, and the kernel waits (griddepcontrol.wait)
 *               for that kernel to complete and flush its memory before its
 *               first global memory access, so results and stream order are
 *               unchanged; launch latency overlaps the previous kernel.  The
 *               decode kernels signal their own dependents as soon as they
 *               start, the streaming kernel as each of its CTAs finishes
 *               (kernels launched without the attribute are not affected).  A
 *               clustered launch whose clusters fill every co-resident slot
 *               goes out without the attribute (the next kernel could not be
 *               placed before it drains).
 *   out         host pointer that receives the handle (set to NULL on error)
 * Errors: AR_ERR_INVALID_ARG (out NULL, max_tokens < 1, eps < 0 or not
 * finite), AR_ERR_ALIGNMENT (hidden % 8), AR_ERR_UNSUPPORTED (limits above,
 * or a device older than sm_100), AR_ERR_CUDA.
 */
ARFUSE_API ar_status ar_workspace_create(int device, int ranks, int top_k, int hidden,
                                         int64_t max_tokens, float eps, unsigned flags,
                                         ar_workspace** out);

/* Free the workspace.  NULL is accepted.  Synchronises nothing: the caller
 * must make sure no call using it is still running. */
ARFUSE_API ar_status ar_workspace_destroy(ar_workspace* ws);

/*
 * The fused op (routed + shared + rank sum + residual + RMSNorm).
 *   ws            workspace; R, K, H and eps must equal its values
 *   expert_out    host array [R] of device pointers, each bf16 [rows_e, H]:
 *                 rank r's expert outputs in permuted (expert-grouped) order
 *   rows_e        rows of every expert_out[r] (>= 1 when K > 0)
 *   perm          device int32 [T, K]: perm[t*K + k] is the row of every
 *                 expert_out[r] that holds token t's k-th routed expert
 *                 (a gather index; duplicates are allowed)
 *   topk_w        device fp32 [T, K] routing weights (any routed scaling
 *                 already folded in)
 *   shared_out    host array [R] of device pointers, each bf16 [T, H]: rank
 *                 r's shared-expert partial; or NULL for no shared term
 *   residual      device bf16 [T, H], required (NULL is AR_ERR_INVALID_ARG)
 *   gamma         device bf16 [H] norm weight
 *   weight_bias   added to gamma in fp32 (0 for plain and for Gemma weights
 *                 stored as checkpoint + 1)
 *   eps           must equal the workspace's eps
 *   T, R, K, H    tokens, rank partials, routed experts per token, hidden
 *   out           device bf16 [T, H]
 *   residual_out  device [T, H], bf16 or fp32 (see next); may be the same
 *                 pointer as residual when bf16 (in-place update)
 *   residual_out_is_fp32  0: bf16 residual_out, 1: fp32
 *   stream        cudaStream_t
 * K == 0 means no routed term; K == 0 with shared_out == NULL is
 * AR_ERR_INVALID_ARG (nothing to reduce).  T == 0 returns AR_OK at once.
 * Alignment: every data pointer 16-byte aligned, perm and topk_w 4-byte
 * aligned (else AR_ERR_ALIGNMENT).  out and residual_out must not overlap
 * each other or any input, except the exact in-place residual alias above
 * (else AR_ERR_INVALID_ARG).  T > max_tokens is AR_ERR_CAPACITY.
 */
ARFUSE_API ar_status ar_finalize_rmsnorm(ar_workspace* ws,
                                         const void* const* expert_out, int64_t rows_e,
                                         const int32_t* perm, const float* topk_w,
                                         const void* const* shared_out,
                                         const void* residual, const void* gamma,
                                         float weight_bias, float eps,
                                         int64_t T, int R, int K, int H,
                                         void* out, void* residual_out,
                                         int residual_out_is_fp32, void* stream);

/*
 * The fused op with a gated shared expert: as ar_finalize_rmsnorm, except that
 * each rank's shared partial of token t is scaled by sigmoid(shared_gate[t])
 * before the add (the Qwen-style shared expert carries such a per-token gate,
 * while the DeepSeek-V3 one adds unmodified: sglang PR #37196, Modifications
 * section 2).
 *   shared_gate  device fp32 [T] gate logits (4-byte aligned), required
 *   shared_out   required (a gate needs a shared term)
 * Errors as for ar_finalize_rmsnorm; a NULL shared_gate or shared_out is
 * AR_ERR_INVALID_ARG.
 */
ARFUSE_API ar_status ar_finalize_rmsnorm_gated(ar_workspace* ws,
                                               const void* const* expert_out, int64_t rows_e,
                                               const int32_t* perm, const float* topk_w,
                                               const void* const* shared_out,
                                               const float* shared_gate,
                                               const void* residual, const void* gamma,
                                               float weight_bias, float eps,
                                               int64_t T, int R, int K, int H,
                                               void* out, void* residual_out,
                                               int residual_out_is_fp32, void* stream);

/*
 * Trailing all-reduce + residual RMSNorm without a MoE term (the K = 0 form):
 * h = sum_r partials[r] + residual; out = RMSNorm(h).  `partials` is a host
 * array [R] of device pointers, each bf16 [T, H].  R and H must equal the
 * workspace's; its top_k is not used.  Everything else as for
 * ar_finalize_rmsnorm.
 */
ARFUSE_API ar_status ar_rmsnorm(ar_workspace* ws, const void* const* partials, int R,
                                const void* residual, const void* gamma,
                                float weight_bias, float eps, int64_t T, int H,
                                void* out, void* residual_out, int residual_out_is_fp32,
                                void* stream);

/*
 * Read and clear the workspace's device error word (AR_DEVERR_* bits) into
 * *code (host pointer).  Synchronises the workspace's device first.  Returns
 * AR_ERR_DEVICE_CHECK when a bit was set, AR_OK when none, AR_ERR_INVALID_ARG
 * for NULL arguments, AR_ERR_CUDA on a failed copy.  A set bit means the
 * fused call declined part of its work on the device (rows left unfinished
 * after a wait ran out, or clamped perm values): the caller still owes that
 * reduction and can rerun the step on its own unfused path, as a runtime
 * decline of the fused boundary must allow (sglang PR #37104 "perf(mtp): fuse
 * trailing TP all-reduce with final RMSNorm", Changes).  When a bit was set
 * the workspace's split-row counters are reset too, so the next call starts
 * clean.
 */
ARFUSE_API ar_status ar_workspace_device_error(ar_workspace* ws, int* code);

/*
 * Force a kernel regime (AR_REGIME_*) for later calls on this workspace, e.g.
 * to test both kernels at every T.  AR_REGIME_AUTO restores the tuned choice.
 * A forced regime that cannot run a given call makes that call return
 * AR_ERR_UNSUPPORTED.
 */
ARFUSE_API ar_status ar_workspace_set_regime(ar_workspace* ws, int regime);

/*
 * Force the number of CTAs per token row (the cluster size C, 2..16) that
 * AR_REGIME_CLUSTER, AR_REGIME_SPLIT and AR_REGIME_ONESHOT use (one-shot:
 * a power of two); 0 restores the automatic choice.  A size that cannot be
 * launched for a call makes that call return AR_ERR_UNSUPPORTED.
 */
ARFUSE_API ar_status ar_workspace_set_cluster_size(ar_workspace* ws, int ctas_per_row);

/*
 * Set the target size in bytes of one ring slot of the streaming kernels (a
 * slot holds as many whole row segments as fit, at least one, one bulk copy
 * each, all signalled on one mbarrier); 0 restores the automatic size
 * (64 KB).  Values outside 0 or
 * [1024, 131072] are AR_ERR_INVALID_ARG.  A tuning control: results are
 * identical for every value.
 */
ARFUSE_API ar_status ar_workspace_set_stage_bytes(ar_workspace* ws, int bytes);

/*
 * Cap the producer warps of the streaming kernels (1..4; 0 restores the
 * automatic count, up to four and at most one per ring slot).  Each producer
 * warp fills its own ring slots; the lanes of a bulk-copy instruction are
 * issued one after another, so more warps keep more slots in flight.
 * Other values are AR_ERR_INVALID_ARG.  A tuning control: results are
 * identical for every value.
 */
ARFUSE_API ar_status ar_workspace_set_producer_warps(ar_workspace* ws, int warps);

/*
 * Column groups per row of the split kernel (AR_REGIME_SPLIT): 1..8 (a
 * divisor of the cluster size; the last group may be narrower when G does not
 * divide the row's 16-byte chunks); 0 (the default) picks the most groups (a
 * power of two) that leave a plan, each group at least 128 16-byte chunks
 * wide.  With G groups the C CTAs of a row form G groups
 * of C/G; each group covers 1/G of the row's columns, its CTAs deal the row's
 * segments among themselves (bulk copies of 1/G of a row each) and
 * reduce-scatter only their group's columns, which cuts the distributed-
 * shared-memory exchange G-fold for G-fold more, smaller copies.  A forced
 * value that does not split the cluster into groups of at least two CTAs,
 * or deals a CTA more than 64 segments (32 per copy round), leaves the split
 * regime without a plan (AR_ERR_UNSUPPORTED when the regime is forced).  Other values are AR_ERR_INVALID_ARG.  A tuning control:
 * residual_out equals, bit for bit, that of a split over C/G CTAs without
 * groups (the same segments per CTA, the same slice order); out differs from
 * it only through the summation order of the tile sums of squares.
 */
ARFUSE_API ar_status ar_workspace_set_split_column_groups(ar_workspace* ws, int groups);

/*
 * Cap the split of whole-row streaming (AR_REGIME_STREAM) over its last,
 * partial wave: with T mod SMs = n > 0 rows left for the last wave, each of
 * those rows is split into up to m = min(max_parts, SMs / n, segments / 8)
 * segment intervals on m CTAs, whose fp32 partial rows meet in the workspace scratch;
 * the CTA that brings the last part sums the parts in part order and finishes
 * the row (no CTA waits for another).  max_parts 0 or 1 never splits; 2 ..
 * AR_MAX_SPLIT_PARTS caps m (default AR_MAX_SPLIT_PARTS).  Other values are
 * AR_ERR_INVALID_ARG.  A split row's fp32 sum runs in another order than an
 * unsplit one, so results move within rounding (deterministic for a given
 * setting, T and GPU).
 */
#define AR_MAX_SPLIT_PARTS 8
ARFUSE_API ar_status ar_workspace_set_split_rows(ar_workspace* ws, int max_parts);

/*
 * Failure injection for tests of the device-side timeout path (the clean
 * decline of sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with
 * final RMSNorm", Changes: a fused call that gives up must leave the caller
 * able to finish the reduction itself).  With limit_ns > 0, later calls on
 * this workspace that run whole-row streaming (AR_REGIME_STREAM) make every
 * consumer warp's first wait target a barrier that nothing arrives on, bounded
 * by limit_ns nanoseconds: the wait runs out, the kernel records
 * AR_DEVERR_TIMEOUT in the error word, skips its remaining waits (its rows are
 * left unfinished: out and residual_out of that call are undefined), waits for
 * its own bulk copies still in flight and returns.  Nothing faults or hangs.
 * Calls in any other regime return AR_ERR_UNSUPPORTED while it is set (force
 * AR_REGIME_STREAM with ar_workspace_set_regime).  limit_ns = 0 turns it off;
 * values outside [0, 1e9] are AR_ERR_INVALID_ARG.
 */
ARFUSE_API ar_status ar_workspace_inject_wait_timeout(ar_workspace* ws, int64_t limit_ns);

/* Regime (AR_REGIME_CLUSTER / _STREAM / _ONESHOT / _SPLIT) of the last
 * launched call (on a dry-run workspace: of the last validated call), 0
 * before the first one.  *ctas receives the CTAs per row
 * (cluster, one-shot and split regimes) or the persistent grid size (stream
 * regime); may be NULL. */
ARFUSE_API int ar_workspace_last_regime(const ar_workspace* ws, int* ctas);

/* CTAs launched by the last launched call (on a dry-run workspace: planned
 * for the last validated call), 0 before the first one or for NULL.  For a
 * clustered streaming plan this is the grid after it was capped at the
 * clusters the device co-schedules (a multiple of the CTAs per row). */
ARFUSE_API int ar_workspace_last_grid(const ar_workspace* ws);

/* The launch plan of the last launched call (on a dry-run workspace: of the
 * last validated call, planned without the device's occupancy queries, so
 * without their grid cap and form switches): which of the kernel forms the
 * per-shape choice picked (the crossovers between the fused operator's
 * algorithms move with the shape: sglang PR #37196, Known gaps).  All zero
 * before the first call.  Fields a regime does not use are 0. */
typedef struct ar_plan_info {
    int32_t regime;          /* AR_REGIME_CLUSTER / _STREAM / _ONESHOT / _SPLIT            */
    int32_t ctas_per_row;    /* as ar_workspace_last_regime                                */
    int32_t grid;            /* CTAs launched (as ar_workspace_last_grid)                  */
    int32_t block;           /* threads per CTA                                           */
    int32_t smem_bytes;      /* dynamic shared memory per CTA                             */
    int32_t column_groups;   /* split: column groups per row                              */
    int32_t copy_rounds;     /* split: 1, or 2 (second routed half into reused buffers)   */
    int32_t ring_slots;      /* cluster / stream: bulk-copy ring slots per CTA            */
    int32_t ring_slot_bytes; /* cluster / stream: bytes per ring slot                     */
    int32_t producer_warps;  /* cluster / stream: producer warps; split: 1                */
    int32_t loads_per_thread; /* one-shot: register loads a thread holds (2 or 8)         */
} ar_plan_info;

/* Copy the last call's plan into *info.  AR_ERR_INVALID_ARG for NULL. */
ARFUSE_API ar_status ar_workspace_last_plan(const ar_workspace* ws, ar_plan_info* info);

/*
 * Regime table: the kernel regime (and CTAs per row) that AR_REGIME_AUTO runs
 * at each token count.  The fastest regime depends on T and on the shape, and
 * crossovers measured at one hidden size do not carry over to another
 * (sglang PR #37196 "[Comm] Share the CuTe DSL AR fusion core and wire it for
 * DeepSeek-V3 / GLM-5.x", Known gaps and Related: the shipped bounds did not
 * transfer from H = 8192 to H = 6144, so tuning is per shape).
 *
 * A table is at most AR_MAX_REGIME_RULES rules with strictly ascending
 * max_tokens >= 1; a call with T tokens takes the first rule with
 * T <= max_tokens.  regime is AR_REGIME_CLUSTER, _STREAM, _ONESHOT or _SPLIT,
 * or AR_REGIME_AUTO for the built-in heuristic over that range; ctas_per_row
 * is 0 (the regime's own choice) or, for the cluster, split and one-shot
 * regimes, 2..16 (one-shot: a power of two, else the rule has no plan);
 * stage_bytes and producer_warps are 0 (the workspace's setting, see
 * ar_workspace_set_stage_bytes / _set_producer_warps) or, for the cluster and
 * stream regimes, the ring-slot size (1024..131072) and the producer-warp cap
 * (1..4) of that rule -- smaller slots and fewer producer warps let more
 * CTAs of a clustered plan reside per SM, which wins at some T and loses at
 * others, so the tuner measures them per shape.  A call past the last rule, or one whose rule has no launch plan for
 * it (a cluster size the device cannot co-schedule, a row too long for the
 * split kernel), runs the heuristic.  A regime forced with
 * ar_workspace_set_regime takes precedence over the table.  Every regime
 * meets the same accuracy bound; each sums in its own fixed order, so a
 * table changes results only within rounding, and a given table gives the
 * same bits on every call.
 *
 * ar_workspace_create installs a table measured on GB300 when (ranks, top_k,
 * hidden) is one of the shapes the library carries one for, else none.
 * ar_workspace_set_regime_table replaces it (rules: host array of n rules,
 * copied; n = 0 removes the table).  An invalid table is AR_ERR_INVALID_ARG
 * and leaves the previous one in place.  ar_workspace_get_regime_table copies
 * up to cap rules into rules (host) and stores the table's length in *n
 * (rules may be NULL when cap is 0).  The Python module
 * tp_reduce_moe_gb300.tune measures a table for any shape on the GPU at hand.
 */
typedef struct ar_regime_rule {
    int64_t max_tokens;
    int32_t regime;          /* AR_REGIME_* */
    int32_t ctas_per_row;    /* 0, or 2..16 for AR_REGIME_CLUSTER / _SPLIT / _ONESHOT */
    int32_t stage_bytes;     /* 0, or 1024..131072 for AR_REGIME_CLUSTER / AR_REGIME_STREAM */
    int32_t producer_warps;  /* 0, or 1..4 for AR_REGIME_CLUSTER / AR_REGIME_STREAM */
} ar_regime_rule;
#define AR_MAX_REGIME_RULES 32
ARFUSE_API ar_status ar_workspace_set_regime_table(ar_workspace* ws, const ar_regime_rule* rules,
                                                   int n);
ARFUSE_API ar_status ar_workspace_get_regime_table(const ar_workspace* ws, ar_regime_rule* rules,
                                                   int cap, int* n);

/*
 * ar_mhc_post -- the all-reduce + mHC residual write-back ("hc_post") in one
 * launch.  sglang PR #42020 (Summary and Scope): an mHC layer writes its FFN
 * output back as the FFN's tensor-parallel all-reduce followed by hc_post,
 * which reads the reduced output back and mixes it into the hc_mult (four)
 * residual streams; the fused kernel does both in one pass.  The page gives
 * no formula for the mix, so parity of this entry point is unpinned: its
 * oracle fixes only this library's reading of the page, the per-token linear
 * mix
 *
 *   y[t,j]     = sum_{r<R} partials[r][t,j]                       (fp32)
 *   out[t,i,j] = post[t,i] * y[t,j] + sum_{k<hc} comb[t,i,k] * streams[t,k,j]
 *
 * rounded once to bf16.
 *   ws            a workspace whose ranks equals R and hidden equals H (its
 *                 top_k and eps are not used); T <= its max_tokens.
 *   partials      host array[R] of device pointers, bf16 [T, H], 16-byte aligned.
 *   streams       device bf16 [T, hc, H]: the incoming residual streams.
 *   post          device fp32 [T, hc]; comb device fp32 [T, hc, hc] (row i
 *                 mixes the incoming streams into outgoing stream i); 4-byte
 *                 aligned.
 *   hc            1 .. AR_MAX_HC_STREAMS.
 *   streams_out   device bf16 [T, hc, H], 16-byte aligned; may be `streams`
 *                 itself (in place), otherwise it must not overlap any input.
 * T == 0 returns AR_OK without a launch.  Errors as for ar_rmsnorm; nothing
 * is launched unless AR_OK is returned.
 */
#define AR_MAX_HC_STREAMS 8
ARFUSE_API ar_status ar_mhc_post(ar_workspace* ws, const void* const* partials, int R,
                                 const void* streams, const float* post, const float* comb,
                                 int64_t T, int H, int hc, void* streams_out, void* stream);

/*
 * ar_finalize_rmsnorm_noalloc -- the fused op for callers that cannot allocate
 * device memory.  (No counterpart on the pages: an addition of this library.)
 *
 * Some callers may not call cudaMalloc at all -- code that runs while an
 * engine captures a CUDA graph, plugins whose host engine owns every byte of
 * device memory through its own pool, deployments with a fixed memory budget
 * -- and ar_workspace_create() allocates a small device block.  This entry
 * point needs no workspace and allocates nothing (no cudaMalloc, no cudaFree,
 * no allocating library routine): the kernels' only global memory beyond the
 * caller's inputs and outputs, the 4-byte device status word, lives in a
 * fixed 256-byte array inside this library (kept by every GPU that loads the
 * library until the process exits).  The caller still passes every input and
 * output, with the arguments, layouts, alignment rules and limits of
 * ar_finalize_rmsnorm(); R, K, H and eps are taken from the call.  Sizes
 * beyond the limits are rejected before anything runs: R > AR_MAX_RANKS or
 * K > AR_MAX_TOP_K (AR_ERR_INVALID_ARG), H outside [8, AR_MAX_HIDDEN]
 * (AR_ERR_UNSUPPORTED), T > 2^26 (AR_ERR_CAPACITY).  The status word needs 4
 * bytes for any size, so the array's 256 bytes always suffice.
 *
 *   - The first call on a device (the current device) does a one-time set-up
 *     there: kernel attributes and the device address of the array; the first
 *     call with each new (R, K, H) also measures that shape's launch limits on
 *     the host.  Make those first calls before any stream capture on that
 *     device.
 *   - The plans are those of ar_finalize_rmsnorm() on a workspace of the same
 *     shape, with one difference: without a workspace's split-row scratch,
 *     whole-row streaming never splits the rows of its last, partial wave
 *     over idle CTAs (so at T mod SMs > 0 a call can be slower than the
 *     workspace entry point's).  A plan the device cannot co-schedule is
 *     declined as AR_ERR_UNSUPPORTED before anything is launched.
 *   - Device-side check results (a clamped perm value, a wait past its time
 *     limit) are OR-ed into the status word, which this entry point neither
 *     clears nor reads: check perm ranges on the host where they matter, or
 *     use a workspace.
 *   - Every call shares the array: calls that overlap on the GPU (on
 *     different streams, without ordering between them) race on the status
 *     word.  Their outputs are unaffected.
 */
ARFUSE_API ar_status ar_finalize_rmsnorm_noalloc(const void* const* expert_out, int64_t rows_e,
                                                 const int32_t* perm, const float* topk_w,
                                                 const void* const* shared_out,
                                                 const void* residual, const void* gamma,
                                                 float weight_bias, float eps, int64_t T, int R,
                                                 int K, int H, void* out, void* residual_out,
                                                 int residual_out_is_fp32, void* stream);

/* Static description of a status code; never NULL.  Every status other than
 * AR_OK / AR_VALIDATED is a clean decline: nothing was launched and the
 * caller runs its own split path (sglang PR #37104 "perf(mtp): fuse trailing
 * TP all-reduce with final RMSNorm", Changes). */
ARFUSE_API const char* ar_status_string(ar_status s);

#ifdef __cplusplus
}
#endif

#endif /* ARFUSE_H */

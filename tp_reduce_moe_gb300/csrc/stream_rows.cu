// stream_rows.cu -- the streaming kernel family of libarfuse.
//
// Per token row the op reads nseg = R*(K+1)+1 contiguous rows of H bf16 (R
// shared partials, the residual, R*K gathered expert rows) and writes two.
// Each CTA owns a column tile of every row it processes -- the whole row
// (C = 1, large T) or one of C tiles of the row, the C CTAs forming one
// thread-block cluster (C = 2..16, small T) -- and streams its tile of the
// row's nseg segments through a ring of shared-memory slots:
//
//   * producer warps issue one 1-D bulk async copy per segment
//     (cp.async.bulk, the TMA engine's untiled form, L2 evict-first), the
//     copies of one slot from the lanes of one instruction, completion
//     counted as transaction bytes on the slot's `full` mbarrier.  Issue is
//     costed per copy, not per byte (measured on GB300: 60-160 cycles a copy
//     whatever its size from 0.9 to 14 KB, the lanes of one instruction
//     issued one after another, about one copy per 70 cycles per SM), and
//     one producer warp alone kept too few slots in flight; W producer warps
//     take the slots round-robin;
//   * consumer warps fold each landed slot into fp32 accumulators held in
//     registers (CPT 16-byte chunks per thread, U segments per step with
//     their shared-memory loads issued together and no per-segment guards),
//     then release it on the slot's `empty` mbarrier;
//   * after a row's last segment the consumers finish the row on chip: store
//     residual_out, reduce the sum of squares (warp shuffle + one named
//     barrier), and -- for tiles -- push the CTA's partial into every peer's
//     shared memory as an asynchronous remote store (st.async, distributed
//     shared memory) counted as transaction bytes on the peer's barrier,
//     then scale by rsqrt(mean + eps) * (gamma + weight_bias) and store out.
//     The ring keeps streaming the next row meanwhile.
//
// Every input byte is read once and every output byte written once.  Rows
// go round-robin over persistent CTAs (C = 1) or clusters (C > 1).  With
// programmatic dependent launch a CTA lets the next kernel launch only as it
// finishes: its grid fills the GPU, and dependents made resident early cost
// the running call up to 0.9 us (dsv3 T = 160-192).
//
// Every wait is bounded (arf::mbar_wait_bounded): a wait that runs out sets
// the workspace error word and an abort flag, later waits are skipped (rows
// are left unfinished, never hung), and the producer waits (bounded again)
// for its own copies in flight before the CTA exits.  A clustered CTA needs
// no exit barrier: it leaves only after every peer's partial of its last row
// has arrived, so no peer writes into it afterwards (after an abort it waits
// a bounded grace period instead).
//
// Operation: sglang PR #37196 "[Comm] Share the CuTe DSL AR fusion core and
// wire it for DeepSeek-V3 / GLM-5.x", Motivation and Modifications sections
// 1-2; sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with final
// RMSNorm", Changes.
#include <type_traits>

#include "arf_host.h"

namespace arf {

constexpr int kStreamMaxConsumers = 512;
constexpr int kStreamMaxProducers = 4;
constexpr int kStreamMaxThreads = 32 * kStreamMaxProducers + kStreamMaxConsumers;
constexpr int kStreamMaxStages = 128;
constexpr int kMaxCluster = 16;
constexpr int kMinPartSegs = 8;  // segments per part of a split row, at least

// Shared-memory header: full[n], empty[n], xbar[2] mbarriers; xslot[2][16]
// (pushed partial sums of squares), red[2][32] (per-warp partials), the abort
// flag, rec[n] (0: slot never filled, 1 + parity of its latest fill); the
// ring follows at a 128-byte boundary.
__host__ __device__ constexpr int stream_ring_offset(int nstages) {
    return (nstages * 16 + 16 + 2 * kMaxCluster * 4 + 2 * 32 * 4 + 16 + nstages + 127) / 128 * 128;
}

// Slot and parity of ring position q (0 <= q < 2 * nstages).
__device__ __forceinline__ void ring_pos(int q, int nst, int& slot, uint32_t& parity) {
    parity = q >= nst ? 1u : 0u;
    slot = parity ? q - nst : q;
}

// Stages of one row: first the nsr = nS + 1 segments that need no routing
// metadata (shared partials, residual) in stages of at most P, then the R*K
// routed segments in stages of at most P.  Stage j covers segments
// [s0, s0 + cnt).
__device__ __forceinline__ void stage_range(int j, int P, int nsr, int nseg, int& s0, int& cnt) {
    const int first = (nsr + P - 1) / P;
    if (j < first) {
        s0 = j * P;
        cnt = min(P, nsr - s0);
    } else {
        s0 = nsr + (j - first) * P;
        cnt = min(P, nseg - s0);
    }
}

// Stages of the segment interval [a, b) of a split row: its perm-free
// segments (s < nsr) in stages of at most P, then its routed ones.
__device__ __forceinline__ int part_stage_count(int P, int nsr, int a, int b) {
    const int lo = min(b, nsr) - a, hi = b - max(a, nsr);
    return (lo > 0 ? (lo + P - 1) / P : 0) + (hi > 0 ? (hi + P - 1) / P : 0);
}
__device__ __forceinline__ void part_stage_range(int j, int P, int nsr, int a, int b, int& s0, int& cnt) {
    const int lo = min(b, nsr) - a;
    const int first = lo > 0 ? (lo + P - 1) / P : 0;
    if (j < first) {
        s0 = a + j * P;
        cnt = min(P, min(b, nsr) - s0);
    } else {
        s0 = max(a, nsr) + (j - first) * P;
        cnt = min(P, b - s0);
    }
}

// acc[m] += sum over the slot's cnt segments of coef[i] * segment i's chunk
// lch[m] (for valid[m]): full steps of U segments, loads first, with no
// per-segment guards (the instruction count bounds this loop), then the
// remaining segments one at a time; the same sequential order per column.
template <int CPT, int U>
__device__ __forceinline__ void fold_slot(float (&acc)[CPT][8], const float* coef, const uint8_t* seg,
                                          size_t seg_stride, int cnt, const int (&lch)[CPT],
                                          const bool (&valid)[CPT]) {
    const uint8_t* src[CPT];
#pragma unroll
    for (int m = 0; m < CPT; ++m) src[m] = seg + (size_t)lch[m] * 16;
    int i0 = 0;
    for (; i0 + U <= cnt; i0 += U) {
        float cf[U];
        uint4 v[U][CPT];
#pragma unroll
        for (int u = 0; u < U; ++u) cf[u] = coef[i0 + u];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int m = 0; m < CPT; ++m)
                if (valid[m]) v[u][m] = *reinterpret_cast<const uint4*>(src[m] + (size_t)(i0 + u) * seg_stride);
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int m = 0; m < CPT; ++m)
                if (valid[m]) fma_bf16x8(acc[m], cf[u], v[u][m]);
    }
    for (; i0 < cnt; ++i0) {
        const float cf = coef[i0];
#pragma unroll
        for (int m = 0; m < CPT; ++m)
            if (valid[m]) fma_bf16x8(acc[m], cf, *reinterpret_cast<const uint4*>(src[m] + (size_t)i0 * seg_stride));
    }
}

template <int CPT, int U, bool RES_F32, bool CLUSTERED>
__global__ void __launch_bounds__(kStreamMaxThreads, 1)
    stream_rows_kernel(const __grid_constant__ RowArgs a, const StreamGeom geo) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int nst = geo.nstages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + nst;
    uint64_t* xbar = empty + nst;                                 // [2]
    float* xslot = reinterpret_cast<float*>(xbar + 2);            // [2][kMaxCluster]
    float* red = xslot + 2 * kMaxCluster;                         // [2][32]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 64);
    volatile int* last_flag = reinterpret_cast<volatile int*>(red + 65);
    uint8_t* rec = reinterpret_cast<uint8_t*>(red + 68);          // [nst]
    uint8_t* ring = smem + stream_ring_offset(nst);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int W = geo.producers;             // producer warps 0..W-1
    const int ncw = (blockDim.x >> 5) - W;   // consumer warps
    const int C = CLUSTERED ? geo.C : 1;
    const uint32_t crank = CLUSTERED ? cluster_ctarank() : 0u;
    const int64_t first_row = blockIdx.x / C;
    const int64_t row_step = gridDim.x / C;
    const int H = a.H;
    const int chunk0 = (int)crank * geo.tile_chunks;  // first 16-byte chunk of this tile
    const int nchunk = min(geo.tile_chunks, H / 8 - chunk0);
    const uint32_t tile_bytes = (uint32_t)nchunk * 16u;
    const int nS = a.has_shared ? a.R : 0;
    const int nseg = nS + 1 + a.R * a.K;
    const int P = geo.seg_per_stage;
    const int nstage_row = (nS + 1 + P - 1) / P + (a.R * a.K + P - 1) / P;
    // Whole rows [0, main_rows) go round-robin; with split rows (C = 1 only)
    // each row of the last, partial wave is cut into `parts` segment
    // intervals, one per CTA (CTA b takes part b % parts of row
    // main_rows + b / parts), handled after the CTA's whole rows.
    const int64_t main_rows = CLUSTERED ? a.T : geo.main_rows;
    const int parts = CLUSTERED ? 1 : geo.tail_parts;
    const bool has_part = !CLUSTERED && parts > 1 && (int64_t)blockIdx.x < (a.T - main_rows) * parts;

    // The first row's routing metadata is requested before the barrier
    // set-up (producer lanes k < K, a load the compiler keeps in place), so
    // its memory round trip overlaps the set-up.
    pdl_wait();  // no global memory access before this point
    int32_t raw_first = 0;
    float w_first = 0.0f;
    if (warp < W && lane < a.K && first_row < main_rows) {
        raw_first = (int32_t)ld_early4(a.perm + first_row * a.K + lane);
        w_first = __uint_as_float(ld_early4(a.w + first_row * a.K + lane));
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), (uint32_t)ncw);
            rec[s] = 0;
        }
        mbar_init(smem_addr(&xbar[0]), 1);  // + C * 4 bytes of peer partials per row
        mbar_init(smem_addr(&xbar[1]), 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Cluster barrier: arrived on now (this CTA's barriers exist), waited on
    // by the consumers before their first push into a peer and by the
    // producers before they exit -- the producers' first copies do not wait
    // for the peers.
    if (CLUSTERED) cluster_arrive_relaxed();

    if (warp < W) {
        // ----------------------------------------------------------- producers
        // The CTA's stages are numbered g = (row iteration) * nstage_row + j;
        // stage g fills ring slot g % nst, and slot q belongs to producer warp
        // q % W: each slot has one owner, which fills it in stage order (so
        // its parity never runs more than one lap ahead of the consumers).  One slot = up to P consecutive segments
        // of one row, one bulk copy each, issued by lanes 0..cnt-1 and all
        // counted on the slot's single `full` mbarrier (lane 0 arms it with
        // the slot's total bytes).
        const uint64_t pol = l2_evict_first_policy();
        const int64_t col = (int64_t)chunk0 * 8;
        bool ok = true;
        // Routing metadata one row ahead: lane k holds perm[t, k] of the row
        // being issued and has the next row's value in flight (every
        // producer warp keeps its own copy).
        int32_t raw_next = raw_first;
        float w_next = w_first;
        float gate_next = 0.0f;
        if (a.shared_gate && first_row < main_rows) gate_next = __ldg(a.shared_gate + first_row);
        int64_t g0 = 0;  // stage number of the row's first stage
        for (int64_t t = first_row; t < main_rows && ok; t += row_step, g0 += nstage_row) {
            const int32_t raw = raw_next;
            const float my_w = w_next;
            const float s_coef = a.shared_gate ? 1.0f / (1.0f + expf(-gate_next)) : 1.0f;
            if (a.shared_gate && t + row_step < main_rows) gate_next = __ldg(a.shared_gate + t + row_step);
            int64_t my_row = -1;  // checked lazily, at this warp's first routed stage
            for (int j = 0; j < nstage_row && ok; ++j) {
                const int64_t g = g0 + j;
                const int slot = (int)(g % nst);
                if (slot % W != warp) continue;
                const uint32_t phase = (uint32_t)((g / nst) & 1);
                int s0, cnt;
                stage_range(j, P, nS + 1, nseg, s0, cnt);
                const int s = s0 + lane;
                const int e = s - nS - 1;
                int64_t row_k = 0;
                float w_k = 1.0f;
                if (s0 > nS) {  // routed stage
                    if (my_row < 0) {
                        my_row = lane < a.K ? checked_row(raw, a.rows_e, a.err) : 0;
                        if (lane < a.K && t + row_step < main_rows) {
                            raw_next = __ldg(a.perm + (t + row_step) * a.K + lane);
                            w_next = __ldg(a.w + (t + row_step) * a.K + lane);
                        }
                    }
                    const int k = (lane < cnt) ? e / a.R : 0;
                    row_k = __shfl_sync(0xffffffffu, my_row, k);
                    w_k = __shfl_sync(0xffffffffu, my_w, k);
                }
                int go = 0;
                if (lane == 0) {
                    if (*abort_flag) {
                        go = 0;
                    } else if (mbar_wait_bounded(smem_addr(&empty[slot]), phase ^ 1u, abort_flag)) {
                        go = 1;
                    } else {
                        if (!*abort_flag) atomicOr(a.err, kErrTimeout);
                        *abort_flag = 1;
                    }
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                } else {
                    uint8_t* sbase = ring + (size_t)slot * geo.slot_bytes;
                    // Coefficients into the slot header (published by the
                    // same mbarrier phase as the data).
                    if (lane < cnt)
                        reinterpret_cast<float*>(sbase)[lane] = e >= 0 ? w_k : (s < nS ? s_coef : 1.0f);
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive_expect_tx(smem_addr(&full[slot]), (uint32_t)cnt * tile_bytes);
                        rec[slot] = (uint8_t)(1u + phase);
                    }
                    if (lane < cnt) {
                        const uint16_t* src;
                        if (s < nS) src = a.S[s] + t * H + col;
                        else if (s == nS) src = a.residual + t * H + col;
                        else src = a.E[e % a.R] + row_k * H + col;
                        bulk_g2s(smem_addr(sbase + kSlotHeader + (size_t)lane * geo.seg_stride), src,
                                 tile_bytes, smem_addr(&full[slot]), pol);
                    }
                }
            }
            if (my_row < 0 && lane < a.K && t + row_step < main_rows) {  // no routed stage of this row here
                raw_next = __ldg(a.perm + (t + row_step) * a.K + lane);
                w_next = __ldg(a.w + (t + row_step) * a.K + lane);
            }
        }
        if (has_part && ok) {
            // This CTA's part of a split row: segments [pa, pb) of row t,
            // through the same ring, after the whole rows.
            const int64_t t = main_rows + blockIdx.x / parts;
            const int pa = (int)((int64_t)(blockIdx.x % parts) * nseg / parts);
            const int pb = (int)((int64_t)(blockIdx.x % parts + 1) * nseg / parts);
            const int nsr = nS + 1;
            int64_t my_row = 0;
            float my_w = 0.0f;
            if (lane < a.K) {
                my_w = __ldg(a.w + t * a.K + lane);
                if (pb > nsr) my_row = checked_row(__ldg(a.perm + t * a.K + lane), a.rows_e, a.err);
            }
            const float s_coef = shared_coef(a, t);
            const int nstage = part_stage_count(P, nsr, pa, pb);
            for (int j = 0; j < nstage && ok; ++j) {
                const int64_t g = g0 + j;
                const int slot = (int)(g % nst);
                if (slot % W != warp) continue;
                const uint32_t phase = (uint32_t)((g / nst) & 1);
                int s0, cnt;
                part_stage_range(j, P, nsr, pa, pb, s0, cnt);
                const int s = s0 + lane;
                const int e = s - nsr;
                int64_t row_k = 0;
                float w_k = 1.0f;
                if (s0 >= nsr) {
                    const int k = (lane < cnt) ? e / a.R : 0;
                    row_k = __shfl_sync(0xffffffffu, my_row, k);
                    w_k = __shfl_sync(0xffffffffu, my_w, k);
                }
                int go = 0;
                if (lane == 0) {
                    if (*abort_flag) {
                        go = 0;
                    } else if (mbar_wait_bounded(smem_addr(&empty[slot]), phase ^ 1u, abort_flag)) {
                        go = 1;
                    } else {
                        if (!*abort_flag) atomicOr(a.err, kErrTimeout);
                        *abort_flag = 1;
                    }
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                } else {
                    uint8_t* sbase = ring + (size_t)slot * geo.slot_bytes;
                    if (lane < cnt)
                        reinterpret_cast<float*>(sbase)[lane] = e >= 0 ? w_k : (s < nS ? s_coef : 1.0f);
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive_expect_tx(smem_addr(&full[slot]), (uint32_t)cnt * tile_bytes);
                        rec[slot] = (uint8_t)(1u + phase);
                    }
                    if (lane < cnt) {
                        const uint16_t* src;
                        if (s < nS) src = a.S[s] + t * H + col;
                        else if (s == nS) src = a.residual + t * H + col;
                        else src = a.E[e % a.R] + row_k * H + col;
                        bulk_g2s(smem_addr(sbase + kSlotHeader + (size_t)lane * geo.seg_stride), src,
                                 tile_bytes, smem_addr(&full[slot]), pol);
                    }
                }
            }
        }
        if (CLUSTERED) {
            __syncwarp();
            cluster_wait_acquire();
        }
        // After an abort, wait (briefly, bounded) for every copy still landing
        // in this warp's slots before the CTA may exit.
        if (lane == 0 && *abort_flag) {
            for (int j = warp; j < nst; j += W)
                if (rec[j])
                    (void)mbar_wait_bounded(smem_addr(&full[j]), (uint32_t)(rec[j] - 1), nullptr,
                                            10000000ull);
        }
        pdl_trigger();
        return;
    }

    // -------------------------------------------------------------- consumers
    if (CLUSTERED) cluster_wait_acquire();  // every peer's barriers exist before any push
    const int ci = threadIdx.x - 32 * W;
    const int nct = ncw * 32;
    int lch[CPT];
    bool valid[CPT];
    float gw[CPT][8];
#pragma unroll
    for (int m = 0; m < CPT; ++m) {
        lch[m] = ci + m * nct;
        valid[m] = lch[m] < nchunk;
        if (valid[m]) {
            float gf[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.gamma + (size_t)(chunk0 + lch[m]) * 8), gf);
#pragma unroll
            for (int j = 0; j < 8; ++j) gw[m][j] = gf[j] + a.weight_bias;
        }
    }

    int slot = 0;
    uint32_t phase = 0;
    int par_row = 0;
    uint32_t xph = 0u;  // bit p: phase of xbar[p] to wait for next
    bool ok = true;
    if (!CLUSTERED && a.stall_wait_ns) {
        // Failure injection: xbar[0] is unused by whole rows and nothing
        // arrives on it, so this bounded wait runs out and the CTA takes the
        // same timeout path as a pipeline wait that never completes.
        if (!mbar_wait_bounded(smem_addr(&xbar[0]), 0u, abort_flag, a.stall_wait_ns)) {
            ok = false;
            if (!*abort_flag) atomicOr(a.err, kErrTimeout);
            *abort_flag = 1;
        }
    }
    for (int64_t t = first_row; t < main_rows; t += row_step) {
        float acc[CPT][8];
#pragma unroll
        for (int m = 0; m < CPT; ++m)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[m][j] = 0.0f;
        for (int j = 0; j < nstage_row; ++j) {
            int s0, cnt;
            stage_range(j, P, nS + 1, nseg, s0, cnt);
            if (ok && !mbar_wait_bounded(smem_addr(&full[slot]), phase, abort_flag)) {
                ok = false;
                if (!*abort_flag) atomicOr(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            const uint8_t* base = ring + (size_t)slot * geo.slot_bytes;
            const float* coef = reinterpret_cast<const float*>(base);
            const uint8_t* seg = base + kSlotHeader;
            // U segments at a time: loads first, then FMAs.
            fold_slot<CPT, U>(acc, coef, seg, (size_t)geo.seg_stride, cnt, lch, valid);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty[slot]));
            if (++slot == nst) {
                slot = 0;
                phase ^= 1u;
            }
        }

        // Row epilogue, all on chip.
        float ss = 0.0f;
#pragma unroll
        for (int m = 0; m < CPT; ++m) {
            if (valid[m]) {
                store_residual8<RES_F32>(a.residual_out, t * H + (int64_t)(chunk0 + lch[m]) * 8, acc[m]);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc[m][j] = norm_input(acc[m][j], a.norm_bf16_h);
                    ss = fmaf(acc[m][j], acc[m][j], ss);
                }
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) red[par_row * 32 + (warp - W)] = ss;
        named_barrier_sync(1, nct);
        float tot = 0.0f;
        for (int w = 0; w < ncw; ++w) tot += red[par_row * 32 + w];
        if (CLUSTERED) {
            // Push this CTA's partial into every peer (lane rk -> peer rk, all
            // at once, asynchronous stores that count as transaction bytes on
            // the peer's barrier), then wait for all C partials of the row.
            const uint32_t xb = smem_addr(&xbar[par_row]);
            if (ci == 0) mbar_arrive_expect_tx(xb, (uint32_t)C * 4u);
            if (ci < C && !*abort_flag) {  // nothing remote once this CTA has given up
                const uint32_t mine = smem_addr(&xslot[par_row * kMaxCluster + crank]);
                st_async_remote_f32(map_shared_rank(mine, (uint32_t)ci), tot, map_shared_rank(xb, (uint32_t)ci));
            }
            if (ok && !mbar_wait_bounded<true>(xb, (xph >> par_row) & 1u, abort_flag)) {
                ok = false;
                if (!*abort_flag) atomicOr(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            xph ^= 1u << par_row;
            tot = sum_slots(xslot + par_row * kMaxCluster, C);
        }
        const float inv = rsqrtf(tot / (float)H + a.eps);
#pragma unroll
        for (int m = 0; m < CPT; ++m) {
            if (valid[m]) {
                float o[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = acc[m][j] * inv * gw[m][j];
                st_global16(reinterpret_cast<uint16_t*>(a.out) + t * H + (int64_t)(chunk0 + lch[m]) * 8,
                            f32x8_to_bf16x8(o));
            }
        }
        par_row ^= 1;
    }
    // No exit barrier for clusters: a CTA leaves after it has received every
    // peer's partial of its last row, so nothing more is written into it (and
    // it reads nothing remote).  After an abort, a bounded grace period lets
    // peers' pushes still in flight land first.
    if (CLUSTERED && ci == 0 && *abort_flag) grace_period(1000000ull);
    if (!CLUSTERED && has_part) {
        // This CTA's part of a split row: accumulate its segments, publish the
        // fp32 partial row, count the parts in; the CTA that brings the last
        // part sums all of them in part order (a fixed order, whichever CTA
        // finishes last) and finishes the row.  No CTA waits for another.
        const int64_t t = main_rows + blockIdx.x / parts;
        const int pa = (int)((int64_t)(blockIdx.x % parts) * nseg / parts);
        const int pb = (int)((int64_t)(blockIdx.x % parts + 1) * nseg / parts);
        const int nsr = nS + 1;
        float acc[CPT][8];
#pragma unroll
        for (int m = 0; m < CPT; ++m)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[m][j] = 0.0f;
        const int nstage = part_stage_count(P, nsr, pa, pb);
        for (int j = 0; j < nstage; ++j) {
            int s0, cnt;
            part_stage_range(j, P, nsr, pa, pb, s0, cnt);
            if (ok && !mbar_wait_bounded(smem_addr(&full[slot]), phase, abort_flag)) {
                ok = false;
                if (!*abort_flag) atomicOr(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            const uint8_t* base = ring + (size_t)slot * geo.slot_bytes;
            const float* coef = reinterpret_cast<const float*>(base);
            const uint8_t* seg = base + kSlotHeader;
            fold_slot<CPT, U>(acc, coef, seg, (size_t)geo.seg_stride, cnt, lch, valid);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty[slot]));
            if (++slot == nst) {
                slot = 0;
                phase ^= 1u;
            }
        }
        float* mine = a.part_scratch + (int64_t)blockIdx.x * H;
#pragma unroll
        for (int m = 0; m < CPT; ++m)
            if (valid[m]) {
                float4* q = reinterpret_cast<float4*>(mine + (int64_t)lch[m] * 8);
                __stcg(q, make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]));
                __stcg(q + 1, make_float4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]));
            }
        __threadfence();
        named_barrier_sync(1, nct);
        if (ci == 0) {
            unsigned* count = a.part_count + blockIdx.x / parts;
            const unsigned prev = atomicAdd(count, 1u);
            const int last = prev == (unsigned)(parts - 1);
            if (last) *count = 0u;  // every part has arrived: ready for the next call
            __threadfence();
            *last_flag = last;
        }
        named_barrier_sync(1, nct);
        if (!*last_flag) {
            pdl_trigger();
            return;
        }
        const int64_t first_part = (int64_t)(blockIdx.x / parts) * parts;
        const int my_part = (int)(blockIdx.x % parts);
#pragma unroll
        for (int m = 0; m < CPT; ++m) {
            if (!valid[m]) continue;
            float sum[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) sum[j] = 0.0f;
            for (int p = 0; p < parts; ++p) {
                if (p == my_part) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) sum[j] += acc[m][j];
                } else {
                    const float4* q = reinterpret_cast<const float4*>(
                        a.part_scratch + (first_part + p) * H + (int64_t)lch[m] * 8);
                    const float4 x0 = __ldcg(q), x1 = __ldcg(q + 1);
                    sum[0] += x0.x; sum[1] += x0.y; sum[2] += x0.z; sum[3] += x0.w;
                    sum[4] += x1.x; sum[5] += x1.y; sum[6] += x1.z; sum[7] += x1.w;
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[m][j] = sum[j];
        }
        // the row's epilogue, as for whole rows
        float ss = 0.0f;
#pragma unroll
        for (int m = 0; m < CPT; ++m) {
            if (valid[m]) {
                store_residual8<RES_F32>(a.residual_out, t * H + (int64_t)(chunk0 + lch[m]) * 8, acc[m]);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc[m][j] = norm_input(acc[m][j], a.norm_bf16_h);
                    ss = fmaf(acc[m][j], acc[m][j], ss);
                }
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) red[par_row * 32 + (warp - W)] = ss;
        named_barrier_sync(1, nct);
        float tot = 0.0f;
        for (int w = 0; w < ncw; ++w) tot += red[par_row * 32 + w];
        const float inv = rsqrtf(tot / (float)H + a.eps);
#pragma unroll
        for (int m = 0; m < CPT; ++m) {
            if (valid[m]) {
                float o[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = acc[m][j] * inv * gw[m][j];
                st_global16(reinterpret_cast<uint16_t*>(a.out) + t * H + (int64_t)(chunk0 + lch[m]) * 8,
                            f32x8_to_bf16x8(o));
            }
        }
    }
    pdl_trigger();
}

// ------------------------------------------------------------------ host side
template <bool CL>
struct KernelTable {
    using Fn = void (*)(RowArgs, StreamGeom);
    static constexpr int kU = 4;
    static Fn get(int cpt, bool res_f32) {
        switch (cpt * 2 + (res_f32 ? 1 : 0)) {
            case 2: return stream_rows_kernel<1, kU, false, CL>;
            case 3: return stream_rows_kernel<1, kU, true, CL>;
            case 4: return stream_rows_kernel<2, kU, false, CL>;
            case 5: return stream_rows_kernel<2, kU, true, CL>;
            // four chunks per thread: two segments per step keep the loads in registers
            case 8: return stream_rows_kernel<4, 2, false, CL>;
            case 9: return stream_rows_kernel<4, 2, true, CL>;
        }
        return nullptr;
    }
};

static void* kernel_for(int cpt, bool res_f32, bool clustered) {
    return clustered ? reinterpret_cast<void*>(KernelTable<true>::get(cpt, res_f32))
                     : reinterpret_cast<void*>(KernelTable<false>::get(cpt, res_f32));
}

cudaError_t stream_rows_set_attributes(int smem_optin) {
    for (int cl = 0; cl < 2; ++cl)
        for (int cpt = 1; cpt <= 4; cpt <<= 1)
            for (int f = 0; f < 2; ++f) {
                const void* k = kernel_for(cpt, f != 0, cl != 0);
                cudaError_t e =
                    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
                if (e != cudaSuccess) return e;
                if (cl) {
                    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                    if (e != cudaSuccess) return e;
                }
            }
    return cudaSuccess;
}

static int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Consumer layout for a tile of `chunks` 16-byte chunks.
static bool consumer_layout(int chunks, int* cpt, int* threads) {
    int c = 1;
    while (c < 4 && chunks > c * kStreamMaxConsumers) c <<= 1;
    if (chunks > c * kStreamMaxConsumers) return false;
    *cpt = c;
    *threads = 32 * ceil_div(ceil_div(chunks, c), 32);  // consumer threads
    return true;
}

bool plan_stream_rows(int R, int K, int H, bool shared, int64_t T, int num_sms, int smem_optin,
                      int max_cluster, int C, int stage_bytes, StreamPlan* p, int producers,
                      int max_tail_parts) {
    const int chunks = H / 8;
    const int nseg = (shared ? R : 0) + 1 + R * K;
    if (chunks < 1 || T < 1) return false;
    if (C <= 0) {
        // Enough CTAs to cover every SM: split rows into tiles only when the
        // rows alone cannot, and never so finely that a CTA owns no chunk.
        // Whole rows once there are at least half as many rows as SMs
        // (measured: one row per CTA beats split rows there).
        C = 1;
        if (2 * T < num_sms)
            while (C < kMaxCluster && C * 2 <= max_cluster && (int64_t)C * T < num_sms &&
                   (2 * C - 1) * ceil_div(chunks, 2 * C) < chunks)
                C <<= 1;
    }
    if (C < 1 || C > kMaxCluster || C > max_cluster) return false;
    const int tile = ceil_div(chunks, C);
    if ((C - 1) * tile >= chunks) return false;  // every CTA must own a chunk
    int cpt, threads;
    if (!consumer_layout(tile, &cpt, &threads)) return false;
    const int seg_stride = ceil_div(tile * 16, 128) * 128;
    // Segments per slot: enough for a ~64 KB slot, at most one per producer
    // lane, spread evenly over the row.  Bulk copies are issued one slot per
    // instruction and issue costs per copy, not per byte, so slots are made
    // large (measured on GB300: 64 KB slots beat 16 KB ones for column tiles
    // as well as whole rows).
    const int target = stage_bytes > 0 ? stage_bytes : 65536;
    int P = target / seg_stride;
    if (P < 1) P = 1;
    if (P > 32) P = 32;
    if (P > nseg) P = nseg;
    while (P > 1 && stream_ring_offset(2) + 2 * (kSlotHeader + P * seg_stride) > smem_optin) --P;
    const int nsr = (shared ? R : 0) + 1;
    if (R * K > 0) P = ceil_div(R * K, ceil_div(R * K, P));  // routed stages of equal size
    const int slot_bytes = kSlotHeader + P * seg_stride;
    const int per_row = ceil_div(nsr, P) + ceil_div(R * K, P);
    int nst;
    if (C == 1) {
        // Whole rows: one CTA per SM with the deepest ring that fits.
        nst = kStreamMaxStages;
        while (nst > 2 && stream_ring_offset(nst) + nst * slot_bytes > smem_optin) --nst;
    } else {
        // Tiles: a ring of ~1/3 of shared memory (three CTAs per SM, leaving
        // room for the 1 KB the driver reserves per CTA), at most two rows deep.
        const int budget = smem_optin / 3 - 3072;
        nst = budget / slot_bytes;
        if (nst > 2 * per_row) nst = 2 * per_row;
        if (nst > kStreamMaxStages) nst = kStreamMaxStages;
        if (nst < 2) nst = 2;
    }
    if (nst < 2 || stream_ring_offset(nst) + nst * slot_bytes > smem_optin) return false;
    // Producer warps: up to four (slot q is filled by warp q % W).
    int W = nst < kStreamMaxProducers ? nst : kStreamMaxProducers;
    if (producers > 0) W = producers < nst ? producers : nst;
    if (W > kStreamMaxProducers || threads + 32 * W > kStreamMaxThreads) return false;
    p->geo.producers = W;
    p->geo.nstages = nst;
    p->geo.slot_bytes = slot_bytes;
    p->geo.seg_per_stage = P;
    p->geo.seg_stride = seg_stride;
    p->geo.C = C;
    p->geo.tile_chunks = tile;
    p->cpt = cpt;
    p->threads = threads + 32 * W;
    p->smem = stream_ring_offset(nst) + nst * slot_bytes;
    p->geo.main_rows = T;
    p->geo.tail_parts = 1;
    if (C == 1) {
        p->grid = (int)(T < num_sms ? T : num_sms);
        // The last wave (T mod num_sms rows; all rows when T < num_sms) would
        // leave SMs idle: split each of its rows into m segment intervals on
        // m CTAs, m = the largest that fits beside the others, capped.
        // Parts keep at least kMinPartSegs segments: a light row (K = 0 has
        // three) gains nothing from splitting and pays the parts' reduction.
        const int64_t tail = T % num_sms;
        if (max_tail_parts >= 2 && tail > 0) {
            int64_t m = num_sms / tail;
            if (m > max_tail_parts) m = max_tail_parts;
            if (m > nseg / kMinPartSegs) m = nseg / kMinPartSegs;
            if (m >= 2) {
                p->geo.main_rows = T - tail;
                p->geo.tail_parts = (int)m;
                if (T < num_sms) p->grid = (int)(tail * m);
            }
        }
    } else {
        const int per_sm = smem_optin / p->smem > 0 ? smem_optin / p->smem : 1;
        int64_t clusters = ((int64_t)num_sms * per_sm) / C;
        if (clusters < 1) clusters = 1;
        if (clusters > T) clusters = T;
        p->grid = (int)clusters * C;
    }
    return true;
}

int stream_rows_max_cluster(int threads, int smem, int cpt) {
    for (int C = kMaxCluster; C >= 2; C >>= 1) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3((unsigned)C);
        cfg.blockDim = dim3((unsigned)threads);
        cfg.dynamicSmemBytes = (size_t)smem;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        const void* k = kernel_for(cpt, false, true);
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess && n > 0) return C;
        (void)cudaGetLastError();
    }
    return 1;
}

// Clusters of a clustered plan the device holds at once (0 if the query
// fails).
int stream_rows_active_clusters(const StreamPlan& p, bool res_f32) {
    const void* k = kernel_for(p.cpt, res_f32, true);
    if (!k || p.geo.C < 2) return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)p.geo.C);
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = (size_t)p.smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.geo.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Whether the device can run exactly this plan's blocks (and, for tiles, one
// cluster of them at once).
bool stream_rows_plan_fits(const StreamPlan& p, bool res_f32) {
    const bool clustered = p.geo.C > 1;
    const void* k = kernel_for(p.cpt, res_f32, clustered);
    if (!k) return false;
    int n = 0;
    cudaError_t e;
    if (!clustered) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, p.threads, (size_t)p.smem);
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3((unsigned)p.geo.C);
        cfg.blockDim = dim3((unsigned)p.threads);
        cfg.dynamicSmemBytes = (size_t)p.smem;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)p.geo.C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
    }
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e == cudaSuccess && n > 0;
}

cudaError_t launch_stream_rows(const RowArgs& a, const StreamPlan& p, bool res_f32,
                               cudaStream_t stream, bool pdl) {
    const bool clustered = p.geo.C > 1;
    const void* k = kernel_for(p.cpt, res_f32, clustered);
    if (!k) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = (size_t)p.smem;
    cfg.stream = stream;
    int na = 0;
    if (clustered) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.geo.C;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    void* args[] = {const_cast<RowArgs*>(&a), const_cast<StreamGeom*>(&p.geo)};
    return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace arf

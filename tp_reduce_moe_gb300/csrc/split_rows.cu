// split_rows.cu -- decode-latency kernel: one token row per thread-block
// cluster, the row's segments dealt round-robin over the cluster's CTAs.
//
// At decode sizes a row is nseg = R*(K+1)+1 segments of H bf16 (~1 MB) and
// the TMA engine completes a bulk copy every ~50 ns whatever its size, so the
// number of copies per CTA -- not the bytes -- sets the time.  The C CTAs of
// the cluster form G column groups of Cs = C/G CTAs; group g covers 1/G of the
// row's columns.  CTA cs of a group copies only segments cs, cs+Cs, ... of
// its group's columns (~nseg/Cs copies, all in flight at once), accumulates
// them into an fp32 partial row of the group's columns, and the group then
// reduce-scatters the partials through distributed shared memory: every CTA
// sends slice j of its partial row to CTA j of its group with one bulk copy
// (shared -> peer shared, the TMA engine), completing on that CTA's receive
// mbarrier; each CTA then sums its Cs received slices locally (fixed rank
// order), which is h for its column tile.  The tile sums of squares go to
// every CTA of the cluster as asynchronous remote stores (st.async) counted
// as transaction bytes on the peer's barrier -- no release fence, so they do
// not wait for the residual_out stores just issued; each CTA normalises and
// stores its tile.  Groups cut the bytes through the cluster exchange G-fold
// for G-fold more, smaller copies: measured at DeepSeek-V3 sizes (C = 16,
// T = 1) 6.3 us with one group, 5.1 us with four.
//
//   start: the routing metadata and gamma are requested before the barrier
//     set-up, so their round trips overlap it.
//   copies: the first consumer warp issues the shared partials + residual
//     (they need no routing metadata) on mbarrier 0 while the producer warp
//     issues the routed rows in two halves on mbarriers 1 and 2 (the lanes
//     of a bulk-copy instruction are issued one after another, 60-160 cycles
//     each, so one warp issuing both would delay the routed ones);
//     per-segment coefficients go into a shared-memory table published by
//     the same barrier phases.
//   consumers: fold the CTA's segments into registers (the first routed half
//     while the second lands), write the partial row over the spent segment
//     buffers; wait for the Cs slices of this tile; local sums; wait for the
//     C sums; normalise; store.
//   producer warp, afterwards: sends the partial row's slices to the group
//     peers and the tile's sum of squares to every CTA of the cluster.
//   two rounds (heavy rows, e.g. 177 segments at R = 16, K = 10): the CTA
//     has buffers for the first half of its segments only; the producer warp
//     issues the second routed half into them once every consumer warp has
//     folded the first (one more memory round trip, half the shared memory,
//     so two CTAs fit on an SM where one did).
//
// One cluster barrier (arrived on right after the mbarriers are initialised,
// waited on just before the first send) keeps peers from signalling a
// barrier that does not exist yet.  None is needed at exit: a CTA sends its
// sum of squares only after it has received every slice, so once a CTA holds
// all C sums (its group peers' among them), every copy that reads its partial
// row has landed and nothing more will be written into it.  Every mbarrier wait is bounded
// (arf::mbar_wait_bounded); after one runs out, the CTA waits a bounded grace
// period for copies in flight before it exits.
//
// Operation: sglang PR #37196 "[Comm] Share the CuTe DSL AR fusion core and
// wire it for DeepSeek-V3 / GLM-5.x", Motivation and Modifications sections
// 1-2; sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with final
// RMSNorm", Changes.
#include <algorithm>

#include "arf_host.h"

namespace arf {

constexpr int kSplitMaxSegs = 32;       // segments per CTA and copy round (one producer lane each)
constexpr int kSplitMaxConsumers = 512;
constexpr int kSplitMaxThreads = 32 + kSplitMaxConsumers;
constexpr int kSplitHeader = 1024;      // barriers, coefficient table, partial sums, flags
constexpr int kSplitMinGroupChunks = 128;  // automatic column groups: at least 2 KB per copy

// Header layout (bytes): 0 bar[3] (segment loads: shared partials and
// residual, first and second half of the routed rows), 24 rbar (slices
// received), 32 ssbar (sums of squares received), 40 relbar (two rounds: the
// first round's buffers are folded, one arrival per consumer warp); 64
// coef[64] f32; 320 red[32] f32; 448 ss slots [16] f32 (one per source CTA);
// 512 abort flag; 516 second-round flag; 1024 receive buffer
// [Cs][tile_chunks*8] f32 (slice of every source CTA's partial row); then the
// segment buffers at seg_stride, which the partial row [group_chunks*8] f32
// reuses once the segments are folded in.  With two rounds there are buffers
// for the first nmid segments only: segment i >= nmid lands in buffer
// i - nmid.
template <int CPT, bool RES_F32>
__global__ void __launch_bounds__(kSplitMaxThreads, 1)
    split_rows_kernel(const __grid_constant__ RowArgs a, const SplitGeom geo) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_trigger();
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    uint64_t* rbar = bar + 3;
    uint64_t* ssbar = bar + 4;
    uint64_t* relbar = bar + 5;
    float* coef = reinterpret_cast<float*>(smem + 64);
    float* red = reinterpret_cast<float*>(smem + 320);
    float* ss_slots = reinterpret_cast<float*>(smem + 448);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 512);
    int* round2 = reinterpret_cast<int*>(smem + 516);
    float* recv = reinterpret_cast<float*>(smem + kSplitHeader);
    uint8_t* segbuf = smem + kSplitHeader + geo.part_bytes;
    // the CTA's fp32 partial row reuses the segment buffers once every
    // consumer is done with them
    float* part = reinterpret_cast<float*>(segbuf);

    const int C = geo.C;
    const int Cs = geo.Cs;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ncw = (blockDim.x >> 5) - 1;
    const uint32_t c = cluster_ctarank();
    const int grp = (int)c / Cs;        // column group of this CTA
    const int cs = (int)c - grp * Cs;   // rank within the group
    const int64_t t = blockIdx.x / C;
    const int H = a.H;
    // this CTA's column group: chunks [g0, g0 + chunks) of the row
    const int g0 = grp * geo.group_chunks;
    const int chunks = min(geo.group_chunks, H / 8 - g0);
    const int64_t col0 = (int64_t)g0 * 8;           // first element of the group
    const uint32_t row_bytes = (uint32_t)chunks * 16u;  // bytes of a segment's group
    const int nS = a.has_shared ? a.R : 0;
    const int nsr = nS + 1;                          // shared partials + residual
    const int nseg = nsr + a.R * a.K;
    // Segments of this CTA: s = cs + i*Cs, i < ns; the first nsr_c need no
    // perm; the routed ones i in [nsr_c, nmid) complete on bar[1], the rest on
    // bar[2], so the consumers fold the first half while the second lands.
    const int ns = (nseg - cs + Cs - 1) / Cs;
    const int nsr_c = (nsr > cs) ? (nsr - 1 - cs) / Cs + 1 : 0;
    const int nmid = nsr_c + (ns - nsr_c + 1) / 2;
    // Two rounds: the routed rows [nmid, ns) go out only once the consumers
    // have folded [0, nmid), into the buffers of segments [0, ns - nmid).
    const bool two = geo.rounds == 2;

    const int tile = geo.tile_chunks;
    const int ntile_c = min(tile, chunks - cs * tile);  // chunks of this CTA's tile
    const int tile0 = g0 + cs * tile;  // first chunk of this CTA's tile in the row
    const int ci = threadIdx.x - 32;
    const int nct = ncw * 32;

    // The routing metadata (producer lanes k < K) and gamma (consumers, for
    // this CTA's column tile: work item q = one float4, half a 16-byte bf16
    // chunk; a consumer thread owns items ci + m*nct, m < CPT, enough since a
    // tile is at most half the row) are requested first, with loads the
    // compiler keeps in place: their memory round trips overlap the barrier
    // set-up below instead of following it.
    pdl_wait();  // no global memory access before this point
    int32_t raw = 0;
    float wv = 0.0f;
    if (warp == 0 && lane < a.K) {
        raw = (int32_t)ld_early4(a.perm + t * a.K + lane);
        wv = __uint_as_float(ld_early4(a.w + t * a.K + lane));
    }
    uint2 gpre[CPT];
    bool hv[CPT];
#pragma unroll
    for (int m = 0; m < CPT; ++m) {
        const int q = ci + m * nct;
        hv[m] = warp > 0 && q < 2 * ntile_c;
        gpre[m] = hv[m] ? ld_early8(a.gamma + (int64_t)tile0 * 8 + (int64_t)q * 4) : make_uint2(0, 0);
    }
    // a gated shared expert's gate logit, for the warp that writes the shared
    // partials' coefficients (requested with the metadata, read after its
    // copies are out)
    const uint32_t gate_bits = (warp == 1 && a.shared_gate) ? ld_early4(a.shared_gate + t) : 0u;

    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar[0]), 1);
        mbar_init(smem_addr(&bar[1]), 1);
        mbar_init(smem_addr(&bar[2]), 1);
        mbar_init(smem_addr(rbar), 1);
        mbar_init(smem_addr(ssbar), 1);
        mbar_init(smem_addr(relbar), (uint32_t)ncw);
        *abort_flag = 0;
        *round2 = 0;
        fence_mbar_init();
        // every CTA of the group sends this tile's slice of its partial row,
        // and every CTA of the cluster its tile's sum of squares (4 bytes)
        mbar_arrive_expect_tx(smem_addr(rbar), (uint32_t)(Cs * ntile_c * 32));
        mbar_arrive_expect_tx(smem_addr(ssbar), (uint32_t)C * 4u);
    }
    __syncthreads();
    // barrier A, arrive: this CTA's mbarriers exist
    cluster_arrive_relaxed();

    // A bulk-copy instruction holds its warp while its lanes' copies are
    // issued one after another (60-160 cycles each: ~0.6 us for 16 lanes),
    // so the two kinds of copies go out from two warps at once: the
    // first consumer warp issues the perm-independent copies (shared partials
    // and residual, on bar[0]) before it starts consuming, and the producer
    // warp the routed rows (on bar[1] and bar[2]) -- the routing metadata has
    // been in flight since before the barrier set-up.  Each warp writes its
    // segments' coefficients, then arms its barriers (a phase needs the
    // arming lane's arrival as well as the bytes, so it cannot complete
    // early; the arrival publishes the coefficients).
    if (warp <= 1) {
        const uint64_t pol = l2_evict_first_policy();
        const int i = lane;
        const int s = cs + i * Cs;
        const uint32_t dst = smem_addr(segbuf + (size_t)i * geo.seg_stride);
        if (warp == 1) {
            if (i < nsr_c) {
                const uint16_t* src = (s < nS ? a.S[s] + t * H : a.residual + t * H) + col0;
                bulk_g2s(dst, src, row_bytes, smem_addr(&bar[0]), pol);
                coef[i] = s < nS && a.shared_gate ? 1.0f / (1.0f + expf(-__uint_as_float(gate_bits))) : 1.0f;
            }
            __syncwarp();
            if (lane == 0 && nsr_c > 0) mbar_arrive_expect_tx(smem_addr(&bar[0]), (uint32_t)nsr_c * row_bytes);
        } else {
            const bool routed = i >= nsr_c && i < (two ? nmid : ns);
            const int64_t rowv = lane < a.K ? checked_row(raw, a.rows_e, a.err) : 0;
            const int e = s - nsr;
            const int k = routed ? e / a.R : 0;
            const int64_t row_k = __shfl_sync(0xffffffffu, rowv, k);
            const float w_k = __shfl_sync(0xffffffffu, wv, k);
            if (routed) {
                bulk_g2s(dst, a.E[e % a.R] + row_k * H + col0, row_bytes, smem_addr(&bar[i < nmid ? 1 : 2]), pol);
                coef[i] = w_k;
            }
            __syncwarp();
            if (lane == 0) {
                if (nmid > nsr_c) mbar_arrive_expect_tx(smem_addr(&bar[1]), (uint32_t)(nmid - nsr_c) * row_bytes);
                if (!two && ns > nmid) mbar_arrive_expect_tx(smem_addr(&bar[2]), (uint32_t)(ns - nmid) * row_bytes);
            }
            if (two && ns > nmid) {
                // Second round: once every consumer warp has folded the first
                // (relbar), the routed rows [nmid, ns) into buffers
                // [0, ns - nmid), lane l taking segment nmid + l.
                int go = 0;
                if (lane == 0) {
                    if (mbar_wait_bounded(smem_addr(relbar), 0u, abort_flag)) {
                        go = *abort_flag ? 0 : 1;
                    } else {
                        if (!*abort_flag) atomicOr(a.err, kErrTimeout);
                        *abort_flag = 1;
                    }
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (go) {
                    const int i2 = nmid + lane;
                    const bool routed2 = i2 < ns;
                    const int e2 = cs + i2 * Cs - nsr;
                    const int k2 = routed2 ? e2 / a.R : 0;
                    const int64_t row_k2 = __shfl_sync(0xffffffffu, rowv, k2);
                    const float w_k2 = __shfl_sync(0xffffffffu, wv, k2);
                    if (routed2) {
                        bulk_g2s(smem_addr(segbuf + (size_t)lane * geo.seg_stride),
                                 a.E[e2 % a.R] + row_k2 * H + col0, row_bytes, smem_addr(&bar[2]), pol);
                        coef[i2] = w_k2;
                    }
                    __syncwarp();
                    if (lane == 0) {
                        *round2 = 1;
                        mbar_arrive_expect_tx(smem_addr(&bar[2]), (uint32_t)(ns - nmid) * row_bytes);
                    }
                }
            }
        }
    }
    if (warp > 0) {
        // ------------------------------------------------------------ consumers
        float acc[CPT][8];
        bool valid[CPT];
        const uint8_t* src[CPT];  // this thread's chunk in segment 0
#pragma unroll
        for (int m = 0; m < CPT; ++m) {
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[m][j] = 0.0f;
            valid[m] = ci + m * nct < chunks;
            src[m] = segbuf + (size_t)(ci + m * nct) * 16;
        }
        bool ok = true;
        for (int phase_set = 0; phase_set < 3; ++phase_set) {
            const int i_begin = phase_set == 0 ? 0 : phase_set == 1 ? nsr_c : nmid;
            const int i_end = phase_set == 0 ? nsr_c : phase_set == 1 ? nmid : ns;
            if (phase_set == 2 && two) {
                // this warp is done with the first round's buffers
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(relbar));
            }
            // buffer of segment i: i, or i - nmid in the second round
            const int boff = (phase_set == 2 && two) ? nmid : 0;
            if (i_begin >= i_end) continue;
            if (ok && !mbar_wait_bounded(smem_addr(&bar[phase_set]), 0u, abort_flag)) {
                ok = false;
                if (!*abort_flag) atomicOr(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            // Full steps of SU segments without per-segment guards (the
            // instruction count, not the load latency, bounds this loop),
            // then the remaining segments one at a time; the same
            // sequential order per column either way.
            constexpr int SU = CPT >= 4 ? 2 : 4;  // segments per step (loads in registers)
            const size_t stride = (size_t)geo.seg_stride;
            int i0 = i_begin;
            for (; i0 + SU <= i_end; i0 += SU) {
                float cf[SU];
                uint4 v[SU][CPT];
#pragma unroll
                for (int u = 0; u < SU; ++u) cf[u] = coef[i0 + u];
#pragma unroll
                for (int u = 0; u < SU; ++u)
#pragma unroll
                    for (int m = 0; m < CPT; ++m)
                        if (valid[m])
                            v[u][m] = *reinterpret_cast<const uint4*>(src[m] + (size_t)(i0 + u - boff) * stride);
#pragma unroll
                for (int u = 0; u < SU; ++u)
#pragma unroll
                    for (int m = 0; m < CPT; ++m)
                        if (valid[m]) fma_bf16x8(acc[m], cf[u], v[u][m]);
            }
            for (; i0 < i_end; ++i0) {
                const float cf = coef[i0];
#pragma unroll
                for (int m = 0; m < CPT; ++m)
                    if (valid[m])
                        fma_bf16x8(acc[m], cf, *reinterpret_cast<const uint4*>(src[m] + (size_t)(i0 - boff) * stride));
            }
        }
        // The partial row, locally (over the spent segment buffers); made
        // visible to the bulk-copy engine.
        named_barrier_sync(1, nct);
#pragma unroll
        for (int m = 0; m < CPT; ++m) {
            const int ch = ci + m * nct;
            if (ch < chunks) {
                float4* p = reinterpret_cast<float4*>(part + (size_t)ch * 8);
                p[0] = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
                p[1] = make_float4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    // The partial row is complete (consumers) and the producer warp, idle
    // since its copies went out, takes over the cluster traffic: the remote
    // sends go out from a warp that reads no shared memory afterwards, so the
    // consumers' next shared-memory reads are not queued behind them.
    named_barrier_sync(2, blockDim.x);

    // ---- barrier A, wait: every peer's receive barrier exists
    __syncwarp();
    cluster_wait_acquire();
    // send slice j of the group's partial row to CTA j of the group (one
    // bulk copy each)
    if (warp == 0 && lane < Cs && !*abort_flag) {  // nothing remote once this CTA has given up
        const int j = lane;
        const int nj = min(tile, chunks - j * tile);
        const uint32_t peer = (uint32_t)(grp * Cs + j);
        bulk_s2cluster(map_shared_rank(smem_addr(recv + ((size_t)cs * tile) * 8), peer),
                       smem_addr(part + (size_t)j * tile * 8), (uint32_t)nj * 32u,
                       map_shared_rank(smem_addr(rbar), peer));
    }

    // ---- this CTA's column tile: the C received slices summed locally, in
    // rank order.
    const size_t slice = (size_t)tile * 8;  // floats per source slice
    float4 hq[CPT];
    float ss = 0.0f;
    bool ok2 = true;
    if (warp > 0 && !mbar_wait_bounded(smem_addr(rbar), 0u, abort_flag)) {
        ok2 = false;
        if (!*abort_flag) atomicOr(a.err, kErrTimeout);
        *abort_flag = 1;
    }
#pragma unroll
    for (int m = 0; m < CPT; ++m) {
        const int q = ci + m * nct;
        hq[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!hv[m]) continue;
        const float* src = recv + (size_t)q * 4;
        for (int r = 0; r < Cs; ++r) {
            const float4 x = *reinterpret_cast<const float4*>(src + r * slice);
            hq[m].x += x.x;
            hq[m].y += x.y;
            hq[m].z += x.z;
            hq[m].w += x.w;
        }
        const int64_t elem = t * H + (int64_t)tile0 * 8 + (int64_t)q * 4;
        if (RES_F32) {
            st_global16(reinterpret_cast<float*>(a.residual_out) + elem,
                        make_uint4(__float_as_uint(hq[m].x), __float_as_uint(hq[m].y),
                                   __float_as_uint(hq[m].z), __float_as_uint(hq[m].w)));
        } else {
            *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.residual_out) + elem) =
                make_uint2(pack_bf16x2(hq[m].x, hq[m].y), pack_bf16x2(hq[m].z, hq[m].w));
        }
        hq[m].x = norm_input(hq[m].x, a.norm_bf16_h);
        hq[m].y = norm_input(hq[m].y, a.norm_bf16_h);
        hq[m].z = norm_input(hq[m].z, a.norm_bf16_h);
        hq[m].w = norm_input(hq[m].w, a.norm_bf16_h);
        ss += hq[m].x * hq[m].x + hq[m].y * hq[m].y + hq[m].z * hq[m].z + hq[m].w * hq[m].w;
    }
    if (warp > 0) {
        ss = warp_sum(ss);
        if (lane == 0) red[warp - 1] = ss;
    }
    named_barrier_sync(2, blockDim.x);
    if (warp == 0) {
        // the producer warp pushes this tile's sum of squares into every
        // peer's slot c (asynchronous remote stores counted on the peer's
        // barrier) -- only once every slice has arrived (the consumers waited
        // for them before the barrier; a wait that ran out raised the abort
        // flag), which is what lets the receivers exit without a cluster
        // barrier
        if (lane < C && !*abort_flag) {
            float tot = 0.0f;
            for (int w = 0; w < ncw; ++w) tot += red[w];
            st_async_remote_f32(map_shared_rank(smem_addr(ss_slots + c), (uint32_t)lane), tot,
                                map_shared_rank(smem_addr(ssbar), (uint32_t)lane));
        }
    } else if (ok2 && !mbar_wait_bounded<true>(smem_addr(ssbar), 0u, abort_flag)) {
        if (!*abort_flag) atomicOr(a.err, kErrTimeout);
        *abort_flag = 1;
    }

    const float total = sum_slots(ss_slots, C);

    const float inv = rsqrtf(total / (float)H + a.eps);
    const float wb = a.weight_bias;
#pragma unroll
    for (int m = 0; m < CPT; ++m) {
        if (!hv[m]) continue;
        const int64_t col = (int64_t)tile0 * 8 + (int64_t)(ci + m * nct) * 4;
        const uint2 gv = gpre[m];
        const float g0 = __uint_as_float(gv.x << 16) + wb, g1 = __uint_as_float(gv.x & 0xffff0000u) + wb;
        const float g2 = __uint_as_float(gv.y << 16) + wb, g3 = __uint_as_float(gv.y & 0xffff0000u) + wb;
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + t * H + col) =
            make_uint2(pack_bf16x2(hq[m].x * inv * g0, hq[m].y * inv * g1),
                       pack_bf16x2(hq[m].z * inv * g2, hq[m].w * inv * g3));
    }

    // After an abort, copies may still be landing in or reading from this
    // CTA's shared memory: wait (bounded) for its barriers, then a grace
    // period, before the CTA may exit.
    if (threadIdx.x == 0 && *abort_flag) {
        if (nsr_c > 0) (void)mbar_wait_bounded(smem_addr(&bar[0]), 0u, nullptr, 10000000ull);
        if (nmid > nsr_c) (void)mbar_wait_bounded(smem_addr(&bar[1]), 0u, nullptr, 10000000ull);
        if (ns > nmid && (!two || *round2)) (void)mbar_wait_bounded(smem_addr(&bar[2]), 0u, nullptr, 10000000ull);
        (void)mbar_wait_bounded(smem_addr(rbar), 0u, nullptr, 10000000ull);
        (void)mbar_wait_bounded<true>(smem_addr(ssbar), 0u, nullptr, 10000000ull);
        grace_period(1000000ull);
    }
}

// ------------------------------------------------------------------ host side
static int ceil_div_s(int a, int b) { return (a + b - 1) / b; }

bool plan_split_rows(int R, int K, int H, bool shared, int64_t T, int num_sms, int smem_optin,
                     int max_cluster, int C, SplitPlan* p, int groups, int rounds) {
    const int chunks = H / 8;
    const int nsr = (shared ? R : 0) + 1;  // shared partials + residual
    const int nseg = nsr + R * K;
    if (chunks < 2 || T < 1 || groups < 0 || rounds < 1 || rounds > 2) return false;
    if (groups == 0) {
        // Automatic: the most column groups (of at least kSplitMinGroupChunks
        // chunks) that leave a plan -- fewer bytes through the cluster
        // exchange; measured at DeepSeek-V3 and GLM sizes, four groups of a
        // 16-CTA cluster beat one group by 1.1 us at T = 1.
        for (int g = 8; g > 1; g >>= 1)
            if (ceil_div_s(chunks, g) >= kSplitMinGroupChunks &&
                plan_split_rows(R, K, H, shared, T, num_sms, smem_optin, max_cluster, C, p, g, rounds))
                return true;
        groups = 1;
    }
    // Column groups of gch chunks (the last one may be shorter); Cs = C /
    // groups CTAs per group deal the row's segments and reduce-scatter the
    // group's columns.
    const int gch = ceil_div_s(chunks, groups);
    const int last = chunks - (groups - 1) * gch;
    auto make = [&](int c, SplitPlan* q) {
        if (c < 2 || c > 16 || c > max_cluster || c % groups || last < 1) return false;
        const int cs = c / groups;
        if (cs < 2 || cs > nseg) return false;
        // Segment buffers: every segment of the busiest CTA (rank 0 of a
        // group deals the most), or with two rounds its first nmid, the
        // second half reusing them.  A copy round is one producer lane per
        // segment.
        int nbuf = 0;
        bool second = false;
        for (int r = 0; r < cs; ++r) {
            const int ns_r = (nseg - r + cs - 1) / cs;
            const int nsr_r = nsr > r ? (nsr - 1 - r) / cs + 1 : 0;
            const int nmid_r = nsr_r + (ns_r - nsr_r + 1) / 2;
            if (rounds == 1) {
                if (ns_r > kSplitMaxSegs) return false;
                nbuf = std::max(nbuf, ns_r);
            } else {
                if (nmid_r > kSplitMaxSegs || ns_r - nmid_r > kSplitMaxSegs) return false;
                nbuf = std::max(nbuf, nmid_r);
                second = second || ns_r > nmid_r;
            }
        }
        if (rounds == 2 && !second) return false;  // nothing for a second round
        const int tile = ceil_div_s(gch, cs);
        if ((cs - 1) * tile >= last) return false;  // every CTA owns a tile, the shortest group too
        int cpt = 1;
        while (cpt < 4 && gch > cpt * kSplitMaxConsumers) cpt <<= 1;
        if (gch > cpt * kSplitMaxConsumers) return false;
        const int consumers = ceil_div_s(ceil_div_s(gch, cpt), 32) * 32;
        if (2 * tile > cpt * consumers) return false;  // <= CPT items per thread
        const int seg_stride = ceil_div_s(gch * 16, 128) * 128;
        const int recv = ceil_div_s(cs * tile * 32, 128) * 128;
        const int row_f32 = ceil_div_s(gch * 32, 128) * 128;
        const int smem = kSplitHeader + recv + std::max(row_f32, nbuf * seg_stride);
        if (smem > smem_optin) return false;
        q->geo.C = c;
        q->geo.Cs = cs;
        q->geo.group_chunks = gch;
        q->geo.seg_stride = seg_stride;
        q->geo.part_bytes = recv;
        q->geo.row_f32_bytes = row_f32;
        q->geo.tile_chunks = tile;
        q->geo.rounds = rounds;
        q->cpt = cpt;
        q->threads = 32 + consumers;
        q->smem = smem;
        q->grid = (int)(T * c);
        return true;
    };
    SplitPlan q{};
    if (C <= 0) {
        // Automatic: the largest cluster that fits with its CTAs over all
        // rows on at most three quarters of the SMs (measured: beyond that
        // clusters stop being co-resident and the tiled streaming kernel is
        // faster); no plan otherwise.
        for (int c = 16; c >= 2; c >>= 1)
            if ((int64_t)c * T * 4 <= (int64_t)num_sms * 3 && make(c, &q)) {
                *p = q;
                return true;
            }
        return false;
    }
    if (!make(C, &q)) return false;
    *p = q;
    return true;
}

static const void* split_kernel_for(int cpt, bool res_f32) {
    switch (cpt * 2 + (res_f32 ? 1 : 0)) {
        case 2: return reinterpret_cast<const void*>(split_rows_kernel<1, false>);
        case 3: return reinterpret_cast<const void*>(split_rows_kernel<1, true>);
        case 4: return reinterpret_cast<const void*>(split_rows_kernel<2, false>);
        case 5: return reinterpret_cast<const void*>(split_rows_kernel<2, true>);
        case 8: return reinterpret_cast<const void*>(split_rows_kernel<4, false>);
        case 9: return reinterpret_cast<const void*>(split_rows_kernel<4, true>);
    }
    return nullptr;
}

cudaError_t split_rows_set_attributes(int smem_optin) {
    for (int cpt = 1; cpt <= 4; cpt <<= 1)
        for (int f = 0; f < 2; ++f) {
            const void* k = split_kernel_for(cpt, f != 0);
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

int split_rows_max_cluster(int threads, int smem, int cpt) {
    for (int C = 16; C >= 2; C >>= 1) {
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
        if (cudaOccupancyMaxActiveClusters(&n, split_kernel_for(cpt, false), &cfg) == cudaSuccess && n > 0)
            return C;
        (void)cudaGetLastError();
    }
    return 1;
}

// Whether the device can co-schedule one cluster of exactly this plan's launch.
bool split_rows_plan_fits(const SplitPlan& p, bool res_f32) {
    const void* k = split_kernel_for(p.cpt, res_f32);
    if (!k) return false;
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
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e == cudaSuccess && n > 0;
}

bool split_prefer_two_rounds(int64_t T, int n1, int n2) { return n1 >= 1 && n1 < T && n2 > n1; }

int split_rows_active_clusters(const SplitPlan& p, bool res_f32) {
    const void* k = split_kernel_for(p.cpt, res_f32);
    if (!k) return 0;
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

cudaError_t launch_split_rows(const RowArgs& a, const SplitPlan& p, bool res_f32, cudaStream_t stream,
                              bool pdl) {
    const void* k = split_kernel_for(p.cpt, res_f32);
    if (!k) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)p.threads);
    cfg.dynamicSmemBytes = (size_t)p.smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.geo.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    void* args[] = {const_cast<RowArgs*>(&a), const_cast<SplitGeom*>(&p.geo)};
    return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace arf

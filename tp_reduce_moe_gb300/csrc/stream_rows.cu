// stream_rows.cu -- large-T (prefill) kernel: persistent CTAs that each own
// whole token rows and stream them through a shared-memory ring.
//
// Per token row the op reads R*(K+1)+1 contiguous rows of H bf16 (R shared
// partials, the residual, R*K gathered expert rows) and writes two.  With
// thousands of rows the work is a pure HBM stream, so each SM runs one CTA
// whose producer thread keeps a deep ring of whole-row bulk async copies
// (cp.async.bulk: the TMA engine, completion counted on an mbarrier) in
// flight, while consumer warps fold each landed row into fp32 accumulators
// held in registers (CPT 16-byte column chunks per thread).  After a row's
// last summand the consumers finish it entirely on chip: residual_out, the
// sum of squares (warp shuffle + one named barrier), the scale and the
// bf16 out -- so every input byte is read once and every output byte
// written once, and the next row's copies are already in flight.
//
// Every wait is bounded (arf::mbar_wait_bounded); a wait that runs out sets
// the workspace error word, the CTA stops issuing, drains its own copies and
// returns.
//
// Operation: sglang PR #37196 "[Comm] Share the CuTe DSL AR fusion core and
// wire it for DeepSeek-V3 / GLM-5.x", Motivation and Modifications sections
// 1-2; sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with final
// RMSNorm", Changes.
#include "arf_common.cuh"

namespace arf {

constexpr int kStreamMaxConsumers = 512;
constexpr int kStreamMaxThreads = 32 + kStreamMaxConsumers;
constexpr int kStreamMaxStages = 32;

// Shared-memory header: full[nstages], empty[nstages] mbarriers, the per-row
// sum-of-squares partials [2][32] and the abort flag; the ring follows at a
// 128-byte boundary.
__host__ __device__ constexpr int stream_ring_offset(int nstages) {
    return ((nstages * 16 + 2 * 32 * 4 + 16) + 127) / 128 * 128;
}

template <int CPT, bool RES_F32>
__global__ void __launch_bounds__(kStreamMaxThreads, 1)
    stream_rows_kernel(const __grid_constant__ RowArgs a, int nstages, int stage_bytes) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + nstages;
    float* red = reinterpret_cast<float*>(empty + nstages);        // [2][32]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 64);
    uint8_t* ring = smem + stream_ring_offset(nstages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ncw = (blockDim.x >> 5) - 1;  // consumer warps

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), (uint32_t)ncw);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int H = a.H;
    const int nS = a.has_shared ? a.R : 0;
    const uint32_t row_bytes = (uint32_t)H * 2u;

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first_policy();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0, last_par = 0;  // per-stage bits, for the drain
        bool ok = true;
        auto issue = [&](const void* src) -> bool {
            if (!mbar_wait_bounded(smem_addr(&empty[stage]), phase ^ 1u, abort_flag)) {
                if (!*abort_flag) atomicOr(a.err, kErrTimeout);
                *abort_flag = 1;
                return false;
            }
            const uint32_t fb = smem_addr(&full[stage]);
            mbar_arrive_expect_tx(fb, row_bytes);
            bulk_g2s(smem_addr(ring + (size_t)stage * stage_bytes), src, row_bytes, fb, pol);
            issued |= 1u << stage;
            last_par = (last_par & ~(1u << stage)) | (phase << stage);
            if (++stage == nstages) {
                stage = 0;
                phase ^= 1u;
            }
            return true;
        };
        for (int64_t t = blockIdx.x; t < a.T && ok; t += gridDim.x) {
            int32_t prow[kMaxTopK];
#pragma unroll
            for (int k = 0; k < kMaxTopK; ++k)
                if (k < a.K) prow[k] = __ldg(a.perm + t * a.K + k);
            for (int r = 0; r < nS && ok; ++r) ok = issue(a.S[r] + t * H);
            if (ok) ok = issue(a.residual + t * H);
#pragma unroll
            for (int k = 0; k < kMaxTopK; ++k) {
                if (k < a.K && ok) {
                    const int64_t row = checked_row(prow[k], a.rows_e, a.err);
                    for (int r = 0; r < a.R && ok; ++r) ok = issue(a.E[r] + row * H);
                }
            }
        }
        // Never leave with a copy still landing in this CTA's shared memory.
        for (int s = 0; s < nstages; ++s)
            if ((issued >> s) & 1u) (void)mbar_wait_bounded(smem_addr(&full[s]), (last_par >> s) & 1u, nullptr);
        return;
    }

    // ----------------------------------------------------------- consumers
    const int ci = threadIdx.x - 32;
    const int nct = ncw * 32;
    const int chunks = H / 8;
    int chunk[CPT];
    bool valid[CPT];
    float gw[CPT][8];
#pragma unroll
    for (int m = 0; m < CPT; ++m) {
        chunk[m] = ci + m * nct;
        valid[m] = chunk[m] < chunks;
        if (valid[m]) {
            float gf[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.gamma + (size_t)chunk[m] * 8), gf);
#pragma unroll
            for (int j = 0; j < 8; ++j) gw[m][j] = gf[j] + a.weight_bias;
        }
    }

    int stage = 0;
    uint32_t phase = 0;
    int par = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        float wk[kMaxTopK];
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
            if (k < a.K) wk[k] = __ldg(a.w + t * a.K + k);
        float acc[CPT][8];
#pragma unroll
        for (int m = 0; m < CPT; ++m)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[m][j] = 0.0f;

        auto consume = [&](float coef) {
            if (ok && !mbar_wait_bounded(smem_addr(&full[stage]), phase, abort_flag)) {
                ok = false;
                if (!*abort_flag) atomicOr(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            const uint4* sp = reinterpret_cast<const uint4*>(ring + (size_t)stage * stage_bytes);
#pragma unroll
            for (int m = 0; m < CPT; ++m) {
                if (valid[m]) {
                    float f[8];
                    bf16x8_to_f32(sp[chunk[m]], f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[m][j] = fmaf(coef, f[j], acc[m][j]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty[stage]));
            if (++stage == nstages) {
                stage = 0;
                phase ^= 1u;
            }
        };

        for (int r = 0; r < nS; ++r) consume(1.0f);
        consume(1.0f);  // residual
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
            if (k < a.K)
                for (int r = 0; r < a.R; ++r) consume(wk[k]);

        // Row epilogue, all on chip: residual_out, sum of squares, out.
        float ss = 0.0f;
#pragma unroll
        for (int m = 0; m < CPT; ++m) {
            if (valid[m]) {
#pragma unroll
                for (int j = 0; j < 8; ++j) ss = fmaf(acc[m][j], acc[m][j], ss);
                store_residual8<RES_F32>(a.residual_out, t * H + (int64_t)chunk[m] * 8, acc[m]);
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) red[par * 32 + (warp - 1)] = ss;
        named_barrier_sync(1, nct);
        float tot = 0.0f;
        for (int w = 0; w < ncw; ++w) tot += red[par * 32 + w];
        const float inv = rsqrtf(tot / (float)H + a.eps);
#pragma unroll
        for (int m = 0; m < CPT; ++m) {
            if (valid[m]) {
                float o[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = acc[m][j] * inv * gw[m][j];
                st_global16(reinterpret_cast<uint16_t*>(a.out) + t * H + (int64_t)chunk[m] * 8,
                            f32x8_to_bf16x8(o));
            }
        }
        par ^= 1;
    }
}

template <int CPT, bool RES_F32>
static cudaError_t set_attr_one(int smem_bytes) {
    return cudaFuncSetAttribute(stream_rows_kernel<CPT, RES_F32>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t stream_rows_set_attributes(int smem_bytes) {
    cudaError_t e;
    if ((e = set_attr_one<1, false>(smem_bytes)) != cudaSuccess) return e;
    if ((e = set_attr_one<1, true>(smem_bytes)) != cudaSuccess) return e;
    if ((e = set_attr_one<2, false>(smem_bytes)) != cudaSuccess) return e;
    if ((e = set_attr_one<2, true>(smem_bytes)) != cudaSuccess) return e;
    if ((e = set_attr_one<4, false>(smem_bytes)) != cudaSuccess) return e;
    return set_attr_one<4, true>(smem_bytes);
}

bool plan_stream_rows(int H, int smem_optin, StreamPlan* p) {
    const int chunks = H / 8;
    int cpt = 1;
    while (cpt < 4 && chunks > cpt * kStreamMaxConsumers) cpt <<= 1;
    if (chunks > cpt * kStreamMaxConsumers) return false;
    const int consumers = (chunks + cpt - 1) / cpt;
    const int ncw = (consumers + 31) / 32;
    const int stage_bytes = (H * 2 + 127) / 128 * 128;
    int nstages = kStreamMaxStages;
    while (nstages > 2 && stream_ring_offset(nstages) + nstages * stage_bytes > smem_optin)
        --nstages;
    if (stream_ring_offset(nstages) + nstages * stage_bytes > smem_optin) return false;
    p->cpt = cpt;
    p->threads = 32 * (ncw + 1);
    p->nstages = nstages;
    p->stage_bytes = stage_bytes;
    p->smem = stream_ring_offset(nstages) + nstages * stage_bytes;
    p->ctas_per_sm = 1;
    return true;
}

cudaError_t launch_stream_rows(const RowArgs& a, const StreamPlan& p, int grid, bool res_f32,
                               cudaStream_t stream) {
    const dim3 g((unsigned)grid), b((unsigned)p.threads);
    const size_t sm = (size_t)p.smem;
#define ARF_LAUNCH(CPT_)                                                                    \
    do {                                                                                    \
        if (res_f32)                                                                        \
            stream_rows_kernel<CPT_, true><<<g, b, sm, stream>>>(a, p.nstages, p.stage_bytes); \
        else                                                                                \
            stream_rows_kernel<CPT_, false><<<g, b, sm, stream>>>(a, p.nstages, p.stage_bytes); \
    } while (0)
    switch (p.cpt) {
        case 1: ARF_LAUNCH(1); break;
        case 2: ARF_LAUNCH(2); break;
        case 4: ARF_LAUNCH(4); break;
        default: return cudaErrorInvalidValue;
    }
#undef ARF_LAUNCH
    return cudaGetLastError();
}

}  // namespace arf

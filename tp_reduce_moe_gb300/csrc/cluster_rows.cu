// cluster_rows.cu -- small-T (decode) kernel: one thread-block cluster per
// token row.
//
// At decode sizes (1..~128 tokens) one row carries ~1 MB of gathered expert
// data (R*K rows of H bf16), so a row must be spread over many SMs to get
// enough loads in flight.  The row's H columns are split over the C CTAs of
// a cluster (C <= 16), and inside a CTA the R*(K+1) summands of each 16-byte
// column chunk are split over G thread groups, each thread issuing all of
// its (<= 8) 16-byte loads at once.  Group partials meet in shared memory,
// the row's sum of squares meets across the cluster in distributed shared
// memory, and every CTA normalises and stores its own columns.  Rows of at
// most two loads per thread (the all-reduce of two partials) run an
// instantiation capped at 40 registers, twice the resident CTAs of the
// generic one (80): at T = 128 a call takes 4.8 us instead of 7.1.
//
// Operation: sglang PR #37196 "[Comm] Share the CuTe DSL AR fusion core and
// wire it for DeepSeek-V3 / GLM-5.x", Motivation and Modifications sections
// 1-2 (finalize + shared add + all-reduce folded into the next input RMSNorm,
// scale gamma + weight_bias); sglang PR #37104 "perf(mtp): fuse trailing TP
// all-reduce with final RMSNorm", Changes (K = 0 form, residual required).
#include "arf_host.h"

namespace arf {

constexpr int kClusterMaxTerms = 8;     // 16-byte loads in flight per thread
constexpr int kClusterMaxThreads = 768;

// Grid: T*C CTAs, clusters of C along x; CTA c of a cluster owns chunks
// [c*nch, min((c+1)*nch, H/8)) of row t = blockIdx.x / C (the last CTA of a
// row may be ragged).  blockDim.x = nch * G.  Term q of a thread group:
// q < nS is shared partial S_q; otherwise e = q - nS selects slot k = e / R
// of rank r = e % R.
template <bool RES_F32, int MAXT, int MAX_THREADS, int MIN_BLOCKS>
__global__ void __launch_bounds__(MAX_THREADS, MIN_BLOCKS)
    cluster_rows_kernel(const __grid_constant__ RowArgs a, int C, int nch, int G) {
    extern __shared__ __align__(16) uint8_t dyn_smem[];
    pdl_trigger();
    float4* red = reinterpret_cast<float4*>(dyn_smem);  // [G-1][2][nch]
    __shared__ int64_t s_row[kMaxTopK];
    __shared__ float s_w[kMaxTopK];
    __shared__ float s_warp[32];
    __shared__ float s_parts[16];  // every CTA's sum of squares, pushed in by the CTAs
    __shared__ __align__(8) uint64_t s_bar;  // C * 4 bytes of pushed sums
    __shared__ int s_abort;

    const int tid = threadIdx.x;
    const int64_t t = blockIdx.x / C;
    const uint32_t c = (C > 1) ? cluster_ctarank() : 0u;
    const int i = tid % nch;
    const int g = tid / nch;
    const int H = a.H;
    const int chunk = (int)c * nch + i;
    const bool active = chunk < H / 8;  // ragged last CTA of a row
    const int64_t col = (int64_t)chunk * 8;
    const int nS = a.has_shared ? a.R : 0;
    const int NT = active ? nS + a.R * a.K : 0;
    const int64_t rowoff = t * H + col;

    // Every load that needs no routing metadata -- gamma (needed only at the
    // end), the routing metadata itself, the shared partials, the residual --
    // is requested first, with loads the compiler keeps in place, so their
    // memory round trips overlap the barrier set-up below.
    pdl_wait();  // no global memory access before this point
    uint4 gv = make_uint4(0, 0, 0, 0);
    if (g == 0 && active) gv = ld_early16(a.gamma + col);
    // Pass 1: loads that do not depend on the routing metadata.
    uint4 v[MAXT];
    float coef[MAXT];
    const float s_coef = shared_coef(a, t);
#pragma unroll
    for (int m = 0; m < MAXT; ++m) {
        const int q = g + m * G;
        if (q < nS && q < NT) {
            v[m] = ld_stream16(a.S[q] + rowoff);
            coef[m] = s_coef;
        }
    }
    uint4 res = make_uint4(0, 0, 0, 0);
    if (g == 0 && active) res = ld_stream16(a.residual + rowoff);

    // The exchange barrier exists (and expects its C pushed sums) before any
    // peer may push: cluster barrier arrived on after the block barrier below,
    // waited on before the push.  The last thread sets it up while threads
    // k < K wait for the routing metadata.
    if (tid == (int)blockDim.x - 1) {
        mbar_init(smem_addr(&s_bar), 1);
        s_abort = 0;
        fence_mbar_init();
        mbar_arrive_expect_tx(smem_addr(&s_bar), (uint32_t)C * 4u);
    }
    for (int k = tid; k < a.K; k += blockDim.x) {
        s_row[k] = checked_row(a.perm[t * a.K + k], a.rows_e, a.err);
        s_w[k] = a.w[t * a.K + k];
    }
    __syncthreads();
    if (C > 1) cluster_arrive_relaxed();

    // Pass 2: the routed (gathered) expert rows.
#pragma unroll
    for (int m = 0; m < MAXT; ++m) {
        const int q = g + m * G;
        if (q >= nS && q < NT) {
            const int e = q - nS;
            const int k = e / a.R;
            const int r = e - k * a.R;
            v[m] = ld_stream16(a.E[r] + s_row[k] * H + col);
            coef[m] = s_w[k];
        }
    }

    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
#pragma unroll
    for (int m = 0; m < MAXT; ++m) {
        if (g + m * G < NT) {
            float f[8];
            bf16x8_to_f32(v[m], f);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = fmaf(coef[m], f[j], acc[j]);
        }
    }

    // Group partials meet in shared memory; group 0 finishes the columns.
    if (g > 0) {
        float4* dst = red + (size_t)(g - 1) * 2 * nch + i;
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[nch] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    __syncthreads();

    float h[8];
    float ss = 0.0f;
    if (g == 0 && active) {
        for (int gg = 1; gg < G; ++gg) {
            const float4 x = red[(size_t)(gg - 1) * 2 * nch + i];
            const float4 y = red[(size_t)(gg - 1) * 2 * nch + nch + i];
            acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
            acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
        }
        float rf[8];
        bf16x8_to_f32(res, rf);
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = acc[j] + rf[j];
        store_residual8<RES_F32>(a.residual_out, rowoff, h);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            h[j] = norm_input(h[j], a.norm_bf16_h);
            ss = fmaf(h[j], h[j], ss);
        }
    }

    // Row sum of squares: warps -> CTA -> cluster (fixed order everywhere,
    // so every CTA of the row derives the same scale).
    ss = warp_sum(ss);
    if ((tid & 31) == 0) s_warp[tid >> 5] = ss;
    __syncthreads();
    float total;
    if (C > 1) {
        // Thread rk (and rk + blockDim, ...) sums the CTA's warps and pushes
        // the CTA's sum into peer rk (asynchronous remote stores counted on
        // the peer's barrier);
        // every thread waits for the C sums of the row.  No exit barrier:
        // the pushes are the only remote accesses, and a CTA leaves only
        // after every peer's push into it has landed.
        cluster_wait_acquire();  // every peer's barrier exists
        if (tid < C) {  // a block may have fewer threads than the cluster has CTAs
            float tot = 0.0f;
            const int nw = (blockDim.x + 31) >> 5;
            for (int w = 0; w < nw; ++w) tot += s_warp[w];
            for (int rk = tid; rk < C; rk += blockDim.x)
                st_async_remote_f32(map_shared_rank(smem_addr(&s_parts[c]), (uint32_t)rk), tot,
                                    map_shared_rank(smem_addr(&s_bar), (uint32_t)rk));
        }
        if (!mbar_wait_bounded<true>(smem_addr(&s_bar), 0u, reinterpret_cast<volatile int*>(&s_abort))) {
            if (!s_abort) atomicOr(a.err, kErrTimeout);
            s_abort = 1;
        }
        total = sum_slots(s_parts, C);
    } else {
        total = 0.0f;
        const int nw = (blockDim.x + 31) >> 5;
        for (int w = 0; w < nw; ++w) total += s_warp[w];
    }

    if (g == 0 && active) {
        const float inv = rsqrtf(total / (float)H + a.eps);
        float gf[8], o[8];
        bf16x8_to_f32(gv, gf);
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = h[j] * inv * (gf[j] + a.weight_bias);
        st_global16(reinterpret_cast<uint16_t*>(a.out) + rowoff, f32x8_to_bf16x8(o));
    }
    // after a wait that ran out: let pushes still in flight land first
    if (C > 1 && tid == 0 && s_abort) grace_period(1000000ull);
}

static int ceil_div_c(int a, int b) { return (a + b - 1) / b; }

bool plan_cluster_rows(int R, int K, int H, bool shared, int max_c, int64_t T, int num_sms,
                       ClusterPlan* p, int force_c) {
    const int chunks = H / 8;
    const int NT = (shared ? R : 0) + R * K;
    if (NT < 1 || chunks < 1) return false;
    const int G = ceil_div_c(NT, kClusterMaxTerms);
    if (G > kClusterMaxThreads) return false;
    // Enough CTAs to cover the GPU about twice over, unless the caller fixes
    // the cluster size (a power of two up to 16: fewer, larger CTAs launch
    // and exchange sooner, which can beat the coverage rule at small T).
    int want = 1;
    while (want < 16 && (int64_t)want * T < 2LL * num_sms) want <<= 1;
    if (force_c > 0 && (force_c > 16 || (force_c & (force_c - 1)))) return false;
    int best = 0, largest = 0;
    for (int C = 1; C <= 16 && C <= max_c && C <= chunks; C <<= 1) {
        const int nch = ceil_div_c(chunks, C);
        if (nch * G > kClusterMaxThreads) continue;
        if (force_c > 0) {
            if (C == force_c) best = C;
            continue;
        }
        largest = C;
        if (!best && C >= want) best = C;
    }
    if (!best && force_c > 0) return false;
    if (!best) best = largest;
    if (!best) return false;
    p->C = best;
    p->nch = ceil_div_c(chunks, best);
    p->G = G;
    // loads per thread, rounded up to an instantiated bound: at most two
    // (light rows, e.g. the K = 0 all-reduce of two partials) fits 40
    // registers, so twice the CTAs are resident per SM
    const int terms = ceil_div_c(NT, G);
    p->maxt = terms <= 2 ? 2 : kClusterMaxTerms;
    p->threads = p->nch * G;
    p->smem = (G - 1) * 2 * p->nch * (int)sizeof(float4);
    return true;
}

// The kernel instantiation for (residual_out type, loads per thread):
// maxt 2 -- two loads, 40 registers (two blocks of 768 threads per SM);
// maxt 8 -- eight loads, 80 registers (one block of 768 threads);
// kClusterMaxTerms64 -- eight loads in 64 registers, blocks of at most 512
// threads, two per SM (more resident CTAs once a launch no longer fits one
// wave of the 80-register form; 4 bytes of spills).
static const void* cluster_kernel_for(bool res_f32, int maxt) {
    if (maxt == 2) return res_f32 ? reinterpret_cast<const void*>(cluster_rows_kernel<true, 2, 768, 2>)
                                  : reinterpret_cast<const void*>(cluster_rows_kernel<false, 2, 768, 2>);
    if (maxt == kClusterMaxTerms)
        return res_f32 ? reinterpret_cast<const void*>(cluster_rows_kernel<true, kClusterMaxTerms, 768, 1>)
                       : reinterpret_cast<const void*>(cluster_rows_kernel<false, kClusterMaxTerms, 768, 1>);
    if (maxt == kClusterMaxTerms64)
        return res_f32 ? reinterpret_cast<const void*>(cluster_rows_kernel<true, kClusterMaxTerms, 512, 2>)
                       : reinterpret_cast<const void*>(cluster_rows_kernel<false, kClusterMaxTerms, 512, 2>);
    return nullptr;
}

// Whether an eight-load plan for T rows should run the 64-register form,
// given the resident blocks per SM of each form: only when the launch does
// not fit one wave of the 80-register form and the 64-register form holds
// more blocks.
bool oneshot_prefer_64(const ClusterPlan& p, int64_t T, int num_sms, int blocks80, int blocks64) {
    if (p.maxt != kClusterMaxTerms || p.threads > 512) return false;
    return T * p.C > (int64_t)blocks80 * num_sms && blocks64 > blocks80;
}

// Resident blocks per SM of a plan's kernel instantiation (0 on error).
int cluster_rows_blocks_per_sm(const ClusterPlan& p, bool res_f32) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, cluster_kernel_for(res_f32, p.maxt), p.threads,
                                                      (size_t)p.smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t cluster_rows_set_attributes() {
    for (int f = 0; f < 2; ++f)
        for (int maxt : {2, kClusterMaxTerms, kClusterMaxTerms64}) {
            cudaError_t e = cudaFuncSetAttribute(cluster_kernel_for(f != 0, maxt),
                                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

static cudaLaunchConfig_t cluster_config(const ClusterPlan& p, int64_t T, cudaStream_t s,
                                         cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(T * p.C), 1, 1);
    cfg.blockDim = dim3((unsigned)p.threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)p.smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Largest cluster size (<= 16) the device can co-schedule for a block of
// this shape, 0 if even a single CTA cannot run.
int cluster_rows_max_cluster(int threads, int smem, bool res_f32) {
    for (int C = 16; C >= 1; C >>= 1) {
        cudaLaunchAttribute attr[1];
        ClusterPlan p{C, 1, 1, threads, smem, kClusterMaxTerms};
        cudaLaunchConfig_t cfg = cluster_config(p, 1, nullptr, attr);
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&n, cluster_kernel_for(res_f32, kClusterMaxTerms), &cfg);
        if (e == cudaSuccess && n > 0) return C;
        (void)cudaGetLastError();
    }
    return 0;
}

// Whether the device can co-schedule one cluster of exactly this plan's launch
// (block size, shared memory, cluster size, kernel instantiation).
bool cluster_rows_plan_fits(const ClusterPlan& p, bool res_f32) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(p, 1, nullptr, attr);
    cfg.gridDim = dim3((unsigned)p.C, 1, 1);
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, cluster_kernel_for(res_f32, p.maxt), &cfg);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e == cudaSuccess && n > 0;
}

cudaError_t launch_cluster_rows(const RowArgs& a, const ClusterPlan& p, bool res_f32,
                                cudaStream_t stream, bool pdl) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = cluster_config(p, a.T, stream, attr);
    if (pdl) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    const void* k = cluster_kernel_for(res_f32, p.maxt);
    if (!k) return cudaErrorInvalidValue;
    int C = p.C, nch = p.nch, G = p.G;
    void* args[] = {const_cast<RowArgs*>(&a), &C, &nch, &G};
    return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace arf

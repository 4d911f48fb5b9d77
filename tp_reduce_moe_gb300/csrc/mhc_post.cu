// mhc_post.cu -- all-reduce + mHC residual write-back ("hc_post") in one pass.
//
// An mHC layer writes its FFN output back in two steps: the FFN's
// tensor-parallel all-reduce, then hc_post, which reads the reduced output
// back and mixes it into the hc_mult residual streams (sglang PR #42020,
// Summary and Scope: four streams, at most 16 tokens where the fused form is
// used).  The page gives no formula for the mix; the library computes the
// per-token linear mix
//
//   y[t,j]     = sum_{r<R} P_r[t,j]                                (fp32)
//   out[t,i,j] = post[t,i] * y[t,j] + sum_{k<hc} comb[t,i,k] * x[t,k,j]
//
// with P_r bf16 [T, H], x / out bf16 [T, hc, H], post fp32 [T, hc], comb fp32
// [T, hc, hc].  The reduced output y never leaves registers.
//
// One thread per (token, 16-byte column chunk): all R partial chunks and all
// hc stream chunks are loaded before any arithmetic (R + hc independent
// 16-byte loads in flight per thread, in batches of eight), so a call at
// decode sizes costs about one memory round trip plus launch.  The token's
// coefficients are staged in shared memory.  Every input byte is read once
// and every output byte written once; `out` may be `x` itself (each thread
// reads all of its chunk's streams before it writes any of them, and no
// other thread touches that chunk), so the stream loads use the coherent
// path.
#include "arf_host.h"

namespace arf {

constexpr int kMhcThreads = 128;  // chunks (of 8 columns) per CTA
constexpr int kMhcMaxStreams = 8;

template <int HC>
__global__ void __launch_bounds__(kMhcThreads)
    mhc_post_kernel(const __grid_constant__ MhcArgs a) {
    pdl_trigger();
    pdl_wait();  // no global memory access before this point
    __shared__ float s_post[kMhcMaxStreams];
    __shared__ float s_comb[kMhcMaxStreams * kMhcMaxStreams];
    const int hc = HC > 0 ? HC : a.hc;
    const int chunks = a.H / 8;
    const int per_token = (chunks + kMhcThreads - 1) / kMhcThreads;
    const int64_t t = blockIdx.x / per_token;
    const int chunk = (int)(blockIdx.x % per_token) * kMhcThreads + threadIdx.x;
    // The token's coefficients go to registers first and to shared memory
    // only after the data loads are out: a warp issues in order, so storing
    // a load's value stalls it until the value arrives, and would hold back
    // the loads behind it by a memory round trip.
    const int nq = hc * hc;  // <= 64 < kMhcThreads
    float comb_v = 0.0f, post_v = 0.0f;
    if ((int)threadIdx.x < nq) comb_v = __ldg(a.comb + t * nq + threadIdx.x);
    if ((int)threadIdx.x < hc) post_v = __ldg(a.post + t * hc + threadIdx.x);

    float y[8];
    uint4 xv[kMhcMaxStreams];
    const bool active = chunk < chunks;
    if (active) {
        const int64_t col = (int64_t)chunk * 8;
        // the incoming streams first (coherent loads: `out` may alias them)
#pragma unroll
        for (int k = 0; k < kMhcMaxStreams; ++k)
            if (k < hc) {
                const uint16_t* p = a.x + (t * hc + k) * (int64_t)a.H + col;
                xv[k] = *reinterpret_cast<const uint4*>(p);
            }
        // the all-reduce, eight partials in flight at a time, rank order
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = 0.0f;
        for (int r0 = 0; r0 < a.R; r0 += 8) {
            uint4 pv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (r0 + u < a.R) pv[u] = ld_stream16(a.P[r0 + u] + t * a.H + col);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (r0 + u < a.R) {
                    float f[8];
                    bf16x8_to_f32(pv[u], f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) y[j] += f[j];
                }
        }
    }
    if ((int)threadIdx.x < nq) s_comb[threadIdx.x] = comb_v;
    if ((int)threadIdx.x < hc) s_post[threadIdx.x] = post_v;
    __syncthreads();  // coefficients staged
    if (!active) return;
    const int64_t col = (int64_t)chunk * 8;
#pragma unroll
    for (int i = 0; i < kMhcMaxStreams; ++i) {
        if (i >= hc) break;
        float o[8];
        const float pi = s_post[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = pi * y[j];
#pragma unroll
        for (int k = 0; k < kMhcMaxStreams; ++k)
            if (k < hc) {
                const float c = s_comb[i * hc + k];
                float f[8];
                bf16x8_to_f32(xv[k], f);
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = fmaf(c, f[j], o[j]);
            }
        st_global16(a.out + (t * hc + i) * (int64_t)a.H + col, f32x8_to_bf16x8(o));
    }
}

cudaError_t launch_mhc_post(const MhcArgs& a, cudaStream_t stream, bool pdl) {
    const int chunks = a.H / 8;
    const int per_token = (chunks + kMhcThreads - 1) / kMhcThreads;
    const int64_t grid = a.T * per_token;
    if (grid < 1 || grid > 0x7fffffff) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kMhcThreads);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return a.hc == 4 ? cudaLaunchKernelEx(&cfg, mhc_post_kernel<4>, a) : cudaLaunchKernelEx(&cfg, mhc_post_kernel<0>, a);
}

}  // namespace arf

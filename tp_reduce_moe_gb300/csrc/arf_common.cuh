// arf_common.cuh -- shared device helpers of libarfuse (sm_103a only).
//
// The argument block every kernel receives, bf16 <-> fp32 helpers, and thin
// inline-PTX wrappers for the Blackwell features the kernels use: mbarriers,
// 1-D bulk async copies (cp.async.bulk, the TMA engine's untiled form),
// thread-block-cluster barriers and distributed shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace arf {

constexpr int kMaxRanks = 16;
constexpr int kMaxTopK = 16;

// Device error word bits (same values as AR_DEVERR_* in arfuse.h).
constexpr unsigned kErrPermRange = 0x1u;
constexpr unsigned kErrTimeout = 0x2u;

// Time limit of every spin-wait on an mbarrier: past it the kernel records
// kErrTimeout and stops waiting (it never hangs the GPU).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s
constexpr unsigned kWaitMaxIters = 1u << 30;                // failsafe bound

// Everything one launch needs.  Passed by value as a __grid_constant__ kernel
// parameter: the pointer tables live in the parameter bank, no device table.
struct RowArgs {
    const uint16_t* E[kMaxRanks];  // bf16 [rows_e, H] per rank (K > 0)
    const uint16_t* S[kMaxRanks];  // bf16 [T, H] per rank (has_shared)
    const int32_t* perm;           // [T, K] gather rows into E
    const float* w;                // [T, K] routing weights
    const float* shared_gate;      // [T] gate logits, or nullptr: S scaled by sigmoid(gate[t])
    const uint16_t* residual;      // bf16 [T, H]
    const uint16_t* gamma;         // bf16 [H]
    void* out;                     // bf16 [T, H]
    void* residual_out;            // bf16 or fp32 [T, H]
    unsigned* err;                 // device error word
    float* part_scratch;           // [grid, H] fp32 partial rows of split rows (streaming, C = 1)
    unsigned* part_count;          // [grid] arrival counters of split rows (zero between calls)
    int64_t T;
    int64_t rows_e;
    int R, K, H;
    int has_shared;
    int norm_bf16_h;               // the norm reads h rounded to bf16 (as a bf16 residual_out stores it)
    float weight_bias;
    float eps;
    // Failure injection (whole-row streaming only; 0 = off): the consumers'
    // first wait targets a barrier nothing arrives on, bounded by this many
    // nanoseconds, so the call takes its timeout path (tests of that path).
    unsigned long long stall_wait_ns;
};

// Coefficient of the shared partials of row t: sigmoid of the row's gate
// logit for a gated shared expert, else 1.
__device__ __forceinline__ float shared_coef(const RowArgs& a, int64_t t) {
    return a.shared_gate ? 1.0f / (1.0f + expf(-__ldg(a.shared_gate + t))) : 1.0f;
}

// h as the norm reads it: unrounded, or rounded to bf16 (round to nearest even).
__device__ __forceinline__ float norm_input(float h, int bf16) {
    return bf16 ? __bfloat162float(__float2bfloat16_rn(h)) : h;
}

// ------------------------------------------------------------------ bf16 data
// A bf16 value is the top half of an IEEE binary32 word, so widening is a
// shift; eight of them travel as one 16-byte vector.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float f[8]) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

// acc[0..7] += c * (the 8 bf16 of v), as four packed fp32x2 fused
// multiply-adds (fma.rn.f32x2: two independent round-to-nearest FMAs, so the
// result is bit-identical to eight scalar fmaf).  Decoding a bf16 pair costs
// one shift and one mask, so a pair of elements takes three instructions
// instead of four.
__device__ __forceinline__ void fma_bf16x8(float acc[8], float c, const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float lo = __uint_as_float(w[q] << 16), hi = __uint_as_float(w[q] & 0xffff0000u);
        asm("{\n\t.reg .b64 a2, x2, c2;\n\t"
            "mov.b64 a2, {%0, %1};\n\t"
            "mov.b64 x2, {%2, %3};\n\t"
            "mov.b64 c2, {%4, %4};\n\t"
            "fma.rn.f32x2 a2, c2, x2, a2;\n\t"
            "mov.b64 {%0, %1}, a2;\n\t}"
            : "+f"(acc[2 * q]), "+f"(acc[2 * q + 1])
            : "f"(lo), "f"(hi), "f"(c));
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ uint4 f32x8_to_bf16x8(const float f[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

// 16-byte streaming load of read-once data: non-coherent path, no L1 line.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// 8- and 16-byte read-only loads issued where they stand: volatile, so the
// compiler keeps them ahead of the barrier waits that follow instead of
// sinking them to their first use (a load of data needed only at the end of
// a row -- gamma -- is requested at kernel start and has long arrived by
// then).
__device__ __forceinline__ uint32_t ld_early4(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_early8(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_early16_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_early16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_global16(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Store residual_out for 8 consecutive columns, bf16 (16 B) or fp32 (32 B).
template <bool RES_F32>
__device__ __forceinline__ void store_residual8(void* base, int64_t elem, const float h[8]) {
    if (RES_F32) {
        float* p = reinterpret_cast<float*>(base) + elem;
        st_global16(p, make_uint4(__float_as_uint(h[0]), __float_as_uint(h[1]),
                                  __float_as_uint(h[2]), __float_as_uint(h[3])));
        st_global16(p + 4, make_uint4(__float_as_uint(h[4]), __float_as_uint(h[5]),
                                      __float_as_uint(h[6]), __float_as_uint(h[7])));
    } else {
        st_global16(reinterpret_cast<uint16_t*>(base) + elem, f32x8_to_bf16x8(h));
    }
}

// Routed row of slot (t, k), checked against rows_e.  An out-of-range value
// is clamped into range (so no load ever leaves the buffer) and flagged.
__device__ __forceinline__ int64_t checked_row(int32_t p, int64_t rows_e, unsigned* err) {
    if ((uint64_t)(int64_t)p >= (uint64_t)rows_e) {
        atomicOr(err, kErrPermRange);
        return p < 0 ? 0 : rows_e - 1;
    }
    return p;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns();

// After a wait has run out (an error path only): keep the CTA resident for
// `ns` nanoseconds so that asynchronous copies and stores still in flight to
// or from its shared memory land before it exits.
__device__ __forceinline__ void grace_period(unsigned long long ns) {
    const unsigned long long t0 = global_timer_ns();
    for (unsigned it = 0; it < 1000000u && global_timer_ns() - t0 < ns; ++it) __nanosleep(1000);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// try_wait with acquire at cluster scope: for barriers that peers in the
// cluster arrive on remotely (their prior stores become visible).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase of `bar` with the given parity has completed.  Gives
// up (returns false) when *abort becomes non-zero, after limit_ns, or after
// kWaitMaxIters polls, whichever comes first.
template <bool CLUSTER_ACQUIRE = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    auto poll = [&]() {
        return CLUSTER_ACQUIRE ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (poll()) return true;
    const unsigned long long t0 = global_timer_ns();
    for (unsigned it = 1; it < kWaitMaxIters; ++it) {
        if (poll()) return true;
        if ((it & 31u) == 0u) {
            if (abort != nullptr && *abort) return false;
            if (global_timer_ns() - t0 > limit_ns) return false;
        }
    }
    return false;
}

// ------------------------------------------------------- bulk async copy (TMA)
// L2 policy for data read exactly once: evict it first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Copy `bytes` (multiple of 16, both addresses 16-byte aligned) from global
// memory into this CTA's shared memory; completion is signalled on `bar`
// as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Copy `bytes` (multiple of 16, 16-byte aligned) from this CTA's shared
// memory into a peer's shared memory (addresses from map_shared_rank),
// completing as transaction bytes on the peer's mbarrier `remote_bar`.
__device__ __forceinline__ void bulk_s2cluster(uint32_t remote_dst, uint32_t local_src, uint32_t bytes,
                                               uint32_t remote_bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            remote_dst),
        "r"(local_src), "r"(bytes), "r"(remote_bar)
        : "memory");
}

// ------------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Arrive on the cluster barrier without release semantics.  Used right after
// mbarrier initialisation: fence.mbarrier_init.release.cluster (fence_mbar_init)
// already makes the initialised barriers visible at cluster scope, and the
// peers' barrier.cluster.wait acquires; a release arrive here would also wait
// for every earlier memory operation of the thread (measured on GB300: about
// 0.5 us at kernel start, on the critical path of every decode call).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// Sum of the C per-CTA partials pushed into `slots`, in rank order (every CTA
// of a cluster sums the same values in the same order, so all derive the same
// scale).  Plain loads, issued together: the caller has already waited
// (acquire) on the barrier that counted the pushes.
__device__ __forceinline__ float sum_slots(const float* slots, int C) {
    float v[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) v[r] = r < C ? slots[r] : 0.0f;
    float total = 0.0f;
#pragma unroll
    for (int r = 0; r < 16; ++r)
        if (r < C) total += v[r];
    return total;
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Programmatic dependent launch.  The decode kernels let the next kernel in
// the stream start launching as soon as they start (launch_dependents), the
// streaming kernel as each of its CTAs finishes; every kernel waits
// (griddepcontrol.wait) for the previous kernel to complete and flush its
// memory before its first global memory access: with the launch attribute,
// launch latency and prologue overlap the previous kernel's tail; without
// it both instructions return at once.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Store 4 bytes into a peer CTA's shared memory (addresses from
// map_shared_rank) as an asynchronous store that completes as 4 transaction
// bytes on the peer's mbarrier: no release fence, so it does not wait for the
// issuing thread's earlier global stores; the value is visible to whoever
// observes the barrier's phase complete.
__device__ __forceinline__ void st_async_remote_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr),
                 "r"(__float_as_uint(v)), "r"(remote_bar)
                 : "memory");
}

// Named barrier over a subset of the CTA's warps (id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------ kernel parameters
// Each ring slot starts with a header holding the coefficient of each of its
// segments (1 for shared partials and the residual, w[t,k] for routed rows).
constexpr int kSlotHeader = 128;

// Geometry of one stream_rows launch (kernel parameter).
struct StreamGeom {
    int nstages;      // ring slots
    int slot_bytes;   // bytes per slot: kSlotHeader + seg_per_stage * seg_stride
    int seg_per_stage;  // segments (one bulk copy each) sharing one slot and one mbarrier
    int seg_stride;   // bytes between the segments of a slot (>= tile bytes, multiple of 128)
    int C;            // CTAs per token row (cluster size); 1 = whole rows per CTA
    int tile_chunks;  // 16-byte column chunks per CTA tile (the row's last tile may be shorter)
    int producers;    // producer warps (slot q is filled by warp q % producers)
    int64_t main_rows;  // rows [0, main_rows) whole, round-robin; the rest split (C = 1 only)
    int tail_parts;     // segment intervals per split row (1: no split rows)
};

// Geometry of one split_rows launch (kernel parameter).
struct SplitGeom {
    int C;            // CTAs per row (cluster size) = Cs * column groups
    int Cs;           // CTAs per column group; CTA c = g*Cs + cs copies segments cs, cs+Cs, ...
    int group_chunks;  // 16-byte chunks of a column group (the last group may be shorter)
    int seg_stride;   // bytes between segment buffers in shared memory
    int part_bytes;   // bytes of the fp32 receive buffer (Cs slices of a column tile)
    int row_f32_bytes;  // bytes of the CTA's fp32 partial row (over the segment buffers)
    int tile_chunks;  // 16-byte chunks of the column tile each CTA finishes
    int rounds;       // 1: every segment buffered at once; 2: the second routed half
                      // reuses the first buffers once they are folded
};

// Arguments of the all-reduce + mHC write-back (mhc_post.cu).
struct MhcArgs {
    const uint16_t* P[16];  // R partials, bf16 [T, H]
    const uint16_t* x;      // incoming streams, bf16 [T, hc, H]
    const float* post;      // [T, hc]
    const float* comb;      // [T, hc, hc]
    uint16_t* out;          // outgoing streams, bf16 [T, hc, H] (may be x)
    int64_t T;
    int R, H, hc;
};

}  // namespace arf

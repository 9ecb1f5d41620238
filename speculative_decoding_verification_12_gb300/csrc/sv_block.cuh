// sv_block.cuh -- warp/block primitives used by the row kernel: deterministic reductions and
// scans (fixed association, so repeated runs are bitwise identical), order keys for floats,
// a shared-memory bitonic sort, vectorised row loads and the token-weight function.
#pragma once

#include <cuda_bf16.h>

#include "sv_common.cuh"

namespace sv {

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }

// 2^x via the SFU (ex2.approx, flush-to-zero); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Token weight e = 2^((z - m) * s), rounded the same way at every call site.
__device__ __forceinline__ float weight(float z, float m, float s) {
    return ex2(__fmul_rn(__fsub_rn(z, m), s));
}

// Order-preserving uint32 key of a float: a < b  <=>  fkey(a) < fkey(b) (for non-NaN); -0 and
// +0 share the key of +0, so equal values always tie.
__device__ __forceinline__ uint32_t fkey(float z) {
    uint32_t b = z == 0.f ? 0u : __float_as_uint(z);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// Warp-wide max of a float in one instruction (redux.sync, sm_100 family).
__device__ __forceinline__ float redux_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// A group of NTH threads (whole warps) that synchronises on named barrier BAR (0: the whole
// CTA via __syncthreads).  Reductions combine per-warp partials in warp order, so they are
// deterministic.
template <int NTH, int BAR>
struct Grp {
    static constexpr int kThreads = NTH;
    static constexpr int kWarps = NTH / 32;
    int t;   // thread index within the group
    __device__ __forceinline__ explicit Grp(int t_) : t(t_) {}
    __device__ __forceinline__ int warp() const { return t >> 5; }
    __device__ __forceinline__ int lane() const { return t & 31; }
    __device__ __forceinline__ void sync() const {
        if constexpr (BAR == 0) {
            __syncthreads();
        } else {
            asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NTH) : "memory");
        }
    }
};

// A group of NTH threads (whole warps) synchronised on a named barrier chosen at run time.
template <int NTH>
struct GrpR {
    static constexpr int kThreads = NTH;
    static constexpr int kWarps = NTH / 32;
    int t;     // thread index within the group
    int bar;   // named barrier id (1..15)
    __device__ __forceinline__ GrpR(int t_, int bar_) : t(t_), bar(bar_) {}
    __device__ __forceinline__ int warp() const { return t >> 5; }
    __device__ __forceinline__ int lane() const { return t & 31; }
    __device__ __forceinline__ void sync() const {
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(NTH) : "memory");
    }
};

template <class G>
__device__ __forceinline__ float g_max(const G &g, float v, float *red) {
    v = warp_max(v);
    if (g.lane() == 0) red[g.warp()] = v;
    g.sync();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < G::kWarps; w++) r = fmaxf(r, red[w]);
    g.sync();
    return r;
}
template <class G>
__device__ __forceinline__ float g_sum(const G &g, float v, float *red) {
    v = warp_sum(v);
    if (g.lane() == 0) red[g.warp()] = v;
    g.sync();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < G::kWarps; w++) r += red[w];
    g.sync();
    return r;
}
template <class G>
__device__ __forceinline__ int g_min_i(const G &g, int v, int *red) {
    v = warp_min_i(v);
    if (g.lane() == 0) red[g.warp()] = v;
    g.sync();
    int r = red[0];
#pragma unroll
    for (int w = 1; w < G::kWarps; w++) r = min(r, red[w]);
    g.sync();
    return r;
}
template <class G>
__device__ __forceinline__ int g_max_i(const G &g, int v, int *red) {
    v = warp_max_i(v);
    if (g.lane() == 0) red[g.warp()] = v;
    g.sync();
    int r = red[0];
#pragma unroll
    for (int w = 1; w < G::kWarps; w++) r = max(r, red[w]);
    g.sync();
    return r;
}
template <class G>
__device__ __forceinline__ int g_sum_i(const G &g, int v, int *red) {
    v = warp_sum_i(v);
    if (g.lane() == 0) red[g.warp()] = v;
    g.sync();
    int r = 0;
#pragma unroll
    for (int w = 0; w < G::kWarps; w++) r += red[w];
    g.sync();
    return r;
}

// In-place inclusive prefix sum of a[0..n) in shared memory.  Thread t sums a contiguous
// chunk; chunk totals are scanned across lanes and warps in a fixed order, so the result is
// deterministic.  a[n-1] ends up holding the total.
template <class G>
__device__ __forceinline__ void g_scan_incl(const G &g, float *a, int n, float *red) {
    const int lane = g.lane(), warp = g.warp();
    const int per = (n + G::kThreads - 1) / G::kThreads;
    const int lo = min(n, g.t * per), hi = min(n, lo + per);
    float t = 0.f;
    for (int j = lo; j < hi; j++) t += a[j];
    float incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    if (lane == 31) red[warp] = incl;
    g.sync();
    float run = 0.f;
    for (int w = 0; w < warp; w++) run += red[w];
    run += excl;
    for (int j = lo; j < hi; j++) {
        run += a[j];
        a[j] = run;
    }
    g.sync();
}

// Sorts keys[0..np) (np a power of two) into descending order.
template <class G>
__device__ __forceinline__ void g_sort_desc(const G &g, unsigned long long *keys, int np) {
    for (int k = 2; k <= np; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int t = g.t; t < (np >> 1); t += G::kThreads) {
                int i1 = (t / j) * 2 * j + (t % j);
                int i2 = i1 + j;
                unsigned long long a = keys[i1], b = keys[i2];
                bool desc = (i1 & k) == 0;
                if (desc ? (a < b) : (a > b)) {
                    keys[i1] = b;
                    keys[i2] = a;
                }
            }
            g.sync();
        }
    }
}

// Exclusive prefix of v across the 32 lanes (lane 0 gets 0) and the warp total.
__device__ __forceinline__ float warp_excl_scan(float v, float &total) {
    const int lane = lane_id();
    float incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    total = __shfl_sync(0xffffffffu, incl, 31);
    float ex = __shfl_up_sync(0xffffffffu, incl, 1);
    return lane == 0 ? 0.f : ex;
}

// Inverse-CDF draw by one warp over w[0..n) held 8 per lane (element lane*8 + j in w8[j]):
// the first element whose running sum exceeds u * W, else the last positive one; -1 when
// no weight is positive.  Running sums associate lane-locally then across lanes (fixed).
__device__ __forceinline__ int warp_draw8(const float w8[8], int n, float u) {
    const int lane = lane_id();
    float pre[8], loc = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        loc += w8[j];
        pre[j] = loc;
    }
    float W;
    float ex = warp_excl_scan(loc, W);
    if (!(W > 0.f)) return -1;
    const float target = __fmul_rn(u, W);
    int pick = 0x7fffffff, last = -1;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        int idx = lane * 8 + j;
        if (idx < n) {
            if (ex + pre[j] > target && pick == 0x7fffffff) pick = idx;
            if (w8[j] > 0.f) last = idx;
        }
    }
    pick = warp_min_i(pick);
    last = warp_max_i(last);
    return pick != 0x7fffffff ? pick : last;
}

__device__ __forceinline__ int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// ------------------------------------------------------------------------------------------
// bulk copies into shared memory, completed on mbarriers (every wait is time-bounded)
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(unsigned long long *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
#ifndef SV_WAIT_HINT
#define SV_WAIT_HINT 10000
#endif
// try_wait that may suspend the thread for up to `ns` nanoseconds while the phase is pending.
__device__ __forceinline__ bool mbar_try_wait_for(unsigned long long *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
// Waits for the phase of `parity` to complete; false once WAIT_NS has passed without it.
// The first polls skip the clock so that the common, short waits stay cheap.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity) {
#if SV_WAIT_HINT > 0
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_for(bar, parity, SV_WAIT_HINT))
        if (global_ns() - t0 > WAIT_NS) return false;
    return true;
#else
    for (int i = 0; i < 256; i++)
        if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > WAIT_NS) return false;
    return true;
#endif
}
// As mbar_wait, for waits that are usually long (a warp idle until the next row): between
// polls the thread sleeps, so that it takes no issue slots from the warps doing work.
__device__ __forceinline__ bool mbar_wait_idle(unsigned long long *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    unsigned ns = 64;
    while (!mbar_try_wait(bar, parity)) {
        __nanosleep(ns);
        ns = ns < 1024 ? ns * 2 : 1024;
        if (global_ns() - t0 > WAIT_NS) return false;
    }
    return true;
}

#ifndef SV_L2POL
#define SV_L2POL 0
#endif
// L2 policy of the streamed rows.  0: evict first (rows streamed once should not displace the
// small per-segment statistics the next kernel reads back); 1: normal; 2: evict last.
__device__ __forceinline__ unsigned long long l2_stream_policy() {
    unsigned long long pol;
#if SV_L2POL == 0
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
#elif SV_L2POL == 1
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
#else
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
#endif
    return pol;
}
// One bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16) that
// completes `bytes` of transaction count on `bar`, with an L2 cache policy.
// Bulk prefetch of `bytes` (a multiple of 16) at a 16-byte aligned global address into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, unsigned long long *bar,
                                         unsigned long long pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// ------------------------------------------------------------------------------------------
// row loads: 8 consecutive elements per lane; elements at or beyond V read as -inf
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

template <typename E>
struct Raw8;

template <>
struct Raw8<uint16_t> {   // 8 x bf16
    uint4 a;
};
template <>
struct Raw8<float> {      // 8 x fp32
    uint4 a, b;
};

__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) { return lo | (hi << 16); }

template <bool VEC>
__device__ __forceinline__ Raw8<uint16_t> load_raw8(const uint16_t *row, int base, int V) {
    Raw8<uint16_t> r;
    if (VEC && base + 8 <= V) {
        r.a = ld_stream_v4(row + base);
    } else {
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 8; j++) h[j] = (base + j < V) ? (uint32_t)__ldg(row + base + j) : 0xFF80u;
        r.a = make_uint4(pack_bf16(h[0], h[1]), pack_bf16(h[2], h[3]), pack_bf16(h[4], h[5]),
                         pack_bf16(h[6], h[7]));
    }
    return r;
}

template <bool VEC>
__device__ __forceinline__ Raw8<float> load_raw8(const float *row, int base, int V) {
    Raw8<float> r;
    if (VEC && base + 8 <= V) {
        r.a = ld_stream_v4(row + base);
        r.b = ld_stream_v4(row + base + 4);
    } else {
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 8; j++) h[j] = (base + j < V) ? __float_as_uint(__ldg(row + base + j)) : 0xFF800000u;
        r.a = make_uint4(h[0], h[1], h[2], h[3]);
        r.b = make_uint4(h[4], h[5], h[6], h[7]);
    }
    return r;
}

__device__ __forceinline__ void unpack8(const Raw8<uint16_t> &r, float v[8]) {
    const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
        v[2 * j] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void unpack8(const Raw8<float> &r, float v[8]) {
    v[0] = __uint_as_float(r.a.x);
    v[1] = __uint_as_float(r.a.y);
    v[2] = __uint_as_float(r.a.z);
    v[3] = __uint_as_float(r.a.w);
    v[4] = __uint_as_float(r.b.x);
    v[5] = __uint_as_float(r.b.y);
    v[6] = __uint_as_float(r.b.z);
    v[7] = __uint_as_float(r.b.w);
}

// fp32 draft-probability row: 8 values from base (0 beyond V).
template <bool VEC>
__device__ __forceinline__ void load_q8(const float *row, int base, int V, float v[8]) {
    if (VEC && base + 8 <= V) {
        uint4 a = ld_stream_v4(row + base), b = ld_stream_v4(row + base + 4);
        v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
        v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
        v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
        v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
    } else {
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = (base + j < V) ? __ldg(row + base + j) : 0.f;
    }
}

__device__ __forceinline__ float max8(const float v[8]) {
    float a = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
    float b = fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7]));
    return fmaxf(a, b);
}

}  // namespace sv

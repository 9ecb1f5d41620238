// spec_verify.cu -- batched speculative-decoding verification for GB300 (sm_103a): the
// C-ABI entry points and the verify kernels.
//
// Fast path (16-byte aligned rows): two kernels per call.
//   stream kernel  SCTA persistent CTAs per SM claim work units (whole rows, then parts of the
//                  last wave of rows) from a counter in the workspace.  Warp 0 issues
//                  cp.async.bulk copies of each unit into a shared-memory ring (completion on
//                  mbarriers with transaction counts); warp 1 prepares the units (request
//                  lookup, sampling parameters, penalties of the earlier drafts, the row's draft
//                  gathers); the streamer warps reduce each 256-token segment to the statistics
//                  the row's filters need and write them to the workspace.
//   select kernel  one CTA per row, launched as a programmatic dependent of the stream kernel:
//                  the row's kept set, draws and draft probabilities; the last row of a request
//                  finalises it.
// Every mbarrier wait is bounded in time; on expiry the row fails with SV_DEV_TIMEOUT.
//
// Row kernel (any alignment).  One CTA per row streams it with plain 128-bit or scalar loads
// and then runs the same selection and finalisation code.
//
// Method: "Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust"
// ("The Memory Bandwidth Wall and Speculative Math", "The Verification Algorithm",
// "Orchestrating the Inference Loop"); "Adding Speculative Decoding" ("Verification and
// sampling", table "The existing base"); FreeToken PR #836 ("Design").
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "../../include/spec_verify.h"
#include "sv_select.cuh"
#include "sv_stream.cuh"

namespace sv {

// ------------------------------------------------------------------------------------------
// row kernel: one CTA per row, any alignment
// ------------------------------------------------------------------------------------------

// Bytes of one row's segment statistics: max, second/sum and lane arrays plus the histogram.
__host__ __device__ inline size_t segstats_bytes(int np) { return size_t(3) * np * 4 + 256 * 4; }

__device__ __forceinline__ SegStats carve_segstats(unsigned char *p, int np) {
    SegStats o;
    o.mx = reinterpret_cast<float *>(p);
    o.b = o.mx + np;
    o.lane = reinterpret_cast<int *>(o.b + np);
    o.hist = reinterpret_cast<uint32_t *>(o.lane + np);
    return o;
}

__host__ __device__ inline size_t rows_smem(int nseg) {
    const int np = nseg_pad(nseg);
    return segstats_bytes(np) + scratch_bytes(np);
}

template <typename E, bool VEC, bool QVEC>
__global__ void __launch_bounds__(RT, 4) verify_rows_kernel(const Args A) {
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ RowCtx S;
    const Grp<RT, 0> g(threadIdx.x);
    const int r = blockIdx.x;
    const int np = nseg_pad(A.nseg);
    const SegStats o = carve_segstats(dsm, np);
    const Scratch X = carve_scratch(dsm + segstats_bytes(np), np, dsm, rows_smem(A.nseg));
    SV_MARK(A, r, 0);
    if (g.warp() == 0) locate_row(A, S, r);
    g.sync();
    if (S.b < 0) return;   // a row outside every request: nothing to count
    fail_empty_requests(g, A, S);
    if (S.active) {
        const E *row = reinterpret_cast<const E *>(A.logits) + (size_t)r * A.V;
        if (g.warp() == 0) build_penalties(A, S, S.i);
        for (int d = g.t; d < 256; d += RT) o.hist[d] = 0;
        g.sync();
        SV_MARK(A, r, 1);
        // the last thread prefetches the row's draft gathers while the row streams
        int x = -1;
        E zraw = E(0);
        float qx = 0.f, u1 = 0.f;
        if (g.t == RT - 1 && !S.greedy) u1 = __ldg(A.uni + (size_t)r * 2 + 1);
        if (g.t == RT - 1 && S.i < S.k) {
            x = __ldg(A.tokens + S.d0 + S.i);
            if (x >= 0 && x < A.V) {
                zraw = __ldg(row + x);
                if (!S.greedy) qx = A.onehot ? 1.f : __ldg(A.q + (size_t)(S.d0 + S.i) * A.V + x);
            }
        }
        pass_stats<E, VEC>(g, S, row, A.V, A.nseg, o);
        if (g.t == RT - 1) {
            S.xtok = x;
            S.zx = elem_z_raw(S, zraw, x);
            S.qx = qx;
            S.u1 = u1;
        }
        g.sync();
        SV_MARK(A, r, 2);
        select_row<E, VEC>(g, A, S, X, o);
    }
    SV_MARK(A, r, 4);
    arrive_and_finalize<E, VEC, QVEC>(g, A, S, X);
    SV_MARK(A, r, 5);
}

// ------------------------------------------------------------------------------------------
// Two-kernel path (16-byte aligned rows).  Streaming and selection have opposite needs: the
// stream is bound by HBM bandwidth and wants every issue slot for its reductions; a row's
// selection is a short chain of dependent steps that wants many rows in flight.  So:
//   stream kernel  persistent CTAs stream every row once through a bulk-copy ring and write
//                  per-segment statistics (or, for greedy rows, a (max, position) key) to the
//                  workspace; the last wave of rows is split into parts so that the kernel
//                  does not end on a few CTAs streaming whole rows;
//   select kernel  one CTA per row turns the statistics into the row's kept set, draws and
//                  draft probabilities, and the request's last row finalises it.  It is
//                  launched as a programmatic dependent of the stream kernel: each CTA looks up
//                  its row, penalties and draft gathers while the stream finishes, then waits
//                  for the stream's results.
// ------------------------------------------------------------------------------------------

struct SShared {
    unsigned long long full[PNS_MAX];   // ring stage holds its chunk (transaction count)
    unsigned long long empty[PNS_MAX];  // every streamer warp released the stage
    unsigned long long rb_desc[NRB];    // unit buffer prepared by the scheduler
    unsigned long long rb_done[NRB];    // every streamer warp finished the unit
    int fail;
    RowCtx rc[NRB];
};

__host__ __device__ inline size_t up128(size_t x) { return (x + 127) & ~size_t(127); }
__host__ __device__ inline size_t mask_words(int np) { return (size_t)np / 32; }
// Dynamic shared memory of the stream kernel: the ring, then NRB masks of penalised segments.
__host__ __device__ inline size_t stream_smem(int nseg, int pns) {
    return (size_t)pns * SB + up128((size_t)NRB * mask_words(nseg_pad(nseg)) * 4);
}
// Dynamic shared memory of the select kernel: the row's statistics, then the scratch.
__host__ __device__ inline size_t select_smem(int nseg) {
    const int np = nseg_pad(nseg);
    return up128((size_t)3 * np * 4) + up128(scratch_bytes(np));
}

// Segment statistics (max, second value or weight sum, lane of the max) at base.
__device__ __forceinline__ SegStats stats_at(float *base, int np) {
    SegStats o;
    o.mx = base;
    o.b = base + np;
    o.lane = reinterpret_cast<int *>(base + 2 * np);
    o.hist = nullptr;
    return o;
}

// Chunk range of part p of a row with nc chunks split into P parts.
__device__ __forceinline__ void part_chunks(int nc, int P, int p, int &c0, int &c1) {
    c0 = (int)((long long)nc * p / P);
    c1 = (int)((long long)nc * (p + 1) / P);
}

// A stream CTA gave up on a bounded wait: record SV_DEV_TIMEOUT and raise the call's stream
// failure flag (header word 3), from which every select CTA marks its row KIND_FAIL -- rows
// this CTA had claimed were never reduced, so no request of the call can be trusted.
__device__ __forceinline__ void sfail(const Args &A, SShared &P, int b) {
    P.fail = 1;
    record_error(A, 7, b < 0 ? 0 : b);
    // every writer stores the same value; the select kernel reads it once the stream grid is done
    *reinterpret_cast<volatile int32_t *>(A.hdr + 3) = 1;
}

// The issuer's last act on a failure: waits (bounded) until every bulk copy it issued has
// landed, so that the CTA never exits while a copy still writes its shared memory.  The copy
// numbered j went to stage j mod pns in phase (j / pns) mod 2; only the last pns can be
// outstanding.
__device__ __noinline__ void drain_copies(unsigned long long *full, int q, int pns) {
    for (int t = 0; t < q && t < pns; t++) {
        const int j = q - 1 - t;
        mbar_wait(&full[j % pns], (uint32_t)(j / pns) & 1u);
    }
}

// Work unit u: row u while u < R - nsplit, then part (t mod nparts) of row R - nsplit + t / nparts
// with t = u - (R - nsplit).
// fp32 rows hold twice the registers per segment: two CTAs per SM instead of SCTA
template <typename E>
__host__ __device__ constexpr int stream_ctas() { return sizeof(E) == 2 ? SCTA : (SCTA < 2 ? SCTA : 2); }

template <typename E, bool HIST>
__global__ void __launch_bounds__(ST, stream_ctas<E>()) stream_kernel(const Args A) {
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ SShared P;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int V = A.V, nseg = A.nseg, np = nseg_pad(nseg), PNS = A.pns, NP = A.nparts;
    const uint32_t RB = (uint32_t)V * sizeof(E);
    const int nc = (int)((RB + SB - 1) / SB);
    unsigned char *ring = dsm;
    uint32_t *masks = reinterpret_cast<uint32_t *>(dsm + (size_t)PNS * SB);
    const long long whole = (long long)A.R - A.nsplit;
    const long long units = whole + (long long)A.nsplit * NP;

    // the select kernel's CTAs may be scheduled as soon as SMs free up
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < PNS; s++) {
            mbar_init(&P.full[s], 1);
            mbar_init(&P.empty[s], PSTREAM);
        }
        for (int s = 0; s < NRB; s++) {
            mbar_init(&P.rb_desc[s], 1);
            mbar_init(&P.rb_done[s], PSTREAM);
        }
        P.fail = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // the workspace words this kernel counts on were cleared by the kernel before it (this one
    // may start early, as its programmatic dependent): wait for them
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        // ---- issuer (one thread): bulk copies of each prepared unit, chunk by chunk
        if (lane != 0) return;
        const unsigned long long pol = l2_stream_policy();
        int q = 0;
        RingPos rp{0, 0u};
        for (int j = 0;; j++) {
            const int slot = j % NRB;
            if (!mbar_wait(&P.rb_desc[slot], (uint32_t)(j / NRB) & 1u)) {
                sfail(A, P, -1);
                drain_copies(P.full, q, PNS);
                return;
            }
            const RowCtx &R = P.rc[slot];
            if (R.r < 0) return;
            const unsigned char *src = reinterpret_cast<const unsigned char *>(A.logits) + (size_t)R.r * RB;
            for (int c = R.c0; c < R.c1; c++, q++) {
                const int st = rp.st;
                // the stage's previous fill (one lap earlier) must have been released
                if (q >= PNS && !mbar_wait(&P.empty[st], rp.ph ^ 1u)) {
                    sfail(A, P, R.b);
                    drain_copies(P.full, q, PNS);
                    return;
                }
                const uint32_t off = (uint32_t)c * SB;
                const uint32_t bytes = min((uint32_t)SB, RB - off);
                mbar_expect_tx(&P.full[st], bytes);
                bulk_g2s(ring + st * SB, src + off, bytes, &P.full[st], pol);
                rp.next(PNS);
            }
        }
    } else if (warp == 1) {
        // ---- scheduler (one warp): claim units and prepare them up to NRB ahead
        for (int j = 0;; j++) {
            const int slot = j % NRB;
            bool ok = true;
            if (j >= NRB) ok = mbar_wait(&P.rb_done[slot], (uint32_t)(j / NRB - 1) & 1u);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) sfail(A, P, -1);
                return;
            }
            RowCtx &R = P.rc[slot];
            int u = 0;
            if (lane == 0) u = atomicAdd(A.hdr + 2, 1);
            u = __shfl_sync(0xffffffffu, u, 0);
            if (u >= units) {
                if (lane == 0) {
                    R.r = -1;
                    mbar_arrive(&P.rb_desc[slot]);
                }
                return;
            }
#ifdef SV_TIMING
            if (lane == 0) {
                A.timing[(size_t)u * NTIME + 0] = global_ns();
                A.timing[(size_t)u * NTIME + 6] = (unsigned long long)blockIdx.x;
                A.timing[(size_t)u * NTIME + 10] = 0;
            }
#endif
            int r, part, npu;
            if (u < whole) {
                r = u;
                part = 0;
                npu = 1;
            } else {
                const int t = (int)(u - whole);
                r = (int)whole + t / NP;
                part = t - (t / NP) * NP;
                npu = NP;
            }
            locate_row(A, R, r);
            if (R.active) build_penalties(A, R, R.i);
            __syncwarp();
            if (R.active && (R.npen > 0 || R.hdir)) {
                // segments holding a penalised token take the streamers' slow path: those of
                // the request's history (indexed by the prepass), then the drafts'
                uint32_t *dmask = masks + slot * mask_words(np);
                const uint32_t *hm = R.hdir ? A.hmask + (size_t)R.b * mask_words(np) : nullptr;
                for (int w = lane; w < np / 32; w += 32) dmask[w] = hm ? __ldg(hm + w) : 0u;
                __syncwarp();
                for (int h = lane; h < R.npen; h += 32) {
                    const int x = R.pid[h];
                    if (x >= 0 && x < V) atomicOr(&dmask[(x / SEG) >> 5], 1u << ((x / SEG) & 31));
                }
            }
            __syncwarp();
            if (lane == 0) {
                R.part = part;
                R.nparts = npu;
                R.tix = u;
#ifdef SV_TIMING
                A.timing[(size_t)u * NTIME + 12] = (unsigned long long)r;
#endif
                int c0 = 0, c1 = 0;
                if (R.active) part_chunks(nc, npu, part, c0, c1);
                R.c0 = c0;
                R.c1 = c1;
                // (a test of the failure path withholds the first unit of CTA 0 from its copy
                // and reduction warps: their bounded waits run out, as a stalled scheduler's would)
                if (!(A.withhold && blockIdx.x == 0 && j == 0)) mbar_arrive(&P.rb_desc[slot]);
            }
            if (part == 0) {
                // the row's prepared context for the select kernel, with its draft gathers
                if (lane == 0) prefetch_draft<E>(A, R, reinterpret_cast<const E *>(A.logits) + (size_t)r * V);
                __syncwarp();
                const int4 *src = reinterpret_cast<const int4 *>(&R);
                int4 *dst = A.prep + (size_t)r * (PREP_BYTES / 16);
                for (int t = lane; t < PREP_BYTES / 16; t += 32) dst[t] = src[t];
            }
            __syncwarp();
        }
    } else {
        // ---- streamers: per-segment statistics of each unit from the ring into the workspace
        const int sw = warp - 2;
        RingPos rp{0, 0u};
        for (int j = 0;; j++) {
            const int slot = j % NRB;
            if (!__all_sync(0xffffffffu, mbar_wait(&P.rb_desc[slot], (uint32_t)(j / NRB) & 1u))) {
                if (lane == 0) sfail(A, P, -1);
                return;
            }
            const RowCtx &R = P.rc[slot];
            if (R.r < 0) return;
            const SegStats o = stats_at(A.gstats + (size_t)R.r * 3 * np, np);
            unsigned long long *tslot = nullptr;
#ifdef SV_TIMING
            tslot = A.timing + (size_t)R.tix * NTIME;
#endif
            if (!stream_row_any<E, HIST>(P.full, P.empty, ring, PNS, rp, R.c0, R.c1, nseg, V, sw, R, o,
                                   masks + slot * mask_words(np), A.rowarg + R.r, tslot)) {
                if (lane == 0) sfail(A, P, R.b);
                return;
            }
            __syncwarp();
#ifdef SV_TIMING
            if (lane == 0 && sw == 0) A.timing[(size_t)R.tix * NTIME + 2] = global_ns();
#endif
            if (lane == 0) mbar_arrive(&P.rb_done[slot]);
        }
    }
}

// One CTA per row: the row's kept set, draws and draft probabilities from the statistics the
// stream kernel wrote; the request's last row finalises the request.
template <typename E, bool QVEC>
__global__ void __launch_bounds__(SELT, SELT >= 128 ? 9 : 1152 / SELT) select_kernel(const Args A) {
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ RowCtx S;
    const Grp<SELT, 0> g(threadIdx.x);
    const int r = blockIdx.x;
    const int np = nseg_pad(A.nseg);
    float *sb = reinterpret_cast<float *>(dsm);
    const Scratch X = carve_scratch(dsm + up128((size_t)3 * np * 4), np, dsm, select_smem(A.nseg));
    SV_MARK(A, 4 * A.R + r, 0);
    // the stream kernel's results (and every earlier write on the stream) are visible past here
    asm volatile("griddepcontrol.wait;" ::: "memory");
    SV_MARK(A, 4 * A.R + r, 1);
    // the row's prepared context and segment statistics, in one round of loads
    {
        const int4 *src = A.prep + (size_t)r * (PREP_BYTES / 16);
        for (int t = g.t; t < PREP_BYTES / 16; t += SELT) reinterpret_cast<int4 *>(&S)[t] = __ldcg(src + t);
        const float4 *gs = reinterpret_cast<const float4 *>(A.gstats + (size_t)r * 3 * np);
        for (int t = g.t; t < 3 * np / 4; t += SELT) reinterpret_cast<float4 *>(sb)[t] = __ldcg(gs + t);
    }
    g.sync();
#ifdef SV_TIMING
    if (g.t == 0) S.tix = 4 * A.R + r;   // the select kernel's records follow the stream kernel's
    g.sync();
#endif
    SV_MARK(A, 4 * A.R + r, 2);
    if (S.b < 0) return;   // a row outside every request: nothing to count
    fail_empty_requests(g, A, S);
    if (S.active) {
        if (__ldcg(A.hdr + 3) == 0) {
            select_row<E, true>(g, A, S, X, stats_at(sb, np), A.rowarg + r);
        } else if (g.t == 0) {
            // a stream CTA gave up on a wait: this row's statistics cannot be trusted
            fail_row(A, S);
        }
    }
    SV_MARK(A, 4 * A.R + r, 4);
    arrive_and_finalize<E, true, QVEC>(g, A, S, X);
    SV_MARK(A, 4 * A.R + r, 5);
}

// History prepass (calls with a prior history), one CTA per request: checks the request's
// history (offsets inside [0, prior_len], ids in [0, V) strictly ascending, counts >= 1) and
// indexes it by segment -- hdir[s] = the first entry whose token lies in segment s or later,
// so segment s holds entries hdir[s] .. hdir[s+1] -- plus a bitmask of the segments that hold
// any.  A bad history sets the request's status and the sticky error word.
__global__ void __launch_bounds__(256) history_kernel(const Args A, int prior_len) {
    __shared__ int bad;
    const int b = blockIdx.x;
    const int np = nseg_pad(A.nseg);
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    const int lo = __ldg(A.hoff + b), hi = __ldg(A.hoff + b + 1);
    if (lo < 0 || hi < lo || hi > prior_len || (b == 0 && lo != 0)) {
        if (threadIdx.x == 0) bad = 1;
    } else {
        for (int j = lo + (int)threadIdx.x; j < hi; j += blockDim.x) {
            const int x = __ldg(A.htok + j);
            if (x < 0 || x >= A.V || __ldg(A.hcnt + j) < 1 || (j > lo && __ldg(A.htok + j - 1) >= x)) bad = 1;
        }
    }
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) {
            A.hstat[b] = 8;
            record_error(A, 8, b);
        }
        return;
    }
    int32_t *dir = A.hdir + (size_t)b * (np + 1);
    // entry j is the first of segments seg(x_{j-1}) + 1 .. seg(x_j); the end (j == hi) closes
    // the directory through segment np
    for (int j = lo + (int)threadIdx.x; j <= hi; j += blockDim.x) {
        const int s_lo = j == lo ? 0 : __ldg(A.htok + j - 1) / SEG + 1;
        const int s_hi = j == hi ? np : __ldg(A.htok + j) / SEG;
        for (int s = s_lo; s <= s_hi; s++) dir[s] = j;
    }
    __syncthreads();
    uint32_t *mask = A.hmask + (size_t)b * (np / 32);
    for (int w = threadIdx.x; w < np / 32; w += blockDim.x) {
        uint32_t bits = 0u;
        for (int t = 0; t < 32; t++)
            if (dir[w * 32 + t + 1] > dir[w * 32 + t]) bits |= 1u << t;
        mask[w] = bits;
    }
    if (threadIdx.x == 0) A.hstat[b] = 0;
}

__global__ void rollback_kernel(int32_t *kv, const int32_t *acc, const int32_t *nd, int B, int32_t *hdr) {
    int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    long long L = kv[b], k = nd[b], a = acc[b];
    long long t = L - (k + 1) + 1 + a;   // keep 1 + accepted of the k+1 appended rows
    if (k < 0 || a < 0 || a > k || t < 0 || t > L) {
        atomicCAS(hdr, 0, 1);
        atomicMax(hdr + 1, INT_MAX - b);
        return;
    }
    kv[b] = (int32_t)t;
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

// Devices a process may drive (a device index at or beyond it is SV_ERR_UNSUPPORTED).
constexpr int MAX_DEVICES = 64;

// Opts the kernel into `smem` bytes of dynamic shared memory where it needs more than the
// default 48 KB.  The opt-in belongs to the kernel in the current context, so it is looked up
// there on every call (no per-process cache): a call on another device, or on a context
// created again after a reset, opts in afresh.
template <typename K>
static cudaError_t ensure_smem(K kern, size_t smem) {
    if (smem <= 48 * 1024) return cudaSuccess;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if ((size_t)fa.maxDynamicSharedSizeBytes >= smem) return cudaSuccess;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// The current device, checked against MAX_DEVICES.
static cudaError_t current_device(int &dev) {
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return (dev < 0 || dev >= MAX_DEVICES) ? cudaErrorNotSupported : cudaSuccess;
}

// Clears n16 16-byte words at p (the workspace header, counters and argmax keys).  Lets its
// programmatic dependent (the stream kernel) start at once; that kernel waits before use.
__global__ void __launch_bounds__(256) clear_kernel(uint4 *p, size_t n16) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

template <typename E, bool VEC, bool QVEC>
static cudaError_t launch_rows(const Args &A, cudaStream_t stream) {
    const size_t smem = rows_smem(A.nseg);
    auto kern = verify_rows_kernel<E, VEC, QVEC>;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    kern<<<A.R, RT, smem, stream>>>(A);
    return cudaGetLastError();
}

// Events recorded around the stream kernel when set (sv_set_phase_events): process-wide, for
// every device and stream (a measurement aid for one caller at a time).  Recording them
// separates the two kernels, so the select kernel no longer overlaps the stream's end.
static std::atomic<cudaEvent_t> g_phase_start{nullptr}, g_phase_end{nullptr};

// Testing aid (sv_set_test_withhold): process-wide; while set, every stream kernel withholds
// one work unit so that its bounded waits run out.
static std::atomic<bool> g_withhold{false};

// Launches the stream kernel (SCTA CTAs per SM) and the select kernel as its programmatic
// dependent; returns cudaErrorNotSupported (nothing launched) when the kernels cannot be
// resident for this vocabulary.
template <typename E, bool QVEC>
static cudaError_t launch_two_kernels(const Args &A, cudaStream_t stream, int dev) {
    static std::atomic<int> sms[MAX_DEVICES];   // multiprocessors per device (0: not read yet)
    cudaError_t e;
    int nsm = sms[dev].load(std::memory_order_relaxed);
    if (!nsm) {
        if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        sms[dev].store(nsm, std::memory_order_relaxed);
    }
    Args B = A;
    const long long ctas = (long long)nsm * stream_ctas<E>();
    // the last wave of rows (one per CTA) is split into parts of at least 2 chunks
    const long long nc = ((long long)A.V * sizeof(E) + SB - 1) / SB;
    B.nparts = (int)(nc / 2 < SPLIT_PARTS ? nc / 2 : SPLIT_PARTS);
    if (B.nparts < 2 || A.R < 2) B.nparts = 1;
    B.nsplit = B.nparts > 1 ? (int)(ctas * SPLIT_WAVES < A.R ? ctas * SPLIT_WAVES : A.R) : 0;
    // shared memory of one stream CTA when SCTA share an SM (228 KB, 1 KB reserved per CTA)
    const size_t budget = (stream_ctas<E>() == 1 ? (size_t)232448 : (size_t)233472 / stream_ctas<E>() - 1024) - sizeof(SShared);
    B.pns = PNS_MAX;
    while (B.pns > 3 && stream_smem(A.nseg, B.pns) > budget) B.pns--;
    const size_t smem1 = stream_smem(A.nseg, B.pns), smem2 = select_smem(A.nseg);
    if (smem1 > budget || smem2 > (size_t)232448 - sizeof(RowCtx)) return cudaErrorNotSupported;
    // the stream kernel with the history variants only when the call passes a history
    const int hist = A.hoff ? 1 : 0;
    auto k1 = hist ? stream_kernel<E, true> : stream_kernel<E, false>;
    auto k2 = select_kernel<E, QVEC>;
    if ((e = ensure_smem(k1, smem1)) != cudaSuccess) return e;
    if ((e = ensure_smem(k2, smem2)) != cudaSuccess) return e;
    const long long units = (long long)A.R - B.nsplit + (long long)B.nsplit * B.nparts;
    const int grid = (int)(ctas < units ? ctas : units);
    const cudaEvent_t ph0 = g_phase_start.load(), ph1 = g_phase_end.load();
    if (ph0 && (e = cudaEventRecord(ph0, stream)) != cudaSuccess) return e;
    {
        // a programmatic dependent of the clearing kernel (or of the history prepass)
        cudaLaunchConfig_t cfg1 = {};
        cfg1.gridDim = dim3((unsigned)grid);
        cfg1.blockDim = dim3(ST);
        cfg1.dynamicSmemBytes = smem1;
        cfg1.stream = stream;
        cudaLaunchAttribute attr1[1];
        attr1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr1[0].val.programmaticStreamSerializationAllowed = 1;
        cfg1.attrs = attr1;
        cfg1.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg1, k1, B)) != cudaSuccess) return e;
    }
    if (ph1 && (e = cudaEventRecord(ph1, stream)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)A.R);
    cfg.blockDim = dim3(SELT);
    cfg.dynamicSmemBytes = smem2;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k2, B);
}

}  // namespace sv

using namespace sv;

extern "C" size_t sv_workspace_bytes(int32_t B, int32_t total_rows, int32_t V) {
    if (B < 1 || total_rows < B || V < 1) return 0;
    return ws_layout(B, total_rows, V).total;
}

extern "C" const char *sv_status_string(sv_status s) {
    switch (s) {
        case SV_OK: return "ok";
        case SV_ERR_INVALID_ARG: return "invalid argument";
        case SV_ERR_WORKSPACE: return "workspace too small or misaligned";
        case SV_ERR_CUDA: return "CUDA runtime error";
        case SV_ERR_UNSUPPORTED: return "unsupported shape";
        case SV_ERR_DEVICE_DATA: return "invalid device data";
    }
    return "unknown status";
}

// Both verification schemes: onehot == false is the accept test against q; onehot == true
// samples every row and keeps the drafts that equal the samples (draft_probs unused).
static sv_status verify_call(const void *target_logits, sv_dtype logits_dtype, const float *draft_probs,
                             const int32_t *draft_tokens, const int32_t *num_drafts, const int32_t *row_offsets,
                             int32_t B, int32_t k_max, int32_t V, int32_t total_rows, sv_params params,
                             const float *uniforms, int32_t *out_tokens, int32_t *accept_len, float *out_pq,
                             void *workspace, size_t workspace_bytes, void *stream, bool onehot) {
    if (onehot) draft_probs = nullptr;
    if (B < 1 || k_max < 0 || V < 1 || total_rows < B) return SV_ERR_INVALID_ARG;
    if (k_max > MAXK || V > MAXV) return SV_ERR_UNSUPPORTED;
    if (logits_dtype != SV_F32 && logits_dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (!row_offsets && (long long)total_rows != (long long)B * (k_max + 1)) return SV_ERR_INVALID_ARG;
    const int D = total_rows - B;
    if (!target_logits || !num_drafts || !uniforms || !out_tokens || !accept_len || !workspace) return SV_ERR_INVALID_ARG;
    if (D > 0 && ((!onehot && !draft_probs) || !draft_tokens)) return SV_ERR_INVALID_ARG;
    if (!params.temperature || !params.top_k || !params.top_p || !params.greedy) return SV_ERR_INVALID_ARG;
    if (params.prior_offsets && (!params.prior_tokens || !params.prior_counts || params.prior_len < 0))
        return SV_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(B, total_rows, V);
    if (((uintptr_t)workspace & 255) != 0 || workspace_bytes < L.total) return SV_ERR_WORKSPACE;

    char *ws = static_cast<char *>(workspace);
    Args A;
    A.logits = target_logits;
    A.q = draft_probs;
    A.tokens = draft_tokens;
    A.nd = num_drafts;
    A.row_off = row_offsets;
    A.T = params.temperature;
    A.topk = params.top_k;
    A.topp = params.top_p;
    A.pres = params.presence_penalty;
    A.freq = params.frequency_penalty;
    A.greedy = params.greedy;
    A.hoff = params.prior_offsets;
    A.htok = params.prior_tokens;
    A.hcnt = params.prior_counts;
    A.uni = uniforms;
    A.out_tok = out_tokens;
    A.acc = accept_len;
    A.out_pq = out_pq;
    A.hdr = reinterpret_cast<int32_t *>(ws);
    A.counters = reinterpret_cast<int32_t *>(ws + L.counters);
    A.rowarg = reinterpret_cast<unsigned long long *>(ws + L.rowarg);
    A.prep = reinterpret_cast<int4 *>(ws + L.prep);
    A.hdir = reinterpret_cast<int32_t *>(ws + L.hdir);
    A.hmask = reinterpret_cast<uint32_t *>(ws + L.hmask);
    A.hstat = reinterpret_cast<int32_t *>(ws + L.hstat);
    A.gstats = reinterpret_cast<float *>(ws + L.gstats);
    A.stats = reinterpret_cast<RowStat *>(ws + L.stats);
    A.pq = reinterpret_cast<float *>(ws + L.pq);
    A.timing = reinterpret_cast<unsigned long long *>(ws + L.timing);
    A.B = B;
    A.k_max = k_max;
    A.V = V;
    A.R = total_rows;
    A.nseg = nseg_of(V);
    A.pns = 0;
    A.nparts = 1;
    A.nsplit = 0;
    A.onehot = onehot ? 1 : 0;
    A.withhold = g_withhold.load() ? 1 : 0;
    const size_t esz = logits_dtype == SV_BF16 ? 2 : 4;
    const bool vec = ((uintptr_t)target_logits % 16 == 0) && ((size_t)V * esz) % 16 == 0;
    const bool qvec = (!draft_probs || (uintptr_t)draft_probs % 16 == 0) && ((size_t)V * 4) % 16 == 0;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (current_device(dev) != cudaSuccess) return SV_ERR_UNSUPPORTED;
    // clear the error word, the work claim counter, the per-request arrival counters, the
    // per-row part counters and the greedy rows' argmax keys
    {
        // (the clear ends below the statistics region, which starts at a 256-byte boundary)
        const size_t n16 = (L.rowarg + (size_t)total_rows * 8 + 15) / 16;
        const unsigned blocks = (unsigned)((n16 + 255) / 256 < 304 ? (n16 + 255) / 256 : 304);
        clear_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<uint4 *>(ws), n16);
        if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    }
    if (A.hoff) {
        history_kernel<<<B, 256, 0, st>>>(A, params.prior_len);
        if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    }
    cudaError_t e = cudaErrorNotSupported;
    if (vec) {
        if (logits_dtype == SV_BF16)
            e = qvec ? launch_two_kernels<uint16_t, true>(A, st, dev) : launch_two_kernels<uint16_t, false>(A, st, dev);
        else
            e = qvec ? launch_two_kernels<float, true>(A, st, dev) : launch_two_kernels<float, false>(A, st, dev);
    }
    if (e == cudaErrorNotSupported) {
        cudaGetLastError();   // clear a sticky "not supported" from the probe, if any
        if (logits_dtype == SV_BF16) {
            if (vec) e = qvec ? launch_rows<uint16_t, true, true>(A, st) : launch_rows<uint16_t, true, false>(A, st);
            else e = qvec ? launch_rows<uint16_t, false, true>(A, st) : launch_rows<uint16_t, false, false>(A, st);
        } else {
            if (vec) e = qvec ? launch_rows<float, true, true>(A, st) : launch_rows<float, true, false>(A, st);
            else e = qvec ? launch_rows<float, false, true>(A, st) : launch_rows<float, false, false>(A, st);
        }
    }
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status spec_verify(const void *target_logits, sv_dtype logits_dtype, const float *draft_probs,
                                 const int32_t *draft_tokens, const int32_t *num_drafts, const int32_t *row_offsets,
                                 int32_t B, int32_t k_max, int32_t V, int32_t total_rows, sv_params params,
                                 const float *uniforms, int32_t *out_tokens, int32_t *accept_len, float *out_pq,
                                 void *workspace, size_t workspace_bytes, void *stream) {
    return verify_call(target_logits, logits_dtype, draft_probs, draft_tokens, num_drafts, row_offsets, B, k_max, V,
                       total_rows, params, uniforms, out_tokens, accept_len, out_pq, workspace, workspace_bytes,
                       stream, false);
}

extern "C" sv_status spec_verify_onehot(const void *target_logits, sv_dtype logits_dtype, const int32_t *draft_tokens,
                                        const int32_t *num_drafts, const int32_t *row_offsets, int32_t B,
                                        int32_t k_max, int32_t V, int32_t total_rows, sv_params params,
                                        const float *uniforms, int32_t *out_tokens, int32_t *accept_len,
                                        float *out_pq, void *workspace, size_t workspace_bytes, void *stream) {
    return verify_call(target_logits, logits_dtype, nullptr, draft_tokens, num_drafts, row_offsets, B, k_max, V,
                       total_rows, params, uniforms, out_tokens, accept_len, out_pq, workspace, workspace_bytes,
                       stream, true);
}

extern "C" sv_status spec_rollback(int32_t *kv_seq_len, const int32_t *accept_len, const int32_t *num_drafts,
                                   int32_t B, void *workspace, void *stream) {
    if (B < 1 || !kv_seq_len || !accept_len || !num_drafts || !workspace) return SV_ERR_INVALID_ARG;
    if (((uintptr_t)workspace & 255) != 0) return SV_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int threads = 256;
    rollback_kernel<<<(B + threads - 1) / threads, threads, 0, st>>>(kv_seq_len, accept_len, num_drafts, B,
                                                                     reinterpret_cast<int32_t *>(workspace));
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status sv_read_device_error(const void *workspace, int32_t *code, int32_t *first_bad_request) {
    if (!workspace) return SV_ERR_INVALID_ARG;
    int32_t h[2] = {0, 0};
    if (cudaMemcpy(h, workspace, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return SV_ERR_CUDA;
    if (code) *code = h[0];
    if (first_bad_request) *first_bad_request = h[1] ? INT_MAX - h[1] : -1;
    return h[0] ? SV_ERR_DEVICE_DATA : SV_OK;
}

// ------------------------------------------------------------------------------------------
// spec_verify_static: spec_verify on a workspace the library owns (a file-scope device array),
// for callers that cannot hand the library device memory.  Nothing is allocated: the array is
// part of the loaded module.  Every call shares it, so calls must not overlap in time.
// ------------------------------------------------------------------------------------------

static __device__ __align__(256) unsigned char sv_static_workspace[SV_STATIC_WORKSPACE_BYTES];

extern "C" sv_status spec_verify_static(const void *target_logits, sv_dtype logits_dtype, const float *draft_probs,
                                        const int32_t *draft_tokens, const int32_t *num_drafts,
                                        const int32_t *row_offsets, int32_t B, int32_t k_max, int32_t V,
                                        int32_t total_rows, sv_params params, const float *uniforms,
                                        int32_t *out_tokens, int32_t *accept_len, float *out_pq, void *stream) {
    // the array's address on each device, looked up once with that device current (host
    // threads that race on the first lookup store the same address)
    static std::atomic<void *> base[MAX_DEVICES];
    if (B < 1 || k_max < 0 || V < 1 || total_rows < B) return SV_ERR_INVALID_ARG;
    const size_t need = sv_workspace_bytes(B, total_rows, V);
    if (need == 0) return SV_ERR_INVALID_ARG;
    if (need > (size_t)SV_STATIC_WORKSPACE_BYTES) return SV_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES) return SV_ERR_UNSUPPORTED;
    void *ws = base[dev].load(std::memory_order_acquire);
    if (!ws) {
        if (cudaGetSymbolAddress(&ws, sv_static_workspace) != cudaSuccess || !ws) return SV_ERR_CUDA;
        base[dev].store(ws, std::memory_order_release);
    }
    // spec_verify clears what must start at zero (error word, claim and arrival counters,
    // greedy argmax keys) on `stream` before its kernels run
    return spec_verify(target_logits, logits_dtype, draft_probs, draft_tokens, num_drafts, row_offsets, B, k_max, V,
                       total_rows, params, uniforms, out_tokens, accept_len, out_pq, ws,
                       (size_t)SV_STATIC_WORKSPACE_BYTES, stream);
}

extern "C" sv_status sv_set_test_withhold(int32_t on) {
    g_withhold.store(on != 0);
    return SV_OK;
}

extern "C" sv_status sv_set_phase_events(void *stream_kernel_start, void *stream_kernel_end) {
    if ((stream_kernel_start == nullptr) != (stream_kernel_end == nullptr)) return SV_ERR_INVALID_ARG;
    g_phase_start.store(static_cast<cudaEvent_t>(stream_kernel_start));
    g_phase_end.store(static_cast<cudaEvent_t>(stream_kernel_end));
    return SV_OK;
}

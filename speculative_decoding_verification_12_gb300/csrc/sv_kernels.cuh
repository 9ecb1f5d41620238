// sv_kernels.cuh -- the verify kernels (row kernel; stream, select and residual kernels) and
// their launch sequences.  Included by the per-dtype translation units (verify_*.cu), each of
// which instantiates one dtype and one scheme, so that they compile in parallel.
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
// Every mbarrier wait is bounded in time; on expiry the call's requests fail with SV_DEV_TIMEOUT.
//
// Row kernel (any alignment).  One CTA per row streams it with plain 128-bit or scalar loads
// and then runs the same selection and finalisation code.
//
// Lazy scheme: the two kernels over each request's row 0, again over the rows of the requests
// that kept draft 0, then a residual kernel for the whole-row residual draws.
//
// Method: "Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust"
// ("The Memory Bandwidth Wall and Speculative Math", "The Verification Algorithm",
// "Orchestrating the Inference Loop"); "Adding Speculative Decoding" ("Verification and
// sampling", table "The existing base"); FreeToken PR #836 ("Design").
#pragma once

#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "sv_launch.h"
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

// First row of request b, or -1 when the request owns no rows or its offsets leave [0, R).
__device__ __forceinline__ int first_row(const Args &A, int b) {
    if (!A.row_off) return b * (A.k_max + 1);
    const int r0 = __ldg(A.row_off + b), r1 = __ldg(A.row_off + b + 1);
    return (r0 >= 0 && r1 > r0 && r1 <= A.R) ? r0 : -1;
}

// Row li of the rows a launch works on: every row (phase 0), each request's first row (phase 1,
// -1 for a request without rows), or the rows queued by the lazy scheme's first phase (phase 2).
__device__ __forceinline__ int listed_row(const Args &A, int li) {
    if (A.phase == 0) return li;
    if (A.phase == 1) return first_row(A, li);
    return __ldcg(A.listb + li);
}

// A stream CTA gave up on a bounded wait: record SV_DEV_TIMEOUT and raise the call's stream
// failure flag (header word 3).  Rows this CTA had claimed were never reduced: with whole-grid
// selection every select CTA then fails its row's request, with per-row selection those whose
// row never became ready do.
__device__ __forceinline__ void sfail(const Args &A, SShared &P, int b) {
    P.fail = 1;
    record_error(A, 7, b < 0 ? 0 : b);
    // every writer stores the same value
    *reinterpret_cast<volatile int32_t *>(A.hdr + 3) = 1;
}

// The issuer's last act on a failure: waits (bounded) until every bulk copy it issued has
// landed, so that the CTA never exits while a copy still writes its shared memory.  The copy
// numbered j went to stage j mod pns in phase (j / pns) mod 2; only the last pns can be
// outstanding.
static __device__ __noinline__ void drain_copies(unsigned long long *full, int q, int pns) {
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
// One-pass calls: finalisers queue their whole-row residual draws, and A.nworkers worker CTAs
// that follow the row CTAs in the select grid take them slice by slice, instead of the
// finalising CTA drawing them alone.
#ifndef SV_RESIDQ
#define SV_RESIDQ 1
#endif
constexpr bool RESIDQ = SV_RESIDQ != 0;

// How the stream and select kernels of a call work together; each has an instance per scheme,
// which holds none of the others' code.
enum : int {
    SCH_GRID = 0,   // one-pass call: every row selected once the whole stream grid is done
    SCH_ROWS = 1,   // one-pass call: rows streamed in the order the clearing kernel built, each
                    // selected as soon as its own units are streamed (per-row ready words)
    SCH_LAZY = 2    // the lazy scheme's launches (phases 1 and 2)
};

template <typename E, bool HIST, int SCH>
__global__ void __launch_bounds__(stream_threads<E>(), stream_ctas<E>()) stream_kernel(const Args A) {
    constexpr bool LAZY = SCH == SCH_LAZY, PERROW = SCH == SCH_ROWS;
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ SShared P;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int V = A.V, nseg = A.nseg, np = nseg_pad(nseg), PNS = A.pns, NP = A.nparts;
    const uint32_t RB = (uint32_t)V * sizeof(E);
    const int nc = (int)((RB + SB - 1) / SB);
    unsigned char *ring = dsm;
    uint32_t *masks = reinterpret_cast<uint32_t *>(dsm + (size_t)PNS * SB);

    // the select kernel's CTAs may be scheduled as soon as SMs free up
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#ifdef SV_TIMING
    if (threadIdx.x == 0) atomicMin(A.timing + (size_t)5 * A.R * NTIME + 6, global_ns());
#endif
    if (threadIdx.x == 0) {
        for (int s = 0; s < PNS; s++) {
            mbar_init(&P.full[s], 1);
            mbar_init(&P.empty[s], pstream<E>());
        }
        for (int s = 0; s < NRB; s++) {
            mbar_init(&P.rb_desc[s], 1);
            mbar_init(&P.rb_done[s], pstream<E>());
        }
        P.fail = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // the workspace words this kernel counts on were cleared by the kernel before it (this one
    // may start early, as its programmatic dependent): wait for them
    asm volatile("griddepcontrol.wait;" ::: "memory");
#ifdef SV_TIMING
    if (threadIdx.x == 0) atomicMin(A.timing + (size_t)5 * A.R * NTIME + 2, global_ns());
#endif

    if (warp == 0) {
        // ---- issuer (one thread): bulk copies of each prepared unit, chunk by chunk
        // (R.r < 0 ends the CTA's work; an unused unit has no chunks)
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
        // ---- scheduler (one warp): claim units and prepare them up to NRB ahead.  The rows
        // this launch streams (listed_row): every row, each request's first row, or the rows
        // the first phase of the lazy scheme queued (counted once the wait above is over).
        int rows = A.R, nsplit = A.nsplit;
        bool ident = true;   // per-row selection: stream in the order the clearing kernel built
        if constexpr (LAZY) {
            rows = A.phase == 1 ? A.B : __ldcg(A.hdr + 4);
            nsplit = NP > 1 ? min(rows, A.ctas * SPLIT_WAVES) : 0;
        } else if constexpr (PERROW) {
            ident = (__ldcg(A.ordflag) & 1ull) != 0;
        }
        const long long whole = (long long)rows - nsplit;
        const long long units = whole + (long long)nsplit * NP;
        for (int j = 0;; j++) {
            const int slot = j % NRB;
            bool ok = true;
            if (j >= NRB) ok = mbar_wait(&P.rb_done[slot], (uint32_t)(j / NRB - 1) & 1u);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) sfail(A, P, -1);
                return;
            }
            RowCtx &R = P.rc[slot];
            // The unit this slot held is streamed (the streamer warps' arrivals release their
            // writes to this warp): publish it as one share of its row.  The scheduler, not each
            // streamer warp, pays the fence, and it waits on exactly this unit anyway.
            if (PERROW && j >= NRB && lane == 0) row_share_done(A, R.r, R.nparts);
            // With whole-grid selection each CTA's first unit is unit blockIdx.x and the counter
            // hands out the rest (one contended atomic fewer before the first copies); the lazy
            // scheme's second phase claims from a counter of its own.
            constexpr bool FIXED_FIRST = SCH == SCH_GRID;
            int u = 0;
            if (FIXED_FIRST && j == 0) u = (int)blockIdx.x;
            else if (lane == 0) u = (FIXED_FIRST ? (int)gridDim.x : 0) + atomicAdd(A.hdr + (LAZY && A.phase == 2 ? 6 : 2), 1);
            u = __shfl_sync(0xffffffffu, u, 0);
            if (u >= units) {
                if (lane == 0) {
                    R.r = -1;
                    mbar_arrive(&P.rb_desc[slot]);
                }
                if constexpr (PERROW) {
                    // the units still in flight, oldest first, published as they finish
                    for (int jj = j - NRB + 1 < 0 ? 0 : j - NRB + 1; jj < j; jj++) {
                        const int sl = jj % NRB;
                        if (!__all_sync(0xffffffffu, mbar_wait(&P.rb_done[sl], (uint32_t)(jj / NRB) & 1u))) {
                            if (lane == 0) sfail(A, P, -1);
                            return;
                        }
                        if (lane == 0) row_share_done(A, P.rc[sl].r, P.rc[sl].nparts);
                    }
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
            int li, part, npu;
            if (u < whole) {
                li = u;
                part = 0;
                npu = 1;
            } else {
                const int t = (int)(u - whole);
                li = (int)whole + t / NP;
                part = t - (t / NP) * NP;
                npu = NP;
            }
            const int r = LAZY ? listed_row(A, li) : (PERROW && !ident ? order_row(A, li) : li);
            if (!LAZY || r >= 0) {
                locate_row(A, R, r);
                if (R.active) build_penalties(A, R, R.i);
                // a sampled row whose kept set is not built as a candidate list may end in a
                // whole-row residual draw: counted once per row for the select grid's workers
                if (!LAZY && RESIDQ && part == 0 && lane == 0 && R.active && !R.greedy && !A.onehot && R.mode != MODE_TOP2)
                    atomicAdd(A.hdr + 9, 1);
            } else if (lane == 0) {
                R.active = 0;   // a first row the request does not have: nothing to stream
            }
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
                if (LAZY && r < 0) R.r = 0;   // (any row index: the unit has no chunks and no statistics)
                // (a test of the failure path withholds the first unit of CTA 0 from its copy
                // and reduction warps: their bounded waits run out, as a stalled scheduler's would)
                if (!(A.withhold && blockIdx.x == 0 && j == 0)) mbar_arrive(&P.rb_desc[slot]);
            }
            if (part == 0 && (!LAZY || r >= 0)) {
                // the row's prepared context for the select kernel, with its draft gathers
                if (lane == 0) prefetch_draft<E>(A, R, reinterpret_cast<const E *>(A.logits) + (size_t)r * V);
                __syncwarp();
                const int4 *src = reinterpret_cast<const int4 *>(&R);
                int4 *dst = A.prep + (size_t)r * (PREP_BYTES / 16);
                for (int t = lane; t < PREP_BYTES / 16; t += 32) dst[t] = src[t];
                // (published with the unit's completion, by this warp: its lanes' writes are
                // ordered before that by the warp barriers in between)
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

// A row the select kernel cannot trust (it was not streamed in full): its request's outputs
// become -1, its draft's (p, q) NaN, and SV_DEV_TIMEOUT is recorded.  The request is not
// finalised, since this row never arrives.  One warp.
__device__ __forceinline__ void fail_unstreamed_row(const Args &A, int r) {
    const int lane = lane_id();
    const int b = A.row_off ? find_request(A.row_off, A.B, r) : r / (A.k_max + 1);
    if (b < 0 || b >= A.B) {
        if (lane == 0) record_error(A, 7, 0);
        return;
    }
    const int r0 = A.row_off ? __ldg(A.row_off + b) : b * (A.k_max + 1);
    const int kw = A.k_max + 1;
    for (int j = lane; j < kw; j += 32) A.out_tok[(size_t)b * kw + j] = -1;
    if (lane == 0) {
        A.acc[b] = -1;
        record_error(A, 7, b);
        const int i = r - r0, k = min(__ldg(A.nd + b), A.k_max);
        if (i >= 0 && i < k) {
            const size_t d = (size_t)(r0 - b + i);
            A.pq[d * 2] = NAN;
            A.pq[d * 2 + 1] = NAN;
            if (A.out_pq) {
                A.out_pq[d * 2] = NAN;
                A.out_pq[d * 2 + 1] = NAN;
            }
        }
    }
}

// Whole-row residual draws that finalisers queued ("Speculative Decoding in Custom LLM
// Servicing: Implementing Draft Models in Rust", "The Memory Bandwidth Wall and Speculative
// Math": the residual max(0, p - q), normalised; an empty residual draws from p).  A job is
// split into RSL slices of the rejected row; a slice is the per-segment sums of max(0, p - q)
// and of p over its segments, read with many loads in flight, and the job's last slice to
// finish draws the final token from every slice's sums.
#ifndef SV_RSL
#define SV_RSL 8
#endif
constexpr int RSL = SV_RSL;   // slices per residual job
constexpr int RST = 256;   // threads per residual kernel CTA

// Slice p of job j, by the whole group; S (the row context) and rsm (2 np floats) are the
// group's shared scratch, `last` a shared word.
template <typename E, bool QVEC, int U, class G>
__device__ void resid_slice(const G &g, const Args &A, RowCtx &S, float *rsm, int *last, int j, int p) {
    const unsigned long long w = __ldcg(A.jobs + j);
    const int b = (int)((w >> 7) & 0x1FFFFFFu), a = (int)(w & 127u);
    const int V = A.V, nseg = A.nseg, np = nseg_pad(nseg);
    const int lane = g.lane();
    const int r = first_row(A, b) + a;   // (a job comes from a finalised request, so b owns rows)
    g.sync();   // (S and rsm of the group's previous slice are no longer read)
    if (g.warp() == 0) {
        locate_row(A, S, r);
        build_penalties(A, S, a);
    }
    g.sync();
    const RowStat st = load_stat(A.stats + r);
    const E *row = reinterpret_cast<const E *>(A.logits) + (size_t)r * V;
    const float *qrow = A.q + (size_t)(S.d0 + a) * V;
    const WResid wr{st.m, st.s, st.invZ, st.taukey};
    const WProb wp{st.m, st.s, st.invZ, st.taukey};
    float *sumr = A.jobsum + (size_t)j * 2 * np, *sump = sumr + np;
    const int s_lo = (int)((long long)nseg * p / RSL), s_hi = (int)((long long)nseg * (p + 1) / RSL);
    pass_segment_range<E, true, QVEC, true, U>(
        g, S, row, qrow, V, s_lo, s_hi, [&](int seg, const float *v, const float *qv) {
            float x = 0.f, y = 0.f;
#pragma unroll
            for (int t = 0; t < 8; t++) {
                if (seg * SEG + lane * 8 + t < V) {
                    x += wr(v[t], qv[t]);
                    y += wp(v[t], qv[t]);
                }
            }
            x = warp_sum(x);
            y = warp_sum(y);
            if (lane == 0) {
                sumr[seg] = x;
                sump[seg] = y;
            }
        });
    g.sync();
    if (g.t == 0) {
        __threadfence();
        *last = atomicAdd(A.jobcnt + j, 1) == RSL - 1;
    }
    g.sync();
    if (!*last) return;
    __threadfence();
    for (int t = g.t; t < nseg; t += G::kThreads) {
        rsm[t] = __ldcg(sumr + t);
        rsm[np + t] = __ldcg(sump + t);
    }
    g.sync();
    const float u = __ldg(A.uni + (size_t)r * 2 + 1);
    int tok = draw_by_segments<E, true, QVEC>(g, S, row, qrow, V, nseg, rsm, u, wr);
    if (tok < 0) tok = draw_by_segments<E, true, QVEC>(g, S, row, nullptr, V, nseg, rsm + np, u, wp);
    if (g.t == 0) A.out_tok[(size_t)b * (A.k_max + 1) + a] = tok;
}

#ifndef SV_WORKERS_PER_SM
#define SV_WORKERS_PER_SM 8
#endif
#ifndef SV_WORKER_U
#define SV_WORKER_U 1
#endif
constexpr int WORKERS_PER_SM = SV_WORKERS_PER_SM;
static_assert(WORKERS_PER_SM < SEL_PER_SM, "residual workers leave every SM a slot for row CTAs");

// A worker CTA of the one-pass select grid: claims residual slices in turn, waits (bounded) for
// the claimed slice's job to be queued, and leaves once every row CTA is done and no slice is
// left.  Worker CTAs come after every row CTA in the grid and are fewer than the select CTAs an
// SM holds, so they never keep a row CTA from its slot.
template <typename E, bool QVEC>
__device__ void resid_worker(const Grp<SELT, 0> &g, const Args &A, unsigned char *dsm, RowCtx &S) {
    __shared__ int s_sl, s_go, last;
    float *rsm = reinterpret_cast<float *>(dsm);
    const uint32_t *njobs = reinterpret_cast<const uint32_t *>(A.hdr + 5);
    const uint32_t *rowsdone = reinterpret_cast<const uint32_t *>(A.hdr + 7);
    // the header counters were cleared before the stream kernel ran, which is done past here
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // With no row that builds its kept set otherwise than as a candidate list, a job can only
    // come from a candidate overflow: the first worker stays for that, the others leave.
    if ((int)blockIdx.x != A.R && __ldcg(A.hdr + 9) == 0) return;
    for (;;) {
        if (g.t == 0) {
            const int sl = atomicAdd(A.hdr + 8, 1);
            int go = 0;
            const unsigned long long t0 = global_ns();
            unsigned ns = 64;
            for (;;) {
                // (volatile polls; the acquiring loads only once a condition holds)
                if (sl < (int)*reinterpret_cast<const volatile uint32_t *>(njobs) * RSL) {
                    go = 1;
                    break;
                }
                if ((int)*reinterpret_cast<const volatile uint32_t *>(rowsdone) >= A.R) {
                    go = (int)ld_acquire_u32(rowsdone) >= A.R && sl < (int)ld_acquire_u32(njobs) * RSL;
                    break;
                }
                if (global_ns() - t0 > WAIT_NS) {
                    record_error(A, 7, 0);
                    break;
                }
                __nanosleep(ns);
                ns = ns < 256 ? ns * 2 : 256;
            }
            if (go) {
                // the job's record follows the reservation of its slot
                unsigned long long w = 0;
                go = wait_word(A.jobs + sl / RSL, ld_acquire_u64,
                               [&](unsigned long long v) { return (uint32_t)(v >> 32) == A.epoch; }, &w);
                if (!go) record_error(A, 7, 0);
            }
            s_sl = sl;
            s_go = go;
        }
        g.sync();
        if (!s_go) return;
#ifdef SV_TIMING
        if (g.t == 0) atomicMin(A.timing + (size_t)5 * A.R * NTIME + 8, global_ns());
#endif
        resid_slice<E, QVEC, SV_WORKER_U>(g, A, S, rsm, &last, s_sl / RSL, s_sl % RSL);
#ifdef SV_TIMING
        if (g.t == 0) {
            atomicMax(A.timing + (size_t)5 * A.R * NTIME + 9, global_ns());
            atomicAdd(A.timing + (size_t)5 * A.R * NTIME + 10, 1ull);
        }
#endif
    }
}

// One CTA per row: the row's kept set, draws and draft probabilities from the statistics the
// stream kernel wrote; the request's last row finalises the request.
template <typename E, bool QVEC, int SCH>
__device__ __forceinline__ void select_row_cta(const Grp<SELT, 0> &g, const Args &A, unsigned char *dsm, RowCtx &S) {
    constexpr bool LAZY = SCH == SCH_LAZY, PERROW = SCH == SCH_ROWS;
    const int np = nseg_pad(A.nseg);
    float *sb = reinterpret_cast<float *>(dsm);
    const Scratch X = carve_scratch(dsm + up128((size_t)3 * np * 4), np, dsm, select_smem(A.nseg));
    // this CTA's row: the row at its streaming position (one-pass call), each request's first
    // row, or a row the first phase of the lazy scheme queued
    int r = blockIdx.x;
    bool ready = true;
#ifdef SV_TIMING
    const unsigned long long tent = global_ns();
#endif
    if constexpr (PERROW) {
        // Not a wait for the whole stream grid: the order, then this row alone.  The row is
        // selected as soon as every unit of it is streamed, while later rows still stream.  Both
        // waits are bounded, and the second ends early once a stream CTA has given up.
        __shared__ int s_r, s_ok;
        if (g.warp() == 0) {
            unsigned long long of = 0;
            int ok = 1;
            const unsigned long long tag = ((unsigned long long)A.key << 32) | (2ull * A.epoch);
            if (g.lane() == 0)
                ok = wait_word(A.ordflag, ld_acquire_u64, [&](unsigned long long v) { return (v & ~1ull) == tag; }, &of);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            of = __shfl_sync(0xffffffffu, of, 0);
            const int rr = (ok && !(of & 1ull)) ? order_row(A, (int)blockIdx.x) : (int)blockIdx.x;
            if (g.lane() == 0) {
                uint32_t v = 0;
                if (ok) {
                    wait_word(A.ready + rr, ld_acquire_u32,
                              [&](uint32_t x) { return x == A.epoch || *(volatile const int32_t *)(A.hdr + 3) != 0; }, &v);
                }
                s_ok = ok && v == A.epoch;
                s_r = rr;
            }
        }
        g.sync();
        r = s_r;
        ready = s_ok != 0;
    } else {
        // a later launch of the lazy scheme may be scheduled as soon as SMs free up
        if constexpr (LAZY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // the stream kernel's results (and every earlier write on the stream) are visible past here
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if constexpr (LAZY) {
            if (A.phase == 1) {
                r = first_row(A, blockIdx.x);
                if (r < 0) {   // a request that owns no rows
                    fail_request(g, A, blockIdx.x);
                    return;
                }
            } else {
                if ((int)blockIdx.x >= __ldcg(A.hdr + 4)) return;
                r = __ldcg(A.listb + blockIdx.x);
            }
        }
        // a stream CTA gave up on a wait: no row of this launch can be trusted
        ready = __ldcg(A.hdr + 3) == 0;
    }
    SV_MARK(A, 4 * A.R + r, 1);
#ifdef SV_TIMING
    if (g.t == 0) {
        A.timing[(size_t)(4 * A.R + r) * NTIME + 0] = tent;
        atomicMin(A.timing + (size_t)5 * A.R * NTIME + 3, tent);
    }
#endif
    // The CTA of the last position joins the stream grid before it ends, so that this grid
    // (and whatever the stream runs after it) completes after the stream kernel.  That row is
    // streamed last: the join costs the stream kernel's exit, not a wait for the whole stream.
    const bool join = PERROW && (int)blockIdx.x == A.R - 1;
    if (!ready) {
        // The row was not (or not surely) streamed: a stream CTA gave up on a wait.  Its request
        // gets -1 outputs and SV_DEV_TIMEOUT, and is never finalised (this row does not arrive).
        if (g.warp() == 0) fail_unstreamed_row(A, r);
        if (join) asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
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
    if (join) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (S.b < 0) return;   // a row outside every request: nothing to count
    if (!LAZY) fail_empty_requests(g, A, S);
    if (S.active) select_row<E, true>(g, A, S, X, stats_at(sb, np), A.rowarg + r);
    SV_MARK(A, 4 * A.R + r, 4);
    if (LAZY && A.phase == 1) first_row_decision<E, true, QVEC>(g, A, S, X);
    else arrive_and_finalize<E, true, QVEC, LAZY, LAZY || RESIDQ>(g, A, S, X);
    SV_MARK(A, 4 * A.R + r, 5);
}

template <typename E, bool QVEC, int SCH>
__global__ void __launch_bounds__(SELT, SEL_PER_SM) select_kernel(const Args A) {
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ RowCtx S;
    const Grp<SELT, 0> g(threadIdx.x);
    // The next launch on the stream may be scheduled now: the next call's clearing kernel
    // waits for this grid to complete (as any programmatic dependent must before it reads
    // this call's results), so its launch overlaps this kernel's tail.
    if constexpr (SCH != SCH_LAZY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if constexpr (SCH != SCH_LAZY && RESIDQ) {
        if ((int)blockIdx.x >= A.R) {
            resid_worker<E, QVEC>(g, A, dsm, S);
            return;
        }
    }
    select_row_cta<E, QVEC, SCH>(g, A, dsm, S);
    if constexpr (SCH != SCH_LAZY && RESIDQ) {
        // this row CTA is done; a CTA that queued a residual job releases its reservation with
        // the count (the only ordering the workers rely on: the job's record is released on its
        // own), the others count without a fence
        g.sync();
        if (g.t == 0) {
            if (S.last && S.need_resid) {
                int old;
                asm volatile("atom.release.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(A.hdr + 7) : "memory");
            } else {
                atomicAdd(A.hdr + 7, 1);
            }
        }
    }
}

// Lazy scheme, last launch: every slice of every queued job, taken in turn by the grid's CTAs.
template <typename E, bool QVEC>
__global__ void __launch_bounds__(RST) resid_kernel(const Args A) {
    extern __shared__ __align__(16) float rsm[];   // the job's residual sums, then p sums (np each)
    __shared__ RowCtx S;
    __shared__ int last;
    const Grp<RST, 0> g(threadIdx.x);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int nslices = __ldcg(A.hdr + 5) * RSL;
    for (int sl = blockIdx.x; sl < nslices; sl += gridDim.x)
        resid_slice<E, QVEC, sizeof(E) == 2 ? 2 : 1>(g, A, S, rsm, &last, sl / RSL, sl % RSL);
}

// CTAs of a residual launch: one per slice of every job a call can queue (the kernel's loop
// covers any grid).
static unsigned resid_grid(const Args &A) { return (unsigned)((long long)A.B * RSL); }

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
template <typename E, bool VEC, bool QVEC>
static cudaError_t launch_rows(const Args &A, cudaStream_t stream) {
    const size_t smem = rows_smem(A.nseg);
    auto kern = verify_rows_kernel<E, VEC, QVEC>;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    kern<<<A.R, RT, smem, stream>>>(A);
    return cudaGetLastError();
}
// One launch on `stream` as a programmatic dependent of the work before it.
template <typename K>
static cudaError_t launch_dependent(K kern, unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                                    const Args &A) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, A);
}

// Stream-kernel shape for a call: CTAs, parts of a split row, ring stages and the dynamic shared
// memory of the three kernels; false when the kernels cannot be resident for this vocabulary.
struct StreamPlan {
    long long ctas;
    size_t smem1, smem2, smem3;
};

template <typename E>
static bool plan_stream(Args &B, const LaunchOpts &o, StreamPlan &pl) {
    pl.ctas = (long long)o.nsm * stream_ctas<E>();
    B.ctas = (int)pl.ctas;
    // the last wave of rows (one per CTA) is split into parts of at least 2 chunks
#ifndef SV_PART_MIN
#define SV_PART_MIN 6
#endif
    const long long nc = ((long long)B.V * sizeof(E) + SB - 1) / SB;
    B.nparts = (int)(nc / SV_PART_MIN < SPLIT_PARTS ? nc / SV_PART_MIN : SPLIT_PARTS);
    if (B.nparts < 2 || B.R < 2) B.nparts = 1;
    // shared memory of one stream CTA when SCTA share an SM (228 KB, 1 KB reserved per CTA)
    const size_t budget = (stream_ctas<E>() == 1 ? (size_t)232448 : (size_t)233472 / stream_ctas<E>() - 1024) - sizeof(SShared);
    B.pns = PNS_MAX;
    while (B.pns > 3 && stream_smem(B.nseg, B.pns) > budget) B.pns--;
    pl.smem1 = stream_smem(B.nseg, B.pns);
    pl.smem2 = select_smem(B.nseg);
    pl.smem3 = (size_t)2 * nseg_pad(B.nseg) * 4;
    return pl.smem1 <= budget && pl.smem2 <= (size_t)232448 - sizeof(RowCtx) &&
           pl.smem3 <= (size_t)232448 - sizeof(RowCtx);
}

// Grid of a stream launch over `rows` rows (the stream kernel splits the same way).
static unsigned stream_grid(const Args &B, long long ctas, long long rows) {
    const long long nsplit = B.nparts > 1 ? (ctas * SPLIT_WAVES < rows ? ctas * SPLIT_WAVES : rows) : 0;
    const long long units = rows - nsplit + nsplit * B.nparts;
    return (unsigned)(ctas < units ? ctas : units);
}

// Launches the stream kernel (SCTA CTAs per SM) and the select kernel as its programmatic
// dependent, in scheme SCH (SCH_GRID or SCH_ROWS); returns cudaErrorNotSupported (nothing
// launched) when the kernels cannot be resident for this vocabulary.
template <typename E, bool QVEC, int SCH>
static cudaError_t launch_two_kernels(const Args &A, cudaStream_t stream, const LaunchOpts &o) {
    Args B = A;
    StreamPlan pl;
    if (!plan_stream<E>(B, o, pl)) return cudaErrorNotSupported;
    // the stream kernel with the history variants only when the call passes a history
    auto k1 = A.hoff ? stream_kernel<E, true, SCH> : stream_kernel<E, false, SCH>;
    auto k2 = select_kernel<E, QVEC, SCH>;
    cudaError_t e;
    if ((e = ensure_smem(k1, pl.smem1)) != cudaSuccess) return e;
    if ((e = ensure_smem(k2, pl.smem2)) != cudaSuccess) return e;
    B.phase = 0;
    B.nsplit = B.nparts > 1 ? (int)(pl.ctas * SPLIT_WAVES < A.R ? pl.ctas * SPLIT_WAVES : A.R) : 0;
    if (o.ph0 && (e = cudaEventRecord(o.ph0, stream)) != cudaSuccess) return e;
    // a programmatic dependent of the clearing kernel (or of the history prepass)
    if ((e = launch_dependent(k1, stream_grid(B, pl.ctas, A.R), stream_threads<E>(), pl.smem1, stream, B)) != cudaSuccess) return e;
    if (o.ph1 && (e = cudaEventRecord(o.ph1, stream)) != cudaSuccess) return e;
    // With queued residuals, the worker CTAs follow the row CTAs: when the rows take one wave
    // of select CTAs, as many workers as the wave leaves slots for (at least half an SM's
    // worth), so that no second wave of CTAs ends the kernel; otherwise WORKERS_PER_SM per SM,
    // one slot per SM short of the select CTAs an SM holds, so that row CTAs always find slots
    // whatever order the CTAs are dispatched in.  Never more than every job's slices.
    if (RESIDQ && A.R > A.B) {
        const long long slots = (long long)o.nsm * SEL_PER_SM, most = (long long)A.B * RSL;
        long long w = A.R <= slots ? slots - A.R : (long long)o.nsm * WORKERS_PER_SM;
        if (w < o.nsm / 2) w = o.nsm / 2;
        B.nworkers = (int)(w < most ? w : most);
    }
    return launch_dependent(k2, (unsigned)(A.R + B.nworkers), SELT, pl.smem2, stream, B);
}

// The lazy scheme: both kernels over each request's row 0, both over the rows the first phase
// queued, then the residual kernel -- each launch a programmatic dependent of the one before.
template <typename E, bool QVEC>
static cudaError_t launch_lazy_kernels(const Args &A, cudaStream_t stream, const LaunchOpts &o) {
    Args B = A;
    StreamPlan pl;
    if (!plan_stream<E>(B, o, pl)) return cudaErrorNotSupported;
    auto k1 = A.hoff ? stream_kernel<E, true, SCH_LAZY> : stream_kernel<E, false, SCH_LAZY>;
    auto k2 = select_kernel<E, QVEC, SCH_LAZY>;
    auto k3 = resid_kernel<E, QVEC>;
    cudaError_t e;
    if ((e = ensure_smem(k1, pl.smem1)) != cudaSuccess) return e;
    if ((e = ensure_smem(k2, pl.smem2)) != cudaSuccess) return e;
    if ((e = ensure_smem(k3, pl.smem3)) != cudaSuccess) return e;
    B.phase = 1;
    if ((e = launch_dependent(k1, stream_grid(B, pl.ctas, A.B), stream_threads<E>(), pl.smem1, stream, B)) != cudaSuccess) return e;
    if ((e = launch_dependent(k2, (unsigned)A.B, SELT, pl.smem2, stream, B)) != cudaSuccess) return e;
    if (A.R == A.B) return cudaSuccess;   // no drafts: nothing is queued
    B.phase = 2;
    if ((e = launch_dependent(k1, (unsigned)pl.ctas, stream_threads<E>(), pl.smem1, stream, B)) != cudaSuccess) return e;
    if ((e = launch_dependent(k2, (unsigned)(A.R - A.B), SELT, pl.smem2, stream, B)) != cudaSuccess) return e;
    return launch_dependent(k3, resid_grid(A), RST, pl.smem3, stream, B);
}

// The one-pass call for logits of type E with whole-grid selection: the two kernels for aligned
// rows they can hold, else the row kernel (any alignment).
template <typename E>
static cudaError_t launch_onepass_dtype(const Args &A, cudaStream_t st, const LaunchOpts &o, bool vec, bool qvec) {
    cudaError_t e = cudaErrorNotSupported;
    if (vec) e = qvec ? launch_two_kernels<E, true, SCH_GRID>(A, st, o) : launch_two_kernels<E, false, SCH_GRID>(A, st, o);
    if (e == cudaErrorNotSupported) {
        cudaGetLastError();   // clear a sticky "not supported" from the probe, if any
        if (vec) e = qvec ? launch_rows<E, true, true>(A, st) : launch_rows<E, true, false>(A, st);
        else e = qvec ? launch_rows<E, false, true>(A, st) : launch_rows<E, false, false>(A, st);
    }
    return e;
}

}  // namespace sv

// sv_row.cuh -- per-row work of the verify kernels: locating a row and its request, the
// presence/frequency penalties of the drafts before it, the per-segment statistics of the
// streamed row, the kept set (top-k / top-p), and draws by inverse CDF.
//
// Method ("Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust",
// "The Verification Algorithm"; FreeToken PR #836, "Design"): each of a request's k+1 target
// rows becomes p = softmax(z / T) over the tokens kept by top-k and then top-p, where
// z = logit - presence*[c > 0] - frequency*c counts the drafts before the row.
//
// Everything that works on a whole row is templated on a thread group G (sv_block.cuh), so
// the same code serves the one-CTA-per-row kernel and the select kernel.  Sums that feed a decision use a fixed association: results are bitwise
// reproducible run to run.
#pragma once

#include <stddef.h>

#include "sv_block.cuh"

namespace sv {

// One row and its request, plus the scratch the row's selection uses.  The first PREP_BYTES
// (everything about the row that does not depend on its logits' statistics) are laid out so
// that they can be copied verbatim between kernels.
struct __align__(16) RowCtx {
    // ---- the row (prepared once; PREP_BYTES)
    int r, b, i, k, r0, d0, nrows, status, active, greedy, K;
    float T, P, pres, freq, s;
    int topk_on, topp_on, need_sum, mode;
    int npen;
    int xtok;       // the row's draft token (-1 if none), its penalised target value and q value
    float zx, qx;
    float u1;       // slot-1 uniform of the row (sampled rows: extra-token, residual or
                    // one-hot-scheme draw)
    int tix;        // index of the row's (or unit's) timing record
    // the request's prior history (penalised rows with a non-empty history, else all NULL):
    // hdir[s] .. hdir[s+1] index the entries of 256-token segment s in htok / hcnt
    const int32_t *hdir;
    const int32_t *htok;
    const int32_t *hcnt;
    int pid[MAXK];
    float ppen[MAXK];
    // ---- stream kernel: the work unit
    int c0, c1;     // chunks [c0, c1) of the row form this work unit
    int part;       // part index and number of parts of the unit's row (1: streamed whole)
    int nparts;
    int draft_raw[MAXK];
    // selection scratch
    float m;
    float redf[16];
    int redi[16];
    int ncand, nsel, n2;
    float zk;
    uint32_t cutkey;
    int sel_digit;
    long long sel_below;
    unsigned long long sel_mass;
    double sel_target;
    int last, a, tok, need_resid, plast;
    int prepped;    // select path: the candidate segment lists are already built
    double redd[16];          // per-warp partials of fp64 reductions
    double dtarget, dbefore;  // draws over segments: u * W and the running total before the crossing
};

constexpr int PREP_BYTES = 32 * 4 + 2 * MAXK * 4;
static_assert(offsetof(RowCtx, pid) == 128 && offsetof(RowCtx, c0) == PREP_BYTES, "RowCtx prepared prefix");

// Records a device-data error: the first code wins; the lowest request index is kept.
__device__ __forceinline__ void record_error(const Args &A, int code, int b) {
    atomicCAS(A.hdr, 0, code);
    atomicMax(A.hdr + 1, 0x7fffffff - b);
}

// ------------------------------------------------------------------------------------------
// locating a row and its request
// ------------------------------------------------------------------------------------------

// Largest index j in [0, B] with off[j] <= r (off non-decreasing), or -1; run by one warp
// as a 32-way search (each round narrows the range 32-fold).
__device__ __forceinline__ int find_request(const int32_t *off, int B, int r) {
    const int lane = lane_id();
    int lo = 0, hi = B + 1, ans = -1;
    while (lo < hi) {
        int n = hi - lo;
        int step = (n + 31) / 32;
        int idx = lo + lane * step;
        bool le = (lane * step < n) && (__ldg(off + idx) <= r);
        unsigned msk = __ballot_sync(0xffffffffu, le);
        if (msk == 0) break;
        int L = 31 - __clz(msk);
        ans = lo + L * step;
        lo = ans + 1;
        hi = min(hi, ans + step);
    }
    return ans;
}

// ------------------------------------------------------------------------------------------
// streaming order and per-row readiness (one-pass call)
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Waits (one thread, bounded, sleeping between polls) until pred(*p) holds; the word's last
// value goes to *last.  False once WAIT_NS has passed.  `ld` is an acquiring load; the polls
// in between are plain volatile reads, so that many waiters do not fence the memory system.
template <typename T, typename LD, typename PRED>
__device__ __forceinline__ bool wait_word(const T *p, LD ld, PRED pred, T *last) {
    T v = ld(p);
    if (pred(v)) {
        *last = v;
        return true;
    }
    const unsigned long long t0 = global_ns();
    unsigned ns = 32;
    for (;;) {
        __nanosleep(ns);
        ns = ns < 256 ? ns * 2 : 256;
        if (pred(*reinterpret_cast<const volatile T *>(p))) {
            *last = v = ld(p);   // (the condition is monotone: it still holds)
            return true;
        }
        if (global_ns() - t0 > WAIT_NS) {
            *last = *reinterpret_cast<const volatile T *>(p);
            return false;
        }
    }
}

// Row at streaming position li (written by the clearing kernel, read through L2).
__device__ __forceinline__ int order_row(const Args &A, int li) { return __ldcg(A.rowmap + li); }

// The streaming order of a one-pass call: requests with sampled rows first, greedy ones last
// (each group in request order), as the row at each position.  A greedy row's selection is
// short, so rows streamed last finish soon after the stream; the sampled rows' longer
// selections overlap the greedy rows' streaming.  Run by one block of NT threads, which first
// zeroes every row's ready word; the stream kernel waits for this block.  A request's first
// position is the rows of the requests before it in its own group (one block-wide scan per
// group), after every sampled row when it is greedy.  Publishes key << 32 | 2 * epoch in
// *ordflag once written, or with + 1 (the identity order) when row_offsets are inconsistent --
// then every row keeps its place and the kernels' own checks report the layout.
template <int NT>
__device__ void build_order(const Args &A) {
    constexpr int NW = NT / 32;
    __shared__ int s_red[2][NW];
    __shared__ int s_carry[2];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int B = A.B;
    const unsigned long long tag = (unsigned long long)A.key << 32;
    // Every row's ready word, zeroed before the flag below publishes the order: a select CTA
    // reads its row's word only after that flag, so it never sees a stale word, which could
    // hold any value (the workspace is the caller's memory).
    for (int r = t; r < A.R; r += NT) A.ready[r] = 0u;
    // the layout's consistency, and the rows of the sampled group
    bool ok = true;
    int samp = 0;
    for (int b = t; b < B; b += NT) {
        const int r0 = A.row_off ? __ldg(A.row_off + b) : b * (A.k_max + 1);
        const int r1 = A.row_off ? __ldg(A.row_off + b + 1) : r0 + A.k_max + 1;
        if (r1 < r0 || (b == 0 && r0 != 0) || (b == B - 1 && r1 != A.R)) ok = false;
        if (!__ldg(A.greedy + b)) samp += r1 - r0;
    }
    if (!__syncthreads_and(ok)) {
        if (t == 0) st_release_u64(A.ordflag, tag | (2u * A.epoch + 1u));
        return;
    }
    // (consistent offsets: every count is >= 0 and they sum to R, so positions stay below R)
    for (int o = 16; o > 0; o >>= 1) samp += __shfl_xor_sync(0xffffffffu, samp, o);
    if (lane == 0) s_red[0][warp] = samp;
    __syncthreads();
    if (t == 0) {
        int tot = 0;
        for (int w = 0; w < NW; w++) tot += s_red[0][w];
        s_carry[0] = 0;     // next position of the sampled group
        s_carry[1] = tot;   // next position of the greedy group
    }
    __syncthreads();
    for (int b0 = 0; b0 < B; b0 += NT) {
        const int b = b0 + t;
        int r0 = 0, n = 0;
        bool gr = false;
        if (b < B) {
            r0 = A.row_off ? __ldg(A.row_off + b) : b * (A.k_max + 1);
            n = (A.row_off ? __ldg(A.row_off + b + 1) : r0 + A.k_max + 1) - r0;
            gr = __ldg(A.greedy + b) != 0;
        }
        // inclusive warp scans of the two groups' row counts
        int is = gr ? 0 : n, ig = gr ? n : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ys = __shfl_up_sync(0xffffffffu, is, o), yg = __shfl_up_sync(0xffffffffu, ig, o);
            if (lane >= o) {
                is += ys;
                ig += yg;
            }
        }
        if (lane == 31) {
            s_red[0][warp] = is;
            s_red[1][warp] = ig;
        }
        __syncthreads();
        int cs = s_carry[0], cg = s_carry[1];
        for (int w = 0; w < warp; w++) {
            cs += s_red[0][w];
            cg += s_red[1][w];
        }
        const int pos = gr ? cg + ig - n : cs + is - n;
        for (int j = 0; j < n; j++) A.rowmap[pos + j] = r0 + j;
        __syncthreads();
        if (t == 0) {
            for (int w = 0; w < NW; w++) {
                s_carry[0] += s_red[0][w];
                s_carry[1] += s_red[1][w];
            }
        }
        __syncthreads();
    }
    // (the barrier above orders every thread's writes before this release)
    if (t == 0) st_release_u64(A.ordflag, tag | (2u * A.epoch));
}

// One finished share of row r (a streamed unit: the whole row, or one of its parts): the share
// that completes the row publishes it ready for this call.  One thread, whose release covers
// the writes it has synchronised with (the unit's streamer warps, through the unit barrier).
__device__ __forceinline__ void row_share_done(const Args &A, int r, int shares) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(A.partcnt + r) : "memory");
    if (old == shares - 1) st_release_u32(A.ready + r, A.epoch);
}

// Request-level checks shared by every row of the request (one thread).
__device__ __forceinline__ void load_request(const Args &A, RowCtx &S, int b) {
    S.b = b;
    const int k = __ldg(A.nd + b);
    const int greedy = __ldg(A.greedy + b) != 0;
    const float pres = A.pres ? __ldg(A.pres + b) : 0.f;
    const float freq = A.freq ? __ldg(A.freq + b) : 0.f;
    // every field is loaded up front (one round trip); greedy requests ignore T, P and K
    const float T = __ldg(A.T + b);
    const float P = __ldg(A.topp + b);
    const int K = __ldg(A.topk + b);
    int status = 0;
    if (k < 0 || k > A.k_max || k > S.nrows - 1) status = 1;           // SV_DEV_BAD_LAYOUT
    if (!isfinite(pres) || !isfinite(freq)) status = status ? status : 6;
    // the prior history, checked and indexed by the prepass
    S.hdir = nullptr;
    S.htok = nullptr;
    S.hcnt = nullptr;
    if (A.hoff) {
        if (__ldg(A.hstat + b) != 0) {
            status = status ? status : 8;
        } else if (__ldg(A.hoff + b + 1) > __ldg(A.hoff + b) && (pres != 0.f || freq != 0.f)) {
            S.hdir = A.hdir + (size_t)b * (nseg_pad(A.nseg) + 1);
            S.htok = A.htok;
            S.hcnt = A.hcnt;
        }
    }
    S.k = k;
    S.greedy = greedy;
    S.pres = pres;
    S.freq = freq;
    S.T = 1.f;
    S.P = 1.f;
    S.K = 0;
    if (!greedy) {
        if (!(T > 0.f) || !isfinite(T)) status = status ? status : 3;
        if (!(P > 0.f && P <= 1.f)) status = status ? status : 4;
        S.T = T;
        S.P = P;
        S.K = K;
    }
    S.status = status;
}

// Everything about row r that does not depend on its data: request, validity, sampling
// parameters and filter switches.  Run by one warp.
__device__ __forceinline__ void locate_row(const Args &A, RowCtx &S, int r) {
    const int lane = lane_id();
    int b, r0, nrows;
    bool ok = true;
    if (A.row_off) {
        b = find_request(A.row_off, A.B, r);
        ok = b >= 0 && b < A.B;
        r0 = ok ? __ldg(A.row_off + b) : 0;
        const int r1 = ok ? __ldg(A.row_off + b + 1) : 0;
        ok = ok && r0 <= r && r < r1;
        nrows = r1 - r0;
    } else {
        b = r / (A.k_max + 1);
        r0 = b * (A.k_max + 1);
        nrows = A.k_max + 1;
    }
    if (lane == 0) {
        S.r = r;
        S.tix = r;
        S.part = 0;
        S.r0 = r0;
        S.nrows = nrows;
        S.i = r - r0;
        S.d0 = r0 - b;
        S.K = 0;
        S.greedy = 0;
        S.T = 1.f;
        S.P = 1.f;
        if (ok) {
            load_request(A, S, b);
        } else {
            // a row outside every request (inconsistent row_offsets): nothing to count
            S.b = -1;
            S.k = 0;
            S.status = 1;
            record_error(A, 1, b < 0 ? 0 : (b >= A.B ? A.B - 1 : b));
        }
        S.active = ok && S.status == 0 && S.i <= S.k;
        const bool sampled = !S.greedy;
        S.s = sampled ? __fdiv_rn(LOG2E, S.T) : 0.f;
        S.topk_on = sampled && S.K > 0 && S.K < A.V;
        S.topp_on = sampled && S.P < 1.f;
        S.need_sum = sampled && !S.topk_on && !S.topp_on;
        S.mode = !sampled ? MODE_ARG : (S.need_sum ? MODE_SUM : ((S.topk_on && S.K <= KCAP) ? MODE_TOP2 : MODE_MAX));
        S.xtok = -1;
        S.zx = 0.f;
        S.qx = 0.f;
        S.npen = 0;
    }
    __syncwarp();
}

// History entry of token x in the request's prior history, or -1 (one thread).
__device__ __forceinline__ int hist_find(const RowCtx &S, int x) {
    const int seg = x / SEG;
    const int lo = __ldg(S.hdir + seg), hi = __ldg(S.hdir + seg + 1);
    for (int j = lo; j < hi; j++)
        if (__ldg(S.htok + j) == x) return j;
    return -1;
}

// Penalty of history entry j: presence once plus frequency per occurrence.
__device__ __forceinline__ float hist_pen(const RowCtx &S, int j) {
    return __fadd_rn(S.pres, __fmul_rn(S.freq, (float)__ldg(S.hcnt + j)));
}

// Penalties of row i: the distinct drafts d_0..d_{i-1} with pen = presence + frequency * count
// (FreeToken PR #836, "Design": earlier drafts count as already generated).  A draft that is
// also in the request's prior history already carries that entry's penalty (presence and its
// history count), so its list entry adds only frequency * its count among the drafts.  Run by
// one warp.
__device__ __forceinline__ void build_penalties(const Args &A, RowCtx &S, int i) {
    const int lane = lane_id();
    if (lane == 0) S.npen = 0;
    __syncwarp();
    if (i <= 0 || (S.pres == 0.f && S.freq == 0.f)) return;
    for (int j = lane; j < i; j += 32) S.draft_raw[j] = __ldg(A.tokens + S.d0 + j);
    __syncwarp();
    for (int base = 0; base < i; base += 32) {
        int j = base + lane;
        bool keep = false;
        int v = -1;
        float pen = 0.f;
        if (j < i) {
            v = S.draft_raw[j];
            bool first = true;
            int c = 0;
            for (int t = 0; t < i; t++) {
                int dt = S.draft_raw[t];
                if (dt == v) {
                    c++;
                    if (t < j) first = false;
                }
            }
            const bool ok = v >= 0 && v < A.V;
            const bool inhist = ok && first && S.hdir && hist_find(S, v) >= 0;
            pen = inhist ? __fmul_rn(S.freq, (float)c) : __fadd_rn(S.pres, __fmul_rn(S.freq, (float)c));
            keep = first && ok && pen != 0.f;
        }
        unsigned msk = __ballot_sync(0xffffffffu, keep);
        int pos = S.npen + __popc(msk & ((1u << lane) - 1));
        if (keep) {
            S.pid[pos] = v;
            S.ppen[pos] = pen;
        }
        __syncwarp();
        if (lane == 0) S.npen += __popc(msk);
        __syncwarp();
    }
}

// Applies the penalties to the 8 values this lane holds for the segment starting at seg_lo
// (lane owns elements seg_lo + 8*lane .. +7).  Whole warp must call it.
// The history entries of the segment starting at seg_lo, applied to this lane's 8 values.
// Whole warp.
__device__ __forceinline__ void patch_hist(const RowCtx &S, int seg_lo, float v[8]) {
    const int lane = lane_id();
    {
        const int seg = seg_lo / SEG;
        const int lo = __ldg(S.hdir + seg), hi = __ldg(S.hdir + seg + 1);
        const int my = seg_lo + lane * 8;
        for (int j0 = lo; j0 < hi; j0 += 32) {
            const int j = j0 + lane;
            int x = -1;
            float pen = 0.f;
            if (j < hi) {
                x = __ldg(S.htok + j);
                pen = hist_pen(S, j);
            }
            unsigned m = __ballot_sync(0xffffffffu, j < hi);
            while (m) {
                const int h = __ffs(m) - 1;
                m &= m - 1;
                const int d = __shfl_sync(0xffffffffu, x, h) - my;
                const float ph = __shfl_sync(0xffffffffu, pen, h);
#pragma unroll
                for (int t = 0; t < 8; t++)
                    if (d == t) v[t] = __fsub_rn(v[t], ph);
            }
        }
    }
}

// History entries (the request's prior history) are applied first, then the drafts' list;
// every site that penalises values uses this order, so all of them compute the same floats.
// HIST = false leaves the history out (callers that know the row has none).
template <bool HIST = true>
__device__ __forceinline__ void patch_seg(const RowCtx &S, int seg_lo, float v[8]) {
    const int npen = S.npen;
    const int lane = lane_id();
    if constexpr (HIST) {
        if (S.hdir) patch_hist(S, seg_lo, v);
    }
    if (npen == 0) return;
    bool h0 = lane < npen && (unsigned)(S.pid[lane] - seg_lo) < (unsigned)SEG;
    bool h1 = lane + 32 < npen && (unsigned)(S.pid[lane + 32] - seg_lo) < (unsigned)SEG;
    unsigned m0 = __ballot_sync(0xffffffffu, h0);
    unsigned m1 = __ballot_sync(0xffffffffu, h1);
    const int my = seg_lo + lane * 8;
    while (m0 | m1) {
        int h;
        if (m0) {
            h = __ffs(m0) - 1;
            m0 &= m0 - 1;
        } else {
            h = __ffs(m1) - 1 + 32;
            m1 &= m1 - 1;
        }
        int d = S.pid[h] - my;
        float pen = S.ppen[h];
#pragma unroll
        for (int j = 0; j < 8; j++)
            if (d == j) v[j] = __fsub_rn(v[j], pen);
    }
}

// The 8 values one thread holds at tokens base .. base+7 (base a multiple of 8, inside one
// segment), penalised in patch_seg's order.  One thread.
__device__ __forceinline__ void pen_lane8(const RowCtx &S, int base, float v[8]) {
    if (S.hdir) {
        const int seg = base / SEG;
        const int lo = __ldg(S.hdir + seg), hi = __ldg(S.hdir + seg + 1);
        for (int j = lo; j < hi; j++) {
            const int d = __ldg(S.htok + j) - base;
            if ((unsigned)d < 8u) {
                const float pen = hist_pen(S, j);
#pragma unroll
                for (int t = 0; t < 8; t++)
                    if (d == t) v[t] = __fsub_rn(v[t], pen);
            }
        }
    }
    for (int h = 0; h < S.npen; h++) {
        const int d = S.pid[h] - base;
#pragma unroll
        for (int t = 0; t < 8; t++)
            if (d == t) v[t] = __fsub_rn(v[t], S.ppen[h]);
    }
}

// Penalised value of token x (in [0, V)) from its stored value, in patch_seg's order.
__device__ __forceinline__ float elem_z(const RowCtx &S, float z, int x) {
    if (S.hdir) {
        const int j = hist_find(S, x);
        if (j >= 0) z = __fsub_rn(z, hist_pen(S, j));
    }
    for (int h = 0; h < S.npen; h++)
        if (S.pid[h] == x) z = __fsub_rn(z, S.ppen[h]);
    return z;
}
__device__ __forceinline__ float elem_z_raw(const RowCtx &S, uint16_t raw, int x) {
    return elem_z(S, __uint_as_float((uint32_t)raw << 16), x);
}
__device__ __forceinline__ float elem_z_raw(const RowCtx &S, float raw, int x) { return elem_z(S, raw, x); }

// One thread: the row's draft token and, for a valid one, its penalised target value and q.
template <typename E>
__device__ __forceinline__ void prefetch_draft(const Args &A, RowCtx &S, const E *row) {
    int x = -1;
    float zx = 0.f, qx = 0.f;
    if (S.active && S.i < S.k) {
        x = __ldg(A.tokens + S.d0 + S.i);
        if (x >= 0 && x < A.V) {
            const E raw = __ldg(row + x);
            if (!S.greedy) qx = A.onehot ? 1.f : __ldg(A.q + (size_t)(S.d0 + S.i) * A.V + x);
            zx = elem_z_raw(S, raw, x);
        }
    }
    S.xtok = x;
    S.zx = zx;
    S.qx = qx;
    S.u1 = (S.active && !S.greedy) ? __ldg(A.uni + (size_t)S.r * 2 + 1) : 0.f;
}

// Loads and penalises the 8 values of this lane in segment seg (global memory).
template <typename E, bool VEC>
__device__ __forceinline__ void seg_values(const RowCtx &S, const E *row, int V, int seg, float v[8]) {
    Raw8<E> raw = load_raw8<VEC>(row, seg * SEG + lane_id() * 8, V);
    unpack8(raw, v);
    patch_seg(S, seg * SEG, v);
}

// Calls f(seg, v, qv) for every segment s_lo <= seg < nseg of a row held in global memory (v:
// the lane's 8 penalised values; qv: the draft row's 8 values when WITHQ, else zeros).  Each
// warp takes segments s_lo + warp, s_lo + warp + kWarps, ... and has U of them in flight
// before it uses any, so a full pass is not one memory latency per segment.
// With aligned rows, one thread also keeps an L2 prefetch PF_SEGS segments ahead of the
// warps (of q too when it is read and aligned), so that their loads find the data in L2: a
// CTA's own loads in flight are far too few to cover the memory latency.
#ifndef SV_PF_SEGS
#define SV_PF_SEGS 32
#endif
constexpr int PF_SEGS = SV_PF_SEGS;

// Prefetches segments [a, b) of the row (and of q) into L2.  One thread.
template <typename E, bool QVEC, bool WITHQ>
__device__ __forceinline__ void prefetch_segs(const E *row, const float *qrow, int V, int a, int b) {
    const int e0 = a * SEG, e1 = min(b * SEG, V);
    if (e0 >= e1) return;
    bulk_prefetch_l2(row + e0, (uint32_t)((e1 - e0) * (int)sizeof(E)));
    if constexpr (WITHQ && QVEC) {
        if (qrow) bulk_prefetch_l2(qrow + e0, (uint32_t)((e1 - e0) * 4));
    }
}

template <typename E, bool VEC, bool QVEC, bool WITHQ, int U, class G, class F>
__device__ __forceinline__ void pass_segment_range(const G &g, const RowCtx &S, const E *row, const float *qrow,
                                                   int V, int s_lo, int nseg, F &&f) {
    const int lane = g.lane();
    constexpr int STEP = G::kWarps * U;
    if constexpr (VEC && PF_SEGS > 0) {
        if (g.t == 0) prefetch_segs<E, QVEC, WITHQ>(row, qrow, V, s_lo, min(s_lo + PF_SEGS, nseg));
    }
    for (int s0 = s_lo + g.warp(); s0 < nseg; s0 += STEP) {
        if constexpr (VEC && PF_SEGS > 0) {
            // (thread 0 is in warp 0, whose s0 is the step's first segment)
            if (g.t == 0) prefetch_segs<E, QVEC, WITHQ>(row, qrow, V, s0 + PF_SEGS, min(s0 + PF_SEGS + STEP, nseg));
        }
        Raw8<E> raw[U];
        float qv[U][8];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int seg = s0 + u * G::kWarps;
            if (seg < nseg) {
                raw[u] = load_raw8<VEC>(row, seg * SEG + lane * 8, V);
                if constexpr (WITHQ) load_q8<QVEC>(qrow, seg * SEG + lane * 8, V, qv[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int seg = s0 + u * G::kWarps;
            if (seg < nseg) {
                float v[8];
                unpack8(raw[u], v);
                patch_seg(S, seg * SEG, v);
                if constexpr (!WITHQ) {
#pragma unroll
                    for (int j = 0; j < 8; j++) qv[u][j] = 0.f;
                }
                f(seg, v, qv[u]);
            }
        }
    }
}

// As pass_segment_range over the whole row.
template <typename E, bool VEC, bool QVEC, bool WITHQ, int U, class G, class F>
__device__ __forceinline__ void pass_segments(const G &g, const RowCtx &S, const E *row, const float *qrow, int V,
                                              int nseg, F &&f) {
    pass_segment_range<E, VEC, QVEC, WITHQ, U>(g, S, row, qrow, V, 0, nseg, f);
}

// Per-segment statistics of a row, written by the streaming pass.
struct SegStats {
    float *mx;        // max of the segment
    float *b;         // MODE_TOP2: second-largest value (ties count); MODE_SUM: sum of 2^((z - mx) s)
    int *lane;        // MODE_ARG / MODE_TOP2: lowest lane whose 8 elements hold the max
    uint32_t *hist;   // MODE_TOP2: 256-bin histogram of the top byte of the maxima's order keys
};

// Reduces one segment, whose raw elements this lane holds 8 at a time (elements
// seg*SEG + 8*lane + t), to what the row's mode asks for; lane 0 writes it.  Warp-wide maxima
// are single redux.sync instructions; bf16 rows without penalties work on packed pairs.
template <typename E>
__device__ __forceinline__ void seg_stats(const Raw8<E> &raw, int seg, int V, const RowCtx &S, const SegStats &o) {
    const int lane = lane_id();
    const int mode = S.mode;
    float m1, m2 = -INFINITY, sum = 0.f;
    bool done = false;
    if constexpr (sizeof(E) == 2) {
        if (mode != MODE_SUM && S.npen == 0 && !S.hdir && seg * SEG + SEG <= V) {
            const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&raw.a);
            const __nv_bfloat162 a = __hmax2(p[0], p[1]), c = __hmax2(p[2], p[3]);
            const __nv_bfloat162 M = __hmax2(a, c);
            const float lo = __low2float(M), hi = __high2float(M);
            m1 = fmaxf(lo, hi);
            if (mode == MODE_TOP2) {
                // second largest of the lane's 8: max of the smaller half-max and the halves' seconds
                const __nv_bfloat162 b = __hmin2(p[0], p[1]), d = __hmin2(p[2], p[3]);
                const __nv_bfloat162 Sd = __hmax2(__hmin2(a, c), __hmax2(b, d));
                m2 = fmaxf(fminf(lo, hi), fmaxf(__low2float(Sd), __high2float(Sd)));
            }
            done = true;
        }
    }
    float v[8];
    if (!done) {
        unpack8(raw, v);
        const int base = seg * SEG + lane * 8;
        if (base + 8 > V) {
#pragma unroll
            for (int t = 0; t < 8; t++)
                if (base + t >= V) v[t] = -INFINITY;
        }
        patch_seg(S, seg * SEG, v);
        if (mode == MODE_TOP2) {
            m1 = v[0];
#pragma unroll
            for (int t = 1; t < 8; t++) {
                m2 = fmaxf(m2, fminf(m1, v[t]));
                m1 = fmaxf(m1, v[t]);
            }
        } else {
            m1 = max8(v);
        }
    }
    const float mx = redux_max(m1);
    int at = 0;
    float sec = 0.f;
    if (mode == MODE_ARG || mode == MODE_TOP2) {
        at = __ffs(__ballot_sync(0xffffffffu, m1 == mx)) - 1;
        if (mode == MODE_TOP2) sec = redux_max(lane == at ? m2 : m1);
    } else if (mode == MODE_SUM && mx > -INFINITY) {
        const float ms = __fmul_rn(mx, S.s);
#pragma unroll
        for (int t = 0; t < 8; t++) sum += ex2(fmaf(v[t], S.s, -ms));
        sum = warp_sum(sum);
    }
    if (lane == 0) {
        o.mx[seg] = mx;
        if (mode == MODE_ARG || mode == MODE_TOP2) o.lane[seg] = at;
        if (mode == MODE_TOP2) {
            o.b[seg] = sec;
            atomicAdd(&o.hist[fkey(mx) >> 24], 1u);
        }
        if (mode == MODE_SUM) o.b[seg] = sum;
    }
}

// One thread: token id of the first element equal to `target` among the 8 of `lane` in
// segment seg (penalties applied), or -1.
template <typename E, bool VEC>
__device__ __forceinline__ int find_in_lane(const RowCtx &S, const E *row, int V, int seg, int lane, float target) {
    const int base = seg * SEG + lane * 8;
    Raw8<E> raw = load_raw8<VEC>(row, base, V);
    float v[8];
    unpack8(raw, v);
    pen_lane8(S, base, v);
    int pos = -1;
#pragma unroll
    for (int t = 7; t >= 0; t--)
        if (v[t] == target && base + t < V) pos = base + t;
    return pos;
}

// One streaming read of the row by the group's warps with global loads (any alignment).
template <typename E, bool VEC, class G>
__device__ __forceinline__ void pass_stats(const G &g, const RowCtx &S, const E *row, int V, int nseg,
                                           const SegStats &o) {
    constexpr int U = sizeof(E) == 2 ? 2 : 1;   // segments in flight per warp
    const int warp = g.warp(), lane = g.lane();
    for (int s0 = warp; s0 < nseg; s0 += G::kWarps * U) {
        Raw8<E> raw[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            int seg = s0 + u * G::kWarps;
            if (seg < nseg) raw[u] = load_raw8<VEC>(row, seg * SEG + lane * 8, V);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            int seg = s0 + u * G::kWarps;
            if (seg < nseg) seg_stats<E>(raw[u], seg, V, S, o);
        }
    }
}

// Raw elements of segment j of a ring stage for this lane (16-byte aligned rows).
template <typename E>
__device__ __forceinline__ Raw8<E> ring_raw(const unsigned char *buf, int j);
template <>
__device__ __forceinline__ Raw8<uint16_t> ring_raw<uint16_t>(const unsigned char *buf, int j) {
    Raw8<uint16_t> r;
    r.a = *reinterpret_cast<const uint4 *>(buf + j * SEG * 2 + lane_id() * 16);
    return r;
}
template <>
__device__ __forceinline__ Raw8<float> ring_raw<float>(const unsigned char *buf, int j) {
    Raw8<float> r;
    const uint4 *p = reinterpret_cast<const uint4 *>(buf + j * SEG * 4 + lane_id() * 32);
    r.a = p[0];
    r.b = p[1];
    return r;
}

// Values of segment j of a ring stage (16-byte aligned rows: 8 elements per lane).
template <typename E>
__device__ __forceinline__ void ring_values(const unsigned char *buf, int j, float v[8]);
template <>
__device__ __forceinline__ void ring_values<uint16_t>(const unsigned char *buf, int j, float v[8]) {
    Raw8<uint16_t> r;
    r.a = *reinterpret_cast<const uint4 *>(buf + j * SEG * 2 + lane_id() * 16);
    unpack8(r, v);
}
template <>
__device__ __forceinline__ void ring_values<float>(const unsigned char *buf, int j, float v[8]) {
    Raw8<float> r;
    const uint4 *p = reinterpret_cast<const uint4 *>(buf + j * SEG * 4 + lane_id() * 32);
    r.a = p[0];
    r.b = p[1];
    unpack8(r, v);
}

// ------------------------------------------------------------------------------------------
// selection helpers (radix select, MSB first)
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ void digit_round(int round, int &shift, int &width, uint32_t &mask) {
    shift = 24 - 8 * round;
    width = 8;
    mask = round == 0 ? 0u : (0xFFFFFFFFu << (32 - 8 * round));
}

// One warp scans a count histogram from the highest bin down and finds the bin d holding the
// need-th largest element (cum_above(d) < need <= cum_above(d) + cnt[d]).  Writes S.sel_digit
// and S.sel_below (= cum_above(d)).  need >= 1; nbins a multiple of 32.
__device__ __forceinline__ void find_count_bin(RowCtx &S, const uint32_t *cnt, int nbins, long long need) {
    const int lane = lane_id();
    const int per = nbins / 32;
    const int top = nbins - lane * per;   // this lane covers bins [top - per, top)
    long long tot = 0;
    for (int d = top - 1; d >= top - per; d--) tot += cnt[d];
    long long incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    long long excl = incl - tot;
    bool mine = excl < need && need <= incl;
    unsigned msk = __ballot_sync(0xffffffffu, mine);
    int owner = msk ? __ffs(msk) - 1 : 31;
    if (lane == owner) {
        long long c = excl;
        int dsel = top - per;
        for (int d = top - 1; d >= top - per; d--) {
            if (c + (long long)cnt[d] >= need) {
                dsel = d;
                break;
            }
            c += cnt[d];
        }
        S.sel_digit = dsel;
        S.sel_below = c;
    }
}

// A lower bound on the need-th largest of n float keys in shared memory: the top 16 bits of
// that key (two 8-bit radix rounds) with the low 16 bits cleared.  At least `need` keys are
// >= the bound.
// hist1, when given, already holds the first round's histogram of the top byte.
template <class G>
__device__ uint32_t select_bound16(const G &g, RowCtx &S, const float *vals, int n, int need, uint32_t *cnt,
                                   const uint32_t *hist1 = nullptr) {
    uint32_t prefix = 0;
    long long nd = need;
    for (int round = 0; round < 2; round++) {
        const int shift = 24 - 8 * round;
        const uint32_t mask = round == 0 ? 0u : 0xFF000000u;
        const uint32_t *h = cnt;
        if (round == 0 && hist1) {
            h = hist1;
        } else {
            for (int d = g.t; d < 256; d += G::kThreads) cnt[d] = 0;
            g.sync();
            for (int j = g.t; j < n; j += G::kThreads) {
                const uint32_t key = fkey(vals[j]);
                if ((key & mask) == prefix) atomicAdd(&cnt[(key >> shift) & 255u], 1u);
            }
            g.sync();
        }
        if (g.warp() == 0) find_count_bin(S, h, 256, nd);
        g.sync();
        prefix |= (uint32_t)S.sel_digit << shift;
        nd -= S.sel_below;
        g.sync();
    }
    return prefix;
}

// The need-th largest key among the row's tokens (full passes over the row from global).
template <typename E, bool VEC, class G>
__device__ uint32_t select_kth_row(const G &g, RowCtx &S, const E *row, int V, int nseg, int need, uint32_t *cnt) {
    uint32_t prefix = 0;
    long long nd = need;
    const int warp = g.warp(), lane = g.lane();
    for (int round = 0; round < NRADIX; round++) {
        int shift, width;
        uint32_t mask;
        digit_round(round, shift, width, mask);
        const int nb = 1 << width;
        for (int d = g.t; d < nb; d += G::kThreads) cnt[d] = 0;
        g.sync();
        pass_segments<E, VEC, false, false, sizeof(E) == 2 ? 2 : 1>(
            g, S, row, nullptr, V, nseg, [&](int seg, const float *v, const float *) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const int idx = seg * SEG + lane * 8 + j;
                    const uint32_t key = fkey(v[j]);
                    if (idx < V && (key & mask) == prefix) atomicAdd(&cnt[(key >> shift) & (nb - 1)], 1u);
                }
            });
        g.sync();
        if (warp == 0) find_count_bin(S, cnt, nb, nd);
        g.sync();
        prefix |= (uint32_t)S.sel_digit << shift;
        nd -= S.sel_below;
        g.sync();
    }
    return prefix;
}

// One warp scans a fixed-point mass histogram from the top and finds the first bin d where
// the mass above plus the bin's own mass reaches target (above(d) < target <= ... + mass[d]).
__device__ __forceinline__ void find_mass_bin(RowCtx &S, const unsigned long long *mass, int nbins,
                                              unsigned long long above, double target) {
    const int lane = lane_id();
    const int per = nbins / 32;
    const int top = nbins - lane * per;
    unsigned long long tot = 0;
    for (int d = top - 1; d >= top - per; d--) tot += mass[d];
    unsigned long long incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    unsigned long long excl = incl - tot;
    bool mine = (double)(above + incl) >= target && (double)(above + excl) < target;
    unsigned msk = __ballot_sync(0xffffffffu, mine);
    int owner = msk ? __ffs(msk) - 1 : 31;
    if (lane == owner) {
        unsigned long long c = above + excl;
        int dsel = top - per;
        for (int d = top - 1; d >= top - per; d--) {
            if ((double)(c + mass[d]) >= target && mass[d] > 0) {
                dsel = d;
                break;
            }
            c += mass[d];
        }
        S.sel_digit = dsel;
        S.sel_mass = c;
    }
}

// Top-p threshold over the tokens with key >= key_lo: the lowest key level L whose mass
// strictly above is < P * (total mass of those tokens).  Fixed-point (2^-40) weights make the
// histogram sums exact and order-independent.  Each bin's sum is kept as limbs of lbits bits
// in 32-bit counters (V tokens of less than 2^lbits each cannot overflow one), because 32-bit
// shared-memory atomics stay fast where many tokens share a bin and 64-bit ones do not; the
// limbs are combined into the 64-bit histogram `mass` after each pass.
template <typename E, bool VEC, class G>
__device__ uint32_t select_mass_row(const G &g, RowCtx &S, const E *row, int V, int nseg, uint32_t key_lo,
                                    float m, float s, float P, unsigned long long *mass, uint32_t *limb) {
    uint32_t prefix = 0;
    unsigned long long above = 0;
    double target = 0.0;
    const int warp = g.warp(), lane = g.lane();
    const int lbits = V > 1 ? __clz(V - 1) : 31;        // 32 - ceil(log2 V) >= 11 for V <= 2^21
    const int nl = (41 + lbits - 1) / lbits;            // limbs covering 2^40 (at most 4)
    const unsigned long long lmask = (1ull << lbits) - 1ull;
    for (int round = 0; round < NRADIX; round++) {
        int shift, width;
        uint32_t mask;
        digit_round(round, shift, width, mask);
        const int nb = 1 << width;
        for (int d = g.t; d < 4 * nb; d += G::kThreads) limb[d] = 0u;
        g.sync();
        pass_segments<E, VEC, false, false, sizeof(E) == 2 ? 2 : 1>(
            g, S, row, nullptr, V, nseg, [&](int seg, const float *v, const float *) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const int idx = seg * SEG + lane * 8 + j;
                    const uint32_t key = fkey(v[j]);
                    if (idx < V && key >= key_lo && (key & mask) == prefix) {
                        const unsigned long long f = __float2ull_rz(__fmul_rn(weight(v[j], m, s), (float)FIXED_ONE));
                        const int bin = (key >> shift) & (nb - 1);
#pragma unroll
                        for (int l = 0; l < 4; l++) {
                            const uint32_t part = (uint32_t)((f >> (lbits * l)) & lmask);
                            if (l < nl && part) atomicAdd(&limb[l * nb + bin], part);
                        }
                    }
                }
            });
        g.sync();
        for (int d = g.t; d < nb; d += G::kThreads) {
            unsigned long long t = 0;
            for (int l = 0; l < nl; l++) t += (unsigned long long)limb[l * nb + d] << (lbits * l);
            mass[d] = t;
        }
        g.sync();
        if (round == 0) {
            // total mass of the top-k set (every bin of round 0), summed by one warp
            if (warp == 0) {
                unsigned long long t = 0;
                for (int d = lane; d < nb; d += 32) t += mass[d];
#pragma unroll
                for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == 0) S.sel_target = (double)P * (double)t;
            }
            g.sync();
            target = S.sel_target;
        }
        if (warp == 0) find_mass_bin(S, mass, nb, above, target);
        g.sync();
        prefix |= (uint32_t)S.sel_digit << shift;
        above = S.sel_mass;
        g.sync();
    }
    return prefix;
}

// ------------------------------------------------------------------------------------------
// draws by inverse CDF in token order
// ------------------------------------------------------------------------------------------

// Index j of the draw from weights w[0..n) in shared memory with uniform u: the first j whose
// running sum exceeds u * W (W = total); the last positive-weight j if rounding leaves none;
// -1 when no weight is positive.  `pre` (n floats) receives the prefix sums.
template <class G>
__device__ int draw_small(const G &g, const float *w, float *pre, int n, float u, RowCtx &S) {
    for (int j = g.t; j < n; j += G::kThreads) pre[j] = w[j];
    g.sync();
    if (n <= 0) return -1;
    g_scan_incl(g, pre, n, S.redf);
    float W = pre[n - 1];
    if (!(W > 0.f)) return -1;
    float target = __fmul_rn(u, W);
    int best = 0x7fffffff;
    for (int j = g.t; j < n; j += G::kThreads)
        if (pre[j] > target) best = min(best, j);
    best = g_min_i(g, best, S.redi);
    if (best == 0x7fffffff) {
        int last = -1;
        for (int j = g.t; j < n; j += G::kThreads)
            if (w[j] > 0.f) last = max(last, j);
        best = g_max_i(g, last, S.redi);
    }
    return best;
}

// Per-token weight functors for draws over whole rows.
struct WKept {       // unnormalised kept weight (extra-token draw)
    float m, s;
    uint32_t tk;
    __device__ __forceinline__ float operator()(float z, float) const {
        return fkey(z) >= tk ? weight(z, m, s) : 0.f;
    }
};
struct WProb {       // p_v
    float m, s, invZ;
    uint32_t tk;
    __device__ __forceinline__ float operator()(float z, float) const {
        return fkey(z) >= tk ? __fmul_rn(weight(z, m, s), invZ) : 0.f;
    }
};
struct WResid {      // max(0, p_v - q_v)
    float m, s, invZ;
    uint32_t tk;
    __device__ __forceinline__ float operator()(float z, float q) const {
        float p = fkey(z) >= tk ? __fmul_rn(weight(z, m, s), invZ) : 0.f;
        return fmaxf(__fsub_rn(p, q), 0.f);
    }
};

// The segment of a draw over per-segment weights segw[0..nseg): the first segment whose running
// total exceeds u * W (W = the total), with the running totals in fp64 and a fixed association
// (thread chunks, then lanes, then warps), so that the boundary does not drift over a long row.
// S.dtarget receives u * W, S.dbefore the running total before the segment.  With no segment
// above the target (rounding), the last segment of positive weight, and *fallback is set.
// Returns -1 when no weight is positive.
template <class G>
__device__ int crossing_segment(const G &g, RowCtx &S, const float *segw, int nseg, float u, bool &fallback) {
    const int lane = g.lane(), warp = g.warp();
    const int per = (nseg + G::kThreads - 1) / G::kThreads;
    const int lo = min(nseg, g.t * per), hi = min(nseg, lo + per);
    double t = 0.0;
    for (int j = lo; j < hi; j++) t += (double)segw[j];
    double incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) S.redd[warp] = incl;
    g.sync();
    double W = 0.0, run = 0.0;
#pragma unroll
    for (int w = 0; w < G::kWarps; w++) {
        if (w < warp) run += S.redd[w];
        W += S.redd[w];
    }
    run += incl - t;   // this thread's chunk starts here
    const double target = (double)u * W;
    int best = 0x7fffffff;
    double before = 0.0;
    if (W > 0.0) {
        for (int j = lo; j < hi; j++) {
            const double nx = run + (double)segw[j];
            if (nx > target) {
                best = j;
                before = run;
                break;
            }
            run = nx;
        }
    }
    g.sync();
    best = g_min_i(g, best, S.redi);
    fallback = false;
    if (best != 0x7fffffff) {
        if (best >= lo && best < hi) {
            S.dtarget = target;
            S.dbefore = before;
        }
    } else {
        if (!(W > 0.0)) return -1;
        int last = -1;
        for (int j = g.t; j < nseg; j += G::kThreads)
            if (segw[j] > 0.f) last = max(last, j);
        best = g_max_i(g, last, S.redi);
        fallback = true;
        if (best < 0) return -1;
        if (g.t == 0) {
            S.dtarget = target;
            S.dbefore = 0.0;
        }
    }
    g.sync();
    return best;
}

// Draw from a whole row with per-segment weight sums segw[0..nseg): the crossing segment from
// fp64 running totals (crossing_segment), then that segment re-read by the group's first warp
// and scanned lane by lane against what remains of u * W.  Returns the token, or -1 when no
// weight is positive.
template <typename E, bool VEC, bool QVEC, typename WF, class G>
__device__ int draw_by_segments(const G &g, RowCtx &S, const E *row, const float *qrow, int V, int nseg,
                                const float *segw, float u, const WF &wf) {
    bool fallback = false;
    const int best = crossing_segment(g, S, segw, nseg, u, fallback);
    if (best < 0) return -1;
    if (g.warp() == 0) {
        const int lane = g.lane();
        const int seg = best;
        float v[8], qv[8];
        seg_values<E, VEC>(S, row, V, seg, v);
        if (qrow) {
            load_q8<QVEC>(qrow, seg * SEG + lane * 8, V, qv);
        } else {
#pragma unroll
            for (int j = 0; j < 8; j++) qv[j] = 0.f;
        }
        float w[8];
        float loc = 0.f;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            int idx = seg * SEG + lane * 8 + j;
            w[j] = idx < V ? wf(v[j], qv[j]) : 0.f;
            loc += w[j];
        }
        float incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        float run = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) run = 0.f;
        // what remains of the target inside this segment (small: the segment's own scale)
        const float rem = (float)(S.dtarget - S.dbefore);
        int pick = 0x7fffffff, lastpos = -1;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            int idx = seg * SEG + lane * 8 + j;
            run += w[j];
            if (!fallback && run > rem && pick == 0x7fffffff) pick = idx;
            if (w[j] > 0.f) lastpos = idx;
        }
        pick = warp_min_i(pick);
        lastpos = warp_max_i(lastpos);
        if (lane == 0) S.tok = pick != 0x7fffffff ? pick : lastpos;
    }
    g.sync();
    return S.tok;
}

// Per-segment sums of weight functors over the whole row (one pass; q row optional).
template <typename E, bool VEC, bool QVEC, typename WF, typename WF2, class G>
__device__ __forceinline__ void seg_sums(const G &g, const RowCtx &S, const E *row, const float *qrow, int V,
                                         int nseg, float *out1, const WF &wf1, float *out2, const WF2 &wf2) {
    const int lane = g.lane();
    auto body = [&](int seg, const float *v, const float *qv) {
        float a = 0.f, c = 0.f;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int idx = seg * SEG + lane * 8 + j;
            if (idx < V) {
                a += wf1(v[j], qv[j]);
                if (out2) c += wf2(v[j], qv[j]);
            }
        }
        a = warp_sum(a);
        if (out2) c = warp_sum(c);
        if (lane == 0) {
            out1[seg] = a;
            if (out2) out2[seg] = c;
        }
    };
    if (qrow) pass_segments<E, VEC, QVEC, true, sizeof(E) == 2 ? 2 : 1>(g, S, row, qrow, V, nseg, body);
    else pass_segments<E, VEC, QVEC, false, sizeof(E) == 2 ? 2 : 1>(g, S, row, nullptr, V, nseg, body);
    g.sync();
}

}  // namespace sv

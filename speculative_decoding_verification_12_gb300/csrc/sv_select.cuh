// sv_select.cuh -- what happens to a row once its per-segment statistics exist: the kept set
// (top-k / top-p), the draws, p(x_i) and q(x_i) of the row's draft, and -- once every row of a
// request is done -- the request's first-rejection scan and final token.
//
// "Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust":
//  - "The Memory Bandwidth Wall and Speculative Math": accept x_i with probability
//    min(1, p(x_i)/q(x_i)); at the first rejection draw from max(0, p - q) normalised.
//  - "The Verification Algorithm": stop at the first rejection; with every draft accepted the
//    extra token comes from row K.
// "Adding Speculative Decoding", table "The existing base": greedy accepts while the draft is
// the argmax; the token at the first mismatch is that row's argmax.
//
// Everything here is templated on the thread group G that runs it.
#pragma once

#include "sv_row.cuh"

namespace sv {

// Shared-memory scratch of the group that selects rows and finalises requests.
struct Scratch {
    float *segX, *segY;           // per-segment scratch (segment lists, residual sums)
    unsigned long long *cand;     // CAP candidate keys (order key << 32) | ~token
    float *aux, *aux2;            // CAP floats each
    unsigned long long *sorted;   // WCAP keys (aliases aux/aux2)
    uint32_t *hcnt;               // radix histogram (aliases aux)
    unsigned long long *hmass;    // fixed-point mass histogram (aliases aux)
    uint32_t *hlimb;              // its 32-bit limb counters, 4 x HB (aliases cand and hcnt)
    unsigned char *big;           // the group's whole dynamic shared memory (row statistics, then
    size_t big_bytes;             // the areas above), for passes that need it after the row max
};

// Carves a Scratch out of `p`: segX/segY (nsegp floats each) then the candidate area.  `base`
// and `bytes` give the group's whole dynamic shared memory (it starts with the row's segment
// statistics and ends with this scratch).
__device__ __forceinline__ Scratch carve_scratch(unsigned char *p, int nsegp, unsigned char *base, size_t bytes) {
    Scratch c;
    c.big = base;
    c.big_bytes = bytes;
    c.segX = reinterpret_cast<float *>(p);
    c.segY = c.segX + nsegp;
    unsigned char *area = reinterpret_cast<unsigned char *>(c.segY + nsegp);
    c.cand = reinterpret_cast<unsigned long long *>(area);
    c.aux = reinterpret_cast<float *>(area + size_t(CAP) * 8);
    c.aux2 = c.aux + CAP;
    c.sorted = reinterpret_cast<unsigned long long *>(c.aux);
    c.hmass = reinterpret_cast<unsigned long long *>(area + size_t(CAP) * 8);
    c.hlimb = reinterpret_cast<uint32_t *>(area);
    c.hcnt = reinterpret_cast<uint32_t *>(area + size_t(HB) * 8);
    return c;
}
__host__ __device__ inline size_t scratch_bytes(int nsegp) { return size_t(2) * nsegp * 4 + size_t(CAP) * 16; }

#ifdef SV_TIMING
#define SV_MARK(A, r, j)                                                           \
    do {                                                                           \
        if (threadIdx.x % 32 == 0) (A).timing[(size_t)(r) * NTIME + (j)] = global_ns(); \
    } while (0)
#else
#define SV_MARK(A, r, j) \
    do {                 \
    } while (0)
#endif

// Appends this lane's tokens of segment seg whose key reaches tkey to the candidate buffer
// (warp-aggregated; entries beyond CAP are counted but not stored).
__device__ __forceinline__ void append_candidates(RowCtx &S, unsigned long long *cand, int seg, const float v[8],
                                                  uint32_t tkey, int V) {
    const int lane = lane_id();
    int c = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        int idx = seg * SEG + lane * 8 + j;
        c += (idx < V && fkey(v[j]) >= tkey) ? 1 : 0;
    }
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int base = 0;
    if (lane == 0 && total) base = atomicAdd(&S.ncand, total);
    base = __shfl_sync(0xffffffffu, base, 0);
    int pos = base + incl - c;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        int idx = seg * SEG + lane * 8 + j;
        uint32_t key = fkey(v[j]);
        if (idx < V && key >= tkey) {
            if (pos < CAP) cand[pos] = ((unsigned long long)key << 32) | (uint32_t)(~(uint32_t)idx);
            pos++;
        }
    }
}

// Appends this lane's tokens of segment seg whose value is above -inf (the caller masks the
// rest with -inf) to the candidate buffer; as append_candidates.
__device__ __forceinline__ void append_candidates_if(RowCtx &S, unsigned long long *cand, int seg, const float v[8],
                                                     int V) {
    const int lane = lane_id();
    int c = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) c += (v[j] > -INFINITY) ? 1 : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int base = 0;
    if (lane == 0 && total) base = atomicAdd(&S.ncand, total);
    base = __shfl_sync(0xffffffffu, base, 0);
    int pos = base + incl - c;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const int idx = seg * SEG + lane * 8 + j;
        if (v[j] > -INFINITY) {
            if (pos < CAP) cand[pos] = ((unsigned long long)fkey(v[j]) << 32) | (uint32_t)(~(uint32_t)idx);
            pos++;
        }
    }
    (void)V;
}

// One warp: top-k cut, top-p cut and kept mass over n <= WCAP candidates sorted by value
// (descending), 8 per lane.  Writes S.n2 (kept count), S.zk (kept mass), S.cutkey.
__device__ __forceinline__ void warp_cut(RowCtx &S, const unsigned long long *srt, int n, int K, float m, float s,
                                         bool topp, float P) {
    const int lane = lane_id(), base = lane * 8;
    const int kk = min(K, n);
    const uint32_t kkey = (uint32_t)(srt[kk - 1] >> 32);
    uint32_t key[8];
    int c1 = 0;
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const int idx = base + t;
        key[t] = idx < n ? (uint32_t)(srt[idx] >> 32) : 0u;
        c1 += (idx < n && key[t] >= kkey) ? 1 : 0;
    }
    const int n1 = warp_sum_i(c1);
    float pre[8], loc = 0.f;
#pragma unroll
    for (int t = 0; t < 8; t++) {
        loc += (base + t < n1) ? weight(key2f(key[t]), m, s) : 0.f;
        pre[t] = loc;
    }
    float Z1;
    const float ex = warp_excl_scan(loc, Z1);
#pragma unroll
    for (int t = 0; t < 8; t++) pre[t] += ex;
    int n2 = n1;
    if (topp) {
        // a value level is cut when the mass strictly above it reaches P * Z1
        const float PZ = __fmul_rn(P, Z1);
        int cut = 0x7fffffff;
        uint32_t prevkey = base > 0 ? (uint32_t)(srt[base - 1] >> 32) : 0u;
        float prevpre = ex;
#pragma unroll
        for (int t = 0; t < 8; t++) {
            const int idx = base + t;
            if (idx > 0 && idx < n1 && key[t] != prevkey && prevpre >= PZ) cut = min(cut, idx);
            prevkey = key[t];
            prevpre = pre[t];
        }
        cut = warp_min_i(cut);
        if (cut != 0x7fffffff) n2 = cut;
    }
    float zsel = 0.f;
#pragma unroll
    for (int t = 0; t < 8; t++)
        if (base + t == n2 - 1) zsel = pre[t];
    const float Z = __shfl_sync(0xffffffffu, zsel, (n2 - 1) >> 3);
    if (lane == 0) {
        S.n2 = n2;
        S.zk = Z;
        S.cutkey = (uint32_t)(srt[n2 - 1] >> 32);
    }
}

// One warp: the residual draw of a LIST row should its draft be rejected -- r = max(0, p - q)
// over the kept list (p is zero elsewhere, so r is too), q gathered from the draft row; an
// empty residual falls back to p.  ltok/lw: the list in token order (n <= WCAP); lq, when
// given, holds q at those tokens (else q is gathered from qrow).
__device__ __forceinline__ int warp_list_residual(const int *ltok, const float *lw, int n, float invZ,
                                                  const float *qrow, float u, const float *lq = nullptr) {
    const int lane = lane_id();
    float pw[8], rw[8];
    int tk[8];
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const int idx = lane * 8 + t;
        tk[t] = idx < n ? ltok[idx] : -1;
        pw[t] = idx < n ? __fmul_rn(lw[idx], invZ) : 0.f;
    }
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const float q = tk[t] >= 0 ? (lq ? lq[lane * 8 + t] : __ldg(qrow + tk[t])) : 0.f;
        rw[t] = tk[t] >= 0 ? fmaxf(__fsub_rn(pw[t], q), 0.f) : 0.f;
    }
    int j = warp_draw8(rw, n, u);
    if (j < 0) j = warp_draw8(pw, n, u);
    return j >= 0 ? ltok[j] : -1;
}

// Appends j to list[] for each lane where `take` holds (one atomic per warp); the whole warp
// must call it.
__device__ __forceinline__ void warp_append(int *list, int *count, bool take, int j) {
    const unsigned bal = __ballot_sync(0xffffffffu, take);
    if (!bal) return;
    const int lane = lane_id();
    int base = 0;
    if (lane == 0) base = atomicAdd(count, __popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (take) list[base + __popc(bal & ((1u << lane) - 1u))] = j;
}

// Top-k rows, up to 8 segment maxima per thread: in one pass over the maxima, the row max
// (S.m), a lower bound on the need-th largest maximum to 16 bits (two 8-bit radix rounds with
// the keys held in registers) and the candidate segments -- those whose max reaches the bound --
// split into single-candidate (X.segY, count S.n2) and re-read (X.segX, count S.nsel) lists.
// Returns the bound (0 when n < need: every segment is a candidate).  Six group barriers.
template <class G>
__device__ uint32_t top_prepare(const G &g, RowCtx &S, const Scratch &X, const SegStats &o, int n, int need) {
    constexpr int PT = 8;
    static_assert(G::kThreads * PT >= 1024, "top_prepare covers up to 1024 segments");
    const float *vals = o.mx;
    uint32_t *cnt = X.hcnt, *cnt1 = X.hcnt + 256;
    uint32_t key[PT];
    float mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < PT; t++) {
        const int j = g.t + t * G::kThreads;
        const float v = j < n ? vals[j] : -INFINITY;
        mx = fmaxf(mx, v);
        key[t] = j < n ? fkey(v) : 0u;
    }
    mx = warp_max(mx);
    for (int d = g.t; d < 512; d += G::kThreads) cnt[d] = 0;
    if (g.lane() == 0) S.redf[g.warp()] = mx;
    if (g.t == 0) {
        S.nsel = 0;
        S.ncand = 0;
        S.n2 = 0;
    }
    g.sync();
    const bool go = n >= need;
    if (go) {
#pragma unroll
        for (int t = 0; t < PT; t++)
            if (g.t + t * G::kThreads < n) atomicAdd(&cnt[key[t] >> 24], 1u);
    }
    g.sync();
    if (g.warp() == 0) {
        float m = S.redf[0];
        for (int w = 1; w < G::kWarps; w++) m = fmaxf(m, S.redf[w]);
        if (go) find_count_bin(S, cnt, 256, need);
        if (g.lane() == 0) S.m = m;
    }
    g.sync();
    uint32_t tkey = 0u;
    if (go) {
        const uint32_t d0 = (uint32_t)S.sel_digit;
        const long long nd = need - S.sel_below;
#pragma unroll
        for (int t = 0; t < PT; t++)
            if (g.t + t * G::kThreads < n && (key[t] >> 24) == d0) atomicAdd(&cnt1[(key[t] >> 16) & 255u], 1u);
        g.sync();
        if (g.warp() == 0) find_count_bin(S, cnt1, 256, nd);
        g.sync();
        tkey = (d0 << 24) | ((uint32_t)S.sel_digit << 16);
    }
    int *segl = reinterpret_cast<int *>(X.segX);
    int *single = reinterpret_cast<int *>(X.segY);
#pragma unroll
    for (int t = 0; t < PT; t++) {
        const int j = g.t + t * G::kThreads;
        const bool cand = j < n && key[t] >= tkey;
        const bool one = cand && fkey(o.b[j]) < tkey;
        warp_append(single, &S.n2, one, j);
        warp_append(segl, &S.nsel, cand && !one, j);
    }
    g.sync();
    return tkey;
}

// Appends the elements at `base` (8 raw values of one lane, penalties applied) whose key
// reaches tkey to the candidate buffer, one thread per lane-run and one atomic per warp; base
// < 0 contributes nothing.  Returns this thread's count.  The whole warp must call it.
template <typename E>
__device__ __forceinline__ int lane_candidates(RowCtx &S, unsigned long long *cand, const Raw8<E> &raw, int base,
                                               int V, uint32_t tkey) {
    const int lane = lane_id();
    float v[8];
    unpack8(raw, v);
    if (base >= 0) pen_lane8(S, base, v);
    int c = 0;
#pragma unroll
    for (int t = 0; t < 8; t++) c += (base >= 0 && base + t < V && fkey(v[t]) >= tkey) ? 1 : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int pos = 0;
    if (lane == 0 && total) pos = atomicAdd(&S.ncand, total);
    pos = __shfl_sync(0xffffffffu, pos, 0) + incl - c;
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const uint32_t key = fkey(v[t]);
        if (base >= 0 && base + t < V && key >= tkey) {
            if (pos < CAP) cand[pos] = ((unsigned long long)key << 32) | (uint32_t)(~(uint32_t)(base + t));
            pos++;
        }
    }
    return c;
}

// Kept set of a sampled row from the top-k candidates.  Returns false on candidate overflow.
template <typename E, bool VEC, class G>
__device__ bool kept_from_candidates(const G &g, const Args &A, RowCtx &S, const Scratch &X, const E *row,
                                     const SegStats &o, RowStat &st, bool want_bonus) {
    const int warp = g.warp(), lane = g.lane();
    const int V = A.V, nseg = A.nseg, K = S.K, tix = S.tix;
    (void)tix;
    const float m = S.m, s = S.s;
    const float *segA = o.mx;
    // lower bound on the K-th largest token: the K-th largest segment maximum, to 16 bits
    SV_MARK(A, tix, 16);
    // (for up to 8 maxima per thread select_row built the bound and the lists already)
    const bool prepped = S.prepped;
    uint32_t tkey = S.cutkey;
    if (!prepped) tkey = nseg >= K ? select_bound16(g, S, segA, nseg, K, X.hcnt, o.hist) : 0u;
    SV_MARK(A, tix, 17);
    // Segments whose max reaches the bound.  When a segment's second value is below it, its
    // max is its only candidate and the lane holding it is known: one 16-byte load finds the
    // token.  Segments with two or more candidates are re-read whole.  Lists are compacted
    // with warp ballots; both kinds of load go out before any is consumed.
    int *segl = reinterpret_cast<int *>(X.segX);
    int *single = reinterpret_cast<int *>(X.segY);
    if (!prepped) {
        if (g.t == 0) {
            S.nsel = 0;
            S.ncand = 0;
            S.n2 = 0;
        }
        g.sync();
        for (int j0 = warp * 32; j0 < nseg; j0 += G::kThreads) {
            const int j = j0 + lane;
            const bool cand = j < nseg && fkey(segA[j]) >= tkey;
            const bool one = cand && fkey(o.b[j]) < tkey;
            warp_append(single, &S.n2, one, j);
            warp_append(segl, &S.nsel, cand && !one, j);
        }
        g.sync();
    }
    const int nsingle = S.n2, nmulti = S.nsel;
#ifdef SV_TIMING
    if (g.t == 0) {
        A.timing[(size_t)tix * NTIME + 13] = (unsigned long long)nsingle;
        A.timing[(size_t)tix * NTIME + 14] = (unsigned long long)nmulti;
    }
#endif
    SV_MARK(A, tix, 18);
    constexpr int U = sizeof(E) == 2 ? 2 : 1;
    // first round: one single per thread and U multi segments per warp in flight together
    Raw8<E> sraw;
    int sj = -1;
    if (g.t < nsingle) {
        sj = single[g.t];
        sraw = load_raw8<VEC>(row, sj * SEG + o.lane[sj] * 8, V);
    }
    Raw8<E> raw[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
        const int j = warp + u * G::kWarps;
        if (j < nmulti) raw[u] = load_raw8<VEC>(row, segl[j] * SEG + lane * 8, V);
    }
    for (int jj0 = 0; jj0 < nsingle; jj0 += G::kThreads) {
        if (jj0 > 0) {
            sj = jj0 + g.t < nsingle ? single[jj0 + g.t] : -1;
            if (sj >= 0) sraw = load_raw8<VEC>(row, sj * SEG + o.lane[sj] * 8, V);
        }
        // every element of lane `at` that reaches the bound is a candidate (the segment's max
        // among them); the rest of the segment lies below the bound
        int found = 0;
        if (sj >= 0) found = lane_candidates(S, X.cand, sraw, sj * SEG + o.lane[sj] * 8, V, tkey);
        else lane_candidates(S, X.cand, sraw, -1, V, tkey);
        // a single with no element at the bound (cannot happen with consistent statistics) is
        // appended to the multi list, after the segments already in flight
        warp_append(segl, &S.nsel, sj >= 0 && found == 0, sj);
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
        const int j = warp + u * G::kWarps;
        if (j < nmulti) {
            const int seg = segl[j];
            float v[8];
            unpack8(raw[u], v);
            patch_seg(S, seg * SEG, v);
            append_candidates(S, X.cand, seg, v, tkey, V);
        }
    }
    g.sync();
    // further rounds: multi segments beyond the first U per warp (and any fallbacks)
    const int nsel = S.nsel;
    for (int j0 = warp + U * G::kWarps; j0 < nsel; j0 += G::kWarps * U) {
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int j = j0 + u * G::kWarps;
            if (j < nsel) raw[u] = load_raw8<VEC>(row, segl[j] * SEG + lane * 8, V);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int j = j0 + u * G::kWarps;
            if (j < nsel) {
                const int seg = segl[j];
                float v[8];
                unpack8(raw[u], v);
                patch_seg(S, seg * SEG, v);
                append_candidates(S, X.cand, seg, v, tkey, V);
            }
        }
    }
    // fallbacks appended after the first round's multi segments but inside it
    if (nsel > nmulti && nmulti < U * G::kWarps) {
        for (int j0 = nmulti + warp; j0 < min(nsel, U * G::kWarps); j0 += G::kWarps) {
            const int seg = segl[j0];
            float v[8];
            seg_values<E, VEC>(S, row, V, seg, v);
            append_candidates(S, X.cand, seg, v, tkey, V);
        }
    }
    g.sync();
    const int n = S.ncand;
#ifdef SV_TIMING
    if (g.t == 0) A.timing[(size_t)tix * NTIME + 15] = (unsigned long long)n;
#endif
    SV_MARK(A, tix, 19);
    if (n > CAP || n < 1) return false;

    if (n <= WCAP) {
        // rank sort by (value desc, token asc): keys are distinct, so ranks are a permutation.
        // q of each candidate (the residual needs it on the kept list) is gathered meanwhile.
        unsigned long long *srt = X.sorted;
        const bool want_resid = S.i < S.k && !A.onehot;
        const float *qrow = A.q + (size_t)(S.d0 + S.i) * V;
        float *qs = X.aux2;           // q at sorted positions
        float *lq = X.aux2 + WCAP;    // q in token order
        for (int j = g.t; j < n; j += G::kThreads) {
            const unsigned long long c = X.cand[j];
            const float qv = want_resid ? __ldg(qrow + (int)(~(uint32_t)c)) : 0.f;
            int rk = 0;
            for (int i = 0; i < n; i++) rk += X.cand[i] > c ? 1 : 0;
            srt[rk] = c;
            qs[rk] = qv;
        }
        g.sync();
        SV_MARK(A, tix, 20);
        if (warp == 0) warp_cut(S, srt, n, K, m, s, S.topp_on, S.P);
        g.sync();
        SV_MARK(A, tix, 21);
        const int n2 = S.n2;
        const float Z = S.zk;
        st.Z = Z;
        st.invZ = __frcp_rn(Z);
        st.taukey = S.cutkey;
        st.tau = key2f(S.cutkey);
        st.kind = KIND_LIST;
        st.nlist = n2;
        // the kept set in token order (rank by token id), stored for the residual draw
        int *ltok = reinterpret_cast<int *>(X.cand);
        float *lw = reinterpret_cast<float *>(X.cand) + WCAP;
        for (int j = g.t; j < n2; j += G::kThreads) {
            const uint32_t tj = ~(uint32_t)srt[j];
            int rk = 0;
            for (int i = 0; i < n2; i++) rk += (~(uint32_t)srt[i]) < tj ? 1 : 0;
            ltok[rk] = (int)tj;
            lw[rk] = weight(key2f((uint32_t)(srt[j] >> 32)), m, s);
            lq[rk] = qs[j];
        }
        g.sync();
        SV_MARK(A, tix, 22);
        // warp 0: the extra-token draw (last row); warp 1 (or 0): the residual draw should the
        // row's draft be rejected, with q gathered on the kept list
        const int wres = G::kWarps > 1 ? 1 : 0;
        if (want_bonus && warp == 0) {
            const float u = S.u1;
            float w8[8];
#pragma unroll
            for (int t = 0; t < 8; t++) w8[t] = (lane * 8 + t < n2) ? lw[lane * 8 + t] : 0.f;
            const int j = warp_draw8(w8, n2, u);
            if (lane == 0) S.tok = j >= 0 ? ltok[j] : -1;
        }
        if (want_resid && warp == wres) {
            const int t = warp_list_residual(ltok, lw, n2, st.invZ, qrow, S.u1, lq);
            if (lane == 0) S.a = t;
        }
        g.sync();
        if (want_bonus) st.bonus = S.tok;
        if (want_resid) st.resid = S.a;
        SV_MARK(A, tix, 23);
        return true;
    }

    // larger candidate sets: group-wide bitonic sort and scans
    const int np = pow2_at_least(n);
    for (int j = n + g.t; j < np; j += G::kThreads) X.cand[j] = 0ull;
    g.sync();
    g_sort_desc(g, X.cand, np);
    const int kk = min(K, n);
    const uint32_t kkey = (uint32_t)(X.cand[kk - 1] >> 32);
    int c1 = 0;
    for (int j = g.t; j < n; j += G::kThreads) c1 += ((uint32_t)(X.cand[j] >> 32) >= kkey) ? 1 : 0;
    const int n1 = g_sum_i(g, c1, S.redi);
    for (int j = g.t; j < n1; j += G::kThreads) X.aux[j] = weight(key2f((uint32_t)(X.cand[j] >> 32)), m, s);
    g.sync();
    for (int j = g.t; j < n1; j += G::kThreads) X.aux2[j] = X.aux[j];
    g.sync();
    g_scan_incl(g, X.aux2, n1, S.redf);
    int n2 = n1;
    if (S.topp_on) {
        const float PZ = __fmul_rn(S.P, X.aux2[n1 - 1]);
        int cut = 0x7fffffff;
        for (int j = g.t; j < n1; j += G::kThreads) {
            if (j > 0 && (uint32_t)(X.cand[j] >> 32) != (uint32_t)(X.cand[j - 1] >> 32) && X.aux2[j - 1] >= PZ)
                cut = min(cut, j);
        }
        cut = g_min_i(g, cut, S.redi);
        if (cut != 0x7fffffff) n2 = cut;
    }
    const float Z = X.aux2[n2 - 1];
    const uint32_t taukey = (uint32_t)(X.cand[n2 - 1] >> 32);
    st.Z = Z;
    st.invZ = __frcp_rn(Z);
    st.taukey = taukey;
    st.tau = key2f(taukey);
    st.kind = n2 <= LCAP ? KIND_LIST : KIND_THRESH;
    st.nlist = n2 <= LCAP ? n2 : 0;
    g.sync();
    if (n2 <= LCAP || want_bonus) {
        const int np2 = pow2_at_least(n2);
        for (int j = g.t; j < np2; j += G::kThreads) {
            unsigned long long c = X.cand[j];
            X.cand[j] = j < n2 ? ((c << 32) | (c >> 32)) : 0ull;
        }
        g.sync();
        g_sort_desc(g, X.cand, np2);
        for (int j = g.t; j < n2; j += G::kThreads) X.aux[j] = weight(key2f((uint32_t)X.cand[j]), m, s);
        g.sync();
        if (want_bonus) {
            const float u = S.u1;
            int j = draw_small(g, X.aux, X.aux2, n2, u, S);
            st.bonus = j >= 0 ? (int32_t)(~(uint32_t)(X.cand[j] >> 32)) : -1;
        }
        if (n2 <= LCAP && S.i < S.k && !A.onehot) {
            // the residual draw should the row's draft be rejected (as in the small-set path)
            int *ltok = reinterpret_cast<int *>(X.aux2) + CAP / 2;
            for (int j = g.t; j < n2; j += G::kThreads) ltok[j] = (int)(~(uint32_t)(X.cand[j] >> 32));
            g.sync();
            if (warp == 0) {
                const float u = S.u1;
                const float *qrow = A.q + (size_t)(S.d0 + S.i) * V;
                const int t = warp_list_residual(ltok, X.aux, n2, st.invZ, qrow, u);
                if (lane == 0) S.a = t;
            }
            g.sync();
            st.resid = S.a;
        }
    }
    g.sync();
    return true;
}

// Mass bin of a token from a = (z - m) s, the log2 of its weight (<= 0): bins of 1/bpu of a
// unit of log2 weight from the row max down, the last bin collecting everything lower.  The
// bin is monotone in z: a token of a lower bin is strictly more likely than one of a higher.
__device__ __forceinline__ int mass_bin(float a, float bpu, int nb) {
    const float t = __fmul_rn(-a, bpu);
    return t >= (float)(nb - 1) ? nb - 1 : (int)t;
}

// Fixed-point (2^-40) weight of a token from a = (z - m) s: the value weight() rounds to.
__device__ __forceinline__ unsigned long long fixed_weight(float a) {
    return __float2ull_rz(__fmul_rn(ex2(a), (float)FIXED_ONE));
}

// Exclusive prefix sums of v[0..n) (n <= G::kThreads * 4), 64-bit and exact, in place.
template <class G>
__device__ __forceinline__ void g_scan_u64_excl(const G &g, unsigned long long *v, int n, RowCtx &S) {
    const int lane = g.lane(), warp = g.warp();
    const int per = (n + G::kThreads - 1) / G::kThreads;
    const int lo = min(n, g.t * per), hi = min(n, lo + per);
    unsigned long long t = 0;
    for (int j = lo; j < hi; j++) t += v[j];
    unsigned long long incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    unsigned long long *red = reinterpret_cast<unsigned long long *>(S.redd);
    if (lane == 31) red[warp] = incl;
    g.sync();
    unsigned long long run = incl - t;
    for (int w = 0; w < warp; w++) run += red[w];
    for (int j = lo; j < hi; j++) {
        const unsigned long long x = v[j];
        v[j] = run;
        run += x;
    }
    g.sync();
}

// Top-p rows without top-k (FreeToken PR #836, "Design": keep the tokens while the mass
// strictly above them is below top_p).  Two passes over the row instead of a radix select:
//  1. mass bins relative to the row max (64 per unit of log2 weight over 16 units, or fewer
//     when the group's scratch is small), with fixed-point weights summed exactly -- the bin
//     where the running mass from the top reaches P * (total) holds the cut;
//  2. that bin's tokens, sorted: the cut falls between two of its value levels, and the kept
//     mass (the normaliser Z) is the exact fixed-point sum above the cut.
// A draw from the row (want_bonus) adds the weight pass and the draw of kept_by_select.
// Returns false, with nothing written to st, when the cut's bin holds more than CAP tokens or
// the scratch holds fewer than 256 bins; the caller then takes the radix select (which
// rewrites every scratch area it uses).
template <typename E, bool VEC, class G>
__device__ bool kept_by_mass_bins(const G &g, const Args &A, RowCtx &S, const Scratch &X, const E *row, RowStat &st,
                                  bool want_bonus) {
    const int V = A.V, nseg = A.nseg, lane = g.lane();
    const float m = S.m, s = S.s;
    const int lbits = V > 1 ? __clz(V - 1) : 31;        // V tokens of < 2^lbits fit one 32-bit limb
    const int nl = (41 + lbits - 1) / lbits;            // limbs covering 2^40
    int nb = 1024;
    while (nb >= 256 && (size_t)nb * (nl + 1) * 4 > X.big_bytes) nb >>= 1;
    if (nb < 256) return false;
    const float bpu = (float)(nb / 16);
    uint32_t *cnt = reinterpret_cast<uint32_t *>(X.big);   // nb counts, then nl arrays of nb limbs
    uint32_t *limb = cnt + nb;
    const unsigned long long lmask = (1ull << lbits) - 1ull;
    g.sync();   // the row statistics in X.big are no longer read
    for (int d = g.t; d < nb * (nl + 1); d += G::kThreads) cnt[d] = 0u;
    g.sync();
    pass_segments<E, VEC, false, false, sizeof(E) == 2 ? 2 : 1>(
        g, S, row, nullptr, V, nseg, [&](int seg, const float *v, const float *) {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if (seg * SEG + lane * 8 + j < V) {
                    const float a = __fmul_rn(__fsub_rn(v[j], m), s);
                    const int bin = mass_bin(a, bpu, nb);
                    const unsigned long long f = fixed_weight(a);
                    atomicAdd(&cnt[bin], 1u);
#pragma unroll
                    for (int l = 0; l < 4; l++) {
                        const uint32_t part = (uint32_t)((f >> (lbits * l)) & lmask);
                        if (l < nl && part) atomicAdd(&limb[l * nb + bin], part);
                    }
                }
            }
        });
    g.sync();
    // each thread totals a run of bins; the run holding the cut then finds its bin
    const int per = nb / G::kThreads;
    unsigned long long tot = 0;
    for (int d = g.t * per; d < g.t * per + per; d++)
        for (int l = 0; l < nl; l++) tot += (unsigned long long)limb[l * nb + d] << (lbits * l);
    unsigned long long incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    unsigned long long *red = reinterpret_cast<unsigned long long *>(S.redd);
    if (lane == 31) red[g.warp()] = incl;
    g.sync();
    unsigned long long T = 0, run = incl - tot;
    for (int w = 0; w < G::kWarps; w++) {
        if (w < g.warp()) run += red[w];
        T += red[w];
    }
    const double PT = (double)S.P * (double)T;
    if (g.t == 0) S.ncand = -1;
    g.sync();
    if ((double)run < PT && (double)(run + tot) >= PT) {
        // this run holds the first bin whose running mass reaches P * T
        for (int d = g.t * per; d < g.t * per + per; d++) {
            unsigned long long md = 0;
            for (int l = 0; l < nl; l++) md += (unsigned long long)limb[l * nb + d] << (lbits * l);
            if ((double)(run + md) >= PT) {
                S.sel_digit = d;
                S.sel_mass = run;          // the mass of every bin above d
                S.nsel = (int)cnt[d];      // tokens in bin d
                S.ncand = 0;
                break;
            }
            run += md;
        }
    }
    g.sync();
    if (S.ncand < 0 || S.nsel > CAP) return false;
    const int bstar = S.sel_digit;
    const unsigned long long above = S.sel_mass;
    g.sync();   // the bins are dead: the candidates take their place
    // 2. the tokens of the cut's bin
    pass_segments<E, VEC, false, false, sizeof(E) == 2 ? 2 : 1>(
        g, S, row, nullptr, V, nseg, [&](int seg, const float *v, const float *) {
            float vv[8];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const bool in = seg * SEG + lane * 8 + j < V &&
                                mass_bin(__fmul_rn(__fsub_rn(v[j], m), s), bpu, nb) == bstar;
                vv[j] = in ? v[j] : -INFINITY;
            }
            append_candidates_if(S, X.cand, seg, vv, V);
        });
    g.sync();
    const int n = S.ncand;
    if (n > CAP || n < 1) return false;     // too many tokens share the cut's bin
    const int np2 = pow2_at_least(n);
    for (int j = n + g.t; j < np2; j += G::kThreads) X.cand[j] = 0ull;
    g.sync();
    g_sort_desc(g, X.cand, np2);
    // fixed-point weights of the sorted candidates, then their exclusive running sums
    unsigned long long *fw = reinterpret_cast<unsigned long long *>(X.cand + CAP);
    for (int j = g.t; j < n; j += G::kThreads)
        fw[j] = fixed_weight(__fmul_rn(__fsub_rn(key2f((uint32_t)(X.cand[j] >> 32)), m), s));
    g.sync();
    unsigned long long fn = 0;
    if (g.t == 0) fn = fw[n - 1];
    g_scan_u64_excl(g, fw, n, S);
    // the first value level (after the first) whose mass strictly above reaches P * T is cut
    int cut = 0x7fffffff;
    for (int j = g.t; j < n; j += G::kThreads)
        if (j > 0 && (uint32_t)(X.cand[j] >> 32) != (uint32_t)(X.cand[j - 1] >> 32) && (double)(above + fw[j]) >= PT)
            cut = min(cut, j);
    cut = g_min_i(g, cut, S.redi);
    const int n2 = cut != 0x7fffffff ? cut : n;
    if (g.t == 0) {
        const unsigned long long zf = above + (n2 < n ? fw[n2] : fw[n - 1] + fn);
        S.sel_mass = zf;
        S.cutkey = (uint32_t)(X.cand[n2 - 1] >> 32);
    }
    g.sync();
    const float Z = (float)((double)S.sel_mass / FIXED_ONE);
    const uint32_t taukey = S.cutkey;
    st.Z = Z;
    st.invZ = __frcp_rn(Z);
    st.taukey = taukey;
    st.tau = key2f(taukey);
    st.kind = KIND_THRESH;
    st.nlist = 0;
    if (want_bonus) {
        WKept wk{m, s, taukey};
        seg_sums<E, VEC, false>(g, S, row, nullptr, V, nseg, X.segY, wk, nullptr, wk);
        st.bonus = draw_by_segments<E, VEC, false>(g, S, row, nullptr, V, nseg, X.segY, S.u1, wk);
    }
    return true;
}

// Kept set by radix select over the whole row (any top-k / top-p).
template <typename E, bool VEC, class G>
__device__ void kept_by_select(const G &g, const Args &A, RowCtx &S, const Scratch &X, const E *row, RowStat &st,
                               bool want_bonus) {
    const int V = A.V, nseg = A.nseg;
    const float m = S.m, s = S.s;
    if (S.topp_on && !S.topk_on && kept_by_mass_bins<E, VEC>(g, A, S, X, row, st, want_bonus)) return;
    uint32_t key_lo = 0;
    if (S.topk_on) key_lo = select_kth_row<E, VEC>(g, S, row, V, nseg, S.K, X.hcnt);
    if (S.topp_on) key_lo = select_mass_row<E, VEC>(g, S, row, V, nseg, key_lo, m, s, S.P, X.hmass, X.hlimb);
    WKept wk{m, s, key_lo};
    seg_sums<E, VEC, false>(g, S, row, nullptr, V, nseg, X.segY, wk, nullptr, wk);
    float part = 0.f;
    for (int j = g.t; j < nseg; j += G::kThreads) part += X.segY[j];
    const float Z = g_sum(g, part, S.redf);
    st.Z = Z;
    st.invZ = __frcp_rn(Z);
    st.taukey = key_lo;
    st.tau = key_lo ? key2f(key_lo) : -INFINITY;
    st.kind = KIND_THRESH;
    st.nlist = 0;
    if (want_bonus) {
        const float u = S.u1;
        st.bonus = draw_by_segments<E, VEC, false>(g, S, row, nullptr, V, nseg, X.segY, u, wk);
    }
}

// The row's statistics, kept set, draws and draft gathers from its per-segment maxima (segA)
// and weight sums (segB, for rows with no filter); writes the row's RowStat, kept list and
// (p, q) of its draft.  segA/segB are consumed.
template <typename E, bool VEC, class G>
__device__ void select_row(const G &g, const Args &A, RowCtx &S, const Scratch &X, const SegStats &o,
                           const unsigned long long *argkey = nullptr) {
    float *segA = o.mx, *segB = o.b;
    const int V = A.V, nseg = A.nseg, row_idx = S.r;
    const E *row = reinterpret_cast<const E *>(A.logits) + (size_t)row_idx * V;
    RowStat st;
    st.m = 0.f; st.s = 0.f; st.tau = -INFINITY; st.Z = 1.f; st.invZ = 1.f; st.taukey = 0;
    st.argmax = -1; st.bonus = -1; st.kind = KIND_SKIP; st.nlist = 0; st.resid = -1; st.pad1 = 0;
    const bool sampled = !S.greedy;
    // the row's own sample: the extra token of row k, or under the one-hot scheme every row's
    const bool want_bonus = sampled && (S.i == S.k || A.onehot);
    const float s = S.s;
    float m;
    if (!sampled && argkey) {
        // greedy row whose streamers folded (max, lowest position) into one key
        const unsigned long long key = __ldcg(argkey);
        const uint32_t idx = ~(uint32_t)key;
        m = key2f((uint32_t)(key >> 32));
        st.argmax = idx < (uint32_t)V ? (int)idx : 0;   // an all -inf row: token 0
    } else if (sampled && !S.need_sum && S.mode == MODE_TOP2 && nseg <= G::kThreads * 8) {
        // top-k rows: the row max, the candidates' bound and the candidate lists in one pass
        const uint32_t bound = top_prepare(g, S, X, o, nseg, S.K);
        m = S.m;
        g.sync();
        if (g.t == 0) {
            S.cutkey = bound;
            S.prepped = 1;
        }
    } else {
        if (g.t == 0) S.prepped = 0;
        float mx = -INFINITY;
        for (int j = g.t; j < nseg; j += G::kThreads) mx = fmaxf(mx, segA[j]);
        m = g_max(g, mx, S.redf);
    }
    if (g.t == 0) S.m = m;
    g.sync();
    st.m = m;
    st.s = s;

    if (!sampled && argkey) {
        st.kind = KIND_GREEDY;
    } else if (!sampled) {
        // greedy: lowest id of the maximum -- the first segment holding it, the lowest lane of
        // that segment holding it (recorded while streaming), then the first slot of the lane
        int first = 0x7fffffff;
        for (int j = g.t; j < nseg; j += G::kThreads)
            if (segA[j] == m) first = min(first, j);
        first = g_min_i(g, first, S.redi);
        if (g.t == 0) {
            int tok = first != 0x7fffffff ? find_in_lane<E, VEC>(S, row, V, first, o.lane[first], m) : -1;
            S.tok = tok >= 0 ? tok : 0;
        }
        g.sync();
        st.argmax = S.tok;
        st.kind = KIND_GREEDY;
    } else if (S.need_sum) {
        // no filter: Z from the segment sums rescaled to the row max (fixed order)
        float part = 0.f;
        for (int j = g.t; j < nseg; j += G::kThreads) {
            float w = segA[j] > -INFINITY ? __fmul_rn(segB[j], weight(segA[j], m, s)) : 0.f;
            segB[j] = w;
            part += w;
        }
        const float Z = g_sum(g, part, S.redf);
        st.Z = Z;
        st.invZ = __frcp_rn(Z);
        st.kind = KIND_FULL;
        if (want_bonus) {
            const float u = S.u1;
            WKept wk{m, s, 0u};
            st.bonus = draw_by_segments<E, VEC, false>(g, S, row, nullptr, V, nseg, segB, u, wk);
        }
    } else {
        bool done = false;
        if (S.mode == MODE_TOP2) done = kept_from_candidates<E, VEC>(g, A, S, X, row, o, st, want_bonus);
        if (!done) kept_by_select<E, VEC>(g, A, S, X, row, st, want_bonus);
    }
    SV_MARK(A, S.tix, 3);

    // the draft of this row: p(x_i) and q(x_i) (prefetched while the row streamed)
    if (g.t == 0 && S.i < S.k) {
        const int x = S.xtok;
        float p = 0.f, q = 0.f;
        if (!sampled) {
            p = NAN;
            q = NAN;
        } else if (x >= 0 && x < V) {
            const float z = S.zx;
            p = fkey(z) >= st.taukey ? __fmul_rn(weight(z, m, s), st.invZ) : 0.f;
            q = S.qx;
        }
        const size_t d = (size_t)(S.d0 + S.i);
        A.pq[d * 2] = p;
        A.pq[d * 2 + 1] = q;
        if (A.out_pq) {
            A.out_pq[d * 2] = p;
            A.out_pq[d * 2 + 1] = q;
        }
    }
    if (g.t == 0) A.stats[row_idx] = st;
}

// A RowStat written by another CTA, read through L2.
__device__ __forceinline__ RowStat load_stat(const RowStat *p) {
    const int4 *q = reinterpret_cast<const int4 *>(p);
    const int4 a = __ldcg(q), b = __ldcg(q + 1), c = __ldcg(q + 2);
    RowStat st;
    st.m = __int_as_float(a.x);
    st.s = __int_as_float(a.y);
    st.tau = __int_as_float(a.z);
    st.Z = __int_as_float(a.w);
    st.invZ = __int_as_float(b.x);
    st.taukey = (uint32_t)b.y;
    st.argmax = b.z;
    st.bonus = b.w;
    st.kind = c.x;
    st.nlist = c.y;
    st.resid = c.z;
    st.pad1 = c.w;
    return st;
}

// Accept test of one draft: accept with probability min(1, p/q), i.e. iff u < min(1, p/q);
// q == 0 < p accepts and p == 0 rejects.
__device__ __forceinline__ bool accept_test(float p, float q, float u) {
    if (!(p > 0.f)) return false;
    if (q == 0.f) return true;
    const float ratio = __fdiv_rn(p, q);
    return u < (ratio < 1.f ? ratio : 1.f);
}

// Request phase, run by the group that completed the request's last row: validate, find the
// first rejection (one lane per draft, ballot), pick the final token, write the outputs.
// Under the one-hot scheme a draft is rejected when it differs from its row's own sample, and
// the final token is the stopping row's sample.
// `lim`: the last row whose statistics exist (the lazy scheme finalises a request that stops at
// row 0 before its other rows are read); rows past it are never the stopping row.
// QUEUE: a whole-row residual is queued for the residual kernel instead of drawn here.
template <typename E, bool VEC, bool QVEC, bool QUEUE = false, class G>
__device__ void finalize(const G &g, const Args &A, RowCtx &S, const Scratch &X, int lim = 0x7fffffff) {
    const int b = S.b, k = S.k, r0 = S.r0, d0 = S.d0, V = A.V;
#ifdef SV_TIMING
    if (g.t == 0 && b >= 0 && b < A.B) atomicAdd(A.timing + (size_t)(6 * A.R + b) * NTIME, 1ull);
#endif
    int *xs = reinterpret_cast<int *>(X.cand);   // the request's draft tokens, for the outputs
    if (g.warp() == 0) {
        // one round of loads: every row's statistics, draft, (p, q) and uniforms at once; the
        // final token is then taken from the lane that holds the stopping row
        const int lane = g.lane();
        int status = S.status;
        int a = -1, tok = -1, need = 0;
        if (status == 0) {
            const bool greedy = S.greedy;
            bool badtok = false, baduni = false, found = false;
            a = k;
            for (int i0 = 0; i0 <= k; i0 += 32) {
                const int i = i0 + lane;
                bool rej = false;
                int kind = KIND_SKIP, argm = -1, bonus = -1, resid = -1;
                if (i <= k && i <= lim) {
                    const RowStat *st = A.stats + r0 + i;
                    kind = __ldcg(&st->kind);
                    argm = __ldcg(&st->argmax);
                    bonus = __ldcg(&st->bonus);
                    resid = __ldcg(&st->resid);
                }
                if (i < k) {
                    const int x = __ldg(A.tokens + d0 + i);
                    xs[i] = x;
                    if (x < 0 || x >= V) badtok = true;
                    if (greedy) {
                        rej = x != argm;
                    } else if (A.onehot) {
                        rej = x != bonus;   // the row's own sample
                    } else {
                        const float p = __ldcg(A.pq + (size_t)(d0 + i) * 2);
                        const float q = __ldcg(A.pq + (size_t)(d0 + i) * 2 + 1);
                        rej = !accept_test(p, q, __ldg(A.uni + (size_t)(r0 + i) * 2));
                    }
                }
                if (!greedy && i <= k) {
                    // the one-hot scheme reads only the draw slot
                    const float u0 = A.onehot ? 0.f : __ldg(A.uni + (size_t)(r0 + i) * 2);
                    const float u1 = __ldg(A.uni + (size_t)(r0 + i) * 2 + 1);
                    if (!(u0 >= 0.f && u0 < 1.f) || !(u1 >= 0.f && u1 < 1.f)) baduni = true;
                }
                const unsigned msk = __ballot_sync(0xffffffffu, rej);
                // the stopping row: the first rejection, else row k (in the last chunk)
                int stop = -1;
                if (!found && msk) stop = __ffs(msk) - 1;
                else if (!found && i0 + 32 > k) stop = k - i0;
                if (stop >= 0) {
                    found = true;
                    a = i0 + stop;
                    const int kind_a = __shfl_sync(0xffffffffu, kind, stop);
                    const int argm_a = __shfl_sync(0xffffffffu, argm, stop);
                    const int bonus_a = __shfl_sync(0xffffffffu, bonus, stop);
                    const int resid_a = __shfl_sync(0xffffffffu, resid, stop);
                    if (greedy) tok = argm_a;
                    else if (a == k || A.onehot) tok = bonus_a;
                    else if (kind_a == KIND_LIST) tok = resid_a;   // drawn speculatively with the row
                    else need = 1;
                }
            }
            badtok = __any_sync(0xffffffffu, badtok);
            baduni = __any_sync(0xffffffffu, baduni);
            if (badtok) status = 2;
            else if (baduni) status = 5;
            if (status != 0) {
                a = -1;
                tok = -1;
                need = 0;
            }
        }
        if (lane == 0) {
            if (status) record_error(A, status, b);
            S.a = a;
            S.tok = tok;
            S.need_resid = need;
        }
    }
    g.sync();
    if (QUEUE && S.need_resid) {
        // the whole-row residual is queued below, once the outputs are written
    } else if (S.need_resid) {
        // residual max(0, p - q) over a whole row (rows that keep too many tokens for a list)
        const int a = S.a;
        const RowStat st = load_stat(A.stats + r0 + a);
        const float *qrow = A.q + (size_t)(d0 + a) * V;
        const float u = __ldg(A.uni + (size_t)(r0 + a) * 2 + 1);
        if (g.warp() == 0) build_penalties(A, S, a);
        g.sync();
        const E *row = reinterpret_cast<const E *>(A.logits) + (size_t)(r0 + a) * V;
        WResid wr{st.m, st.s, st.invZ, st.taukey};
        WProb wp{st.m, st.s, st.invZ, st.taukey};
        seg_sums<E, VEC, QVEC>(g, S, row, qrow, V, A.nseg, X.segX, wr, X.segY, wp);
        int tok = draw_by_segments<E, VEC, QVEC>(g, S, row, qrow, V, A.nseg, X.segX, u, wr);
        if (tok < 0) tok = draw_by_segments<E, VEC, QVEC>(g, S, row, nullptr, V, A.nseg, X.segY, u, wp);
        if (g.t == 0) S.tok = tok;
        g.sync();
    }
    // outputs: accepted drafts, the final token, -1 padding
    const int a = S.a, kw = A.k_max + 1;
    for (int j = g.t; j < kw; j += G::kThreads) {
        int v = -1;
        if (a >= 0) v = j < a ? xs[j] : (j == a ? S.tok : -1);
        A.out_tok[(size_t)b * kw + j] = v;
    }
    if (g.t == 0) A.acc[b] = a;
    if (QUEUE && S.need_resid) {
        // The whole-row residual goes to the residual workers (or kernel), which draw the final
        // token into out_tokens[b][a] (-1 until then).  Queued after the outputs above, which
        // the barrier orders before the job's release: a worker's token is never overwritten.
        g.sync();
        if (g.t == 0) {
            const int jj = atomicAdd(A.hdr + 5, 1);
            st_release_u64(A.jobs + jj, ((unsigned long long)A.epoch << 32) | ((uint32_t)b << 7) | (uint32_t)a);
        }
    }
}

// Lazy scheme ("Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in
// Rust", "The Verification Algorithm": the loop returns at the first rejection, so the rows
// after it are never needed).  After a request's row 0: it stops there -- it is invalid, has
// no drafts, or row 0 rejects its draft -- and is finalised from that row alone; or it queues
// its rows 1..k for the second phase, having counted row 0 as arrived.  The whole group calls.
template <typename E, bool VEC, bool QVEC, class G>
__device__ void first_row_decision(const G &g, const Args &A, RowCtx &S, const Scratch &X) {
    g.sync();
    if (g.t == 0) {
        bool stop = S.status != 0 || S.k == 0 || !S.active;
        if (!stop) {
            const int x = __ldg(A.tokens + S.d0);
            if (x < 0 || x >= A.V) stop = true;   // (the finaliser reports the bad token)
            else if (S.greedy) stop = x != __ldcg(&A.stats[S.r].argmax);
            else if (A.onehot) stop = x != __ldcg(&A.stats[S.r].bonus);
            else stop = !accept_test(__ldcg(A.pq + (size_t)S.d0 * 2), __ldcg(A.pq + (size_t)S.d0 * 2 + 1),
                                     __ldg(A.uni + (size_t)S.r * 2));
        }
        S.last = stop ? 1 : 0;
        if (!stop) {
            const int pos = atomicAdd(A.hdr + 4, S.k);
            for (int i = 1; i <= S.k; i++) A.listb[pos + i - 1] = S.r0 + i;
            A.counters[S.b] = 1;
        } else if (A.out_pq && S.status == 0) {
            // drafts past the stopping row are never read: no (p, q) for them
            for (int i = 1; i < S.k; i++) {
                A.out_pq[(size_t)(S.d0 + i) * 2] = NAN;
                A.out_pq[(size_t)(S.d0 + i) * 2 + 1] = NAN;
            }
        }
    }
    g.sync();
    if (S.last) finalize<E, VEC, QVEC, true>(g, A, S, X, 0);
    g.sync();
}

// Writes -1 outputs for request b (no rows, or inconsistent row_offsets).
template <class G>
__device__ __forceinline__ void fail_request(const G &g, const Args &A, int b) {
    const int kw = A.k_max + 1;
    for (int j = g.t; j < kw; j += G::kThreads) A.out_tok[(size_t)b * kw + j] = -1;
    if (g.t == 0) {
        A.acc[b] = -1;
        record_error(A, 1, b);
    }
}

// Requests that own no rows (row_offsets[j] == row_offsets[j+1]) get -1 outputs from the first
// row of the nearest non-empty request before them (leading ones from the request of row 0).
template <class G>
__device__ __forceinline__ void fail_empty_requests(const G &g, const Args &A, const RowCtx &S) {
    if (!A.row_off || S.i != 0 || S.b < 0) return;
    if (S.r == 0)
        for (int j = S.b - 1; j >= 0; j--) fail_request(g, A, j);
    for (int j = S.b + 1; j < A.B && __ldg(A.row_off + j) == __ldg(A.row_off + j + 1); j++) fail_request(g, A, j);
}

// After a row: count it towards its request; the group that brings the count to the
// request's row count finalises it.  Every thread of the group must call this.
template <typename E, bool VEC, bool QVEC, bool LAZY = false, bool QUEUE = false, class G>
__device__ __forceinline__ void arrive_and_finalize(const G &g, const Args &A, RowCtx &S, const Scratch &X) {
    g.sync();
    if (g.t == 0) {
        // release this row's results, acquire the other rows' (the group's writes are ordered
        // before by the barrier above)
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(A.counters + S.b) : "memory");
        // every row of the request's slot counts, except under the lazy scheme's second phase,
        // which reads rows 1..k after the first phase counted row 0
        S.last = (old == (LAZY ? S.k : S.nrows - 1));
    }
    g.sync();
    if (S.last) {
        finalize<E, VEC, QVEC, QUEUE>(g, A, S, X);
#ifdef SV_TIMING
        if (g.t == 0) A.timing[(size_t)S.tix * NTIME + 7] = 1;
#endif
    }
    g.sync();
}

}  // namespace sv

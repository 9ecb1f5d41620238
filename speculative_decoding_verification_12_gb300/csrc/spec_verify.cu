// spec_verify.cu -- batched speculative-decoding verification for GB300 (sm_103a): the
// C-ABI entry points and the fused verify kernel.
//
// One CTA per target row streams the row once from HBM (128-bit loads, 8 tokens per lane,
// 256-token segments per warp step) and reduces it to per-segment maxima and weight sums.
// From those it builds the row's kept set:
//   - no filter: p = e / Z with Z from the segment sums (no second pass);
//   - top-k (k <= KCAP): the k-th largest segment maximum bounds the k-th largest token from
//     below, so only the segments whose maximum reaches it are re-read (from L2) to collect
//     candidates; the exact top-k and top-p cut is made on the sorted candidates in shared
//     memory;
//   - otherwise (top-p alone, large top-k, candidate overflow): radix select with 11-bit
//     digits over the row, counts for top-k and fixed-point masses for top-p.
// It then gathers p(x_i) and q(x_i) for the row's draft, and on a request's last row also
// draws the extra token.  The CTA that completes the last row of a request (arrival counter
// per request; no CTA ever waits on another) runs the first-rejection scan and, at a
// rejection, draws from max(0, p - q) of the rejected row: over the stored kept list when it
// is small, else in one pass over the row and its draft row.
//
// Method: "Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust"
// ("The Memory Bandwidth Wall and Speculative Math", "The Verification Algorithm",
// "Orchestrating the Inference Loop"); "Adding Speculative Decoding" ("Verification and
// sampling", table "The existing base"); FreeToken PR #836 ("Design").
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "../../include/spec_verify.h"
#include "sv_row.cuh"

namespace sv {

// Shared-memory carve-up of one CTA (dynamic part).
struct Dyn {
    float *segA, *segB, *segC;   // per-segment max / weight sums
    unsigned long long *cand;    // CAP keys: (order key << 32) | ~token, later (~token << 32) | key
    float *aux, *aux2;           // CAP floats each
    unsigned long long *sorted;  // WCAP keys (aliases aux/aux2)
    unsigned char *ring;         // NS x SB bytes of streamed row data (aliases cand/aux/aux2)
    uint32_t *hcnt;              // radix histogram (aliases cand/aux)
    unsigned long long *hmass;   // fixed-point mass histogram (aliases)
};

__host__ __device__ inline int nseg_pad(int nseg) { return (nseg + 31) & ~31; }   // keeps the ring 128-byte aligned
__host__ __device__ inline size_t dyn_bytes(int nseg) {
    return size_t(3) * nseg_pad(nseg) * 4 + size_t(CAP) * 8 + size_t(CAP) * 4 * 2;
}

__device__ __forceinline__ Dyn carve(unsigned char *base, int nseg) {
    Dyn d;
    const int np = nseg_pad(nseg);
    d.segA = reinterpret_cast<float *>(base);
    d.segB = d.segA + np;
    d.segC = d.segB + np;
    unsigned char *area = reinterpret_cast<unsigned char *>(d.segC + np);
    d.cand = reinterpret_cast<unsigned long long *>(area);
    d.aux = reinterpret_cast<float *>(area + size_t(CAP) * 8);
    d.aux2 = d.aux + CAP;
    d.sorted = reinterpret_cast<unsigned long long *>(d.aux);
    d.ring = area;
    d.hmass = reinterpret_cast<unsigned long long *>(area);                     // HB * 8 bytes
    d.hcnt = reinterpret_cast<uint32_t *>(area + size_t(HB) * 8);               // HB * 4 bytes
    return d;
}

#ifdef SV_TIMING
#define SV_MARK(A, r, j)                                                  \
    do {                                                                  \
        if (threadIdx.x == 0) (A).timing[(size_t)(r) * NTIME + (j)] = global_ns(); \
    } while (0)
#else
#define SV_MARK(A, r, j) \
    do {                 \
    } while (0)
#endif

__device__ __forceinline__ void record_error(const Args &A, int code, int b) {
    atomicCAS(A.hdr, 0, code);
    atomicMax(A.hdr + 1, INT_MAX - b);
}

// ------------------------------------------------------------------------------------------
// the row phase
// ------------------------------------------------------------------------------------------

// Appends this lane's tokens of segment seg whose key reaches tkey to the candidate buffer
// (warp-aggregated; entries beyond CAP are counted but not stored).
__device__ __forceinline__ void append_candidates(Ctx &S, const Dyn &D, int seg, const float v[8], uint32_t tkey,
                                                  int V) {
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
            if (pos < CAP) D.cand[pos] = ((unsigned long long)key << 32) | (uint32_t)(~(uint32_t)idx);
            pos++;
        }
    }
}

// Warp 0: top-k cut, top-p cut and kept mass over n <= WCAP candidates sorted by value
// (descending), 8 per lane.  Writes S.n2 (kept count), S.zk (kept mass), S.cutkey.
__device__ __forceinline__ void warp_cut(Ctx &S, const unsigned long long *srt, int n, int K, float m, float s,
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

// Kept set of a sampled row from the top-k candidates.  Returns false on candidate overflow.
template <typename E, bool VEC>
__device__ bool kept_from_candidates(const Args &A, Ctx &S, const Dyn &D, const E *row, RowStat &st, int row_idx,
                                     bool want_bonus) {
    const int tid = threadIdx.x, warp = warp_id(), lane = lane_id();
    const int V = A.V, nseg = A.nseg, K = S.K;
    const float m = S.m, s = S.s;
    // lower bound on the K-th largest token: the K-th largest segment maximum, to 16 bits
    uint32_t tkey = 0;
    SV_MARK(A, row_idx, 8);
    if (nseg >= K) tkey = select_bound16(S, D.segA, nseg, K, D.hcnt);
    SV_MARK(A, row_idx, 9);
    // the segments holding a token at or above the bound, re-read (from L2) four at a time
    int *segl = reinterpret_cast<int *>(D.segC);
    if (tid == 0) {
        S.nsel = 0;
        S.ncand = 0;
    }
    __syncthreads();
    for (int j = tid; j < nseg; j += NT)
        if (fkey(D.segA[j]) >= tkey) segl[atomicAdd(&S.nsel, 1)] = j;
    __syncthreads();
    const int nsel = S.nsel;
    SV_MARK(A, row_idx, 10);
    constexpr int U = 4;
    for (int j0 = warp; j0 < nsel; j0 += NWARP * U) {
        Raw8<E> raw[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int j = j0 + u * NWARP;
            if (j < nsel) raw[u] = load_raw8<VEC>(row, segl[j] * SEG + lane * 8, V);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int j = j0 + u * NWARP;
            if (j < nsel) {
                const int seg = segl[j];
                float v[8];
                unpack8(raw[u], v);
                patch_seg(S, seg * SEG, v);
                append_candidates(S, D, seg, v, tkey, V);
            }
        }
    }
    __syncthreads();
    const int n = S.ncand;
    SV_MARK(A, row_idx, 11);
    if (n > CAP || n < 1) return false;

    if (n <= WCAP) {
        // rank sort by (value desc, token asc): keys are distinct, so ranks are a permutation
        unsigned long long *srt = D.sorted;
        for (int j = tid; j < n; j += NT) {
            const unsigned long long c = D.cand[j];
            int r = 0;
            for (int i = 0; i < n; i++) r += D.cand[i] > c ? 1 : 0;
            srt[r] = c;
        }
        __syncthreads();
        SV_MARK(A, row_idx, 12);
        if (warp == 0) warp_cut(S, srt, n, K, m, s, S.topp_on, S.P);
        __syncthreads();
        SV_MARK(A, row_idx, 13);
        const int n2 = S.n2;
        const float Z = S.zk;
        st.Z = Z;
        st.invZ = __frcp_rn(Z);
        st.taukey = S.cutkey;
        st.tau = key2f(S.cutkey);
        st.kind = KIND_LIST;
        st.nlist = n2;
        // the kept set in token order (rank by token id), stored for the residual draw
        int *ltok = reinterpret_cast<int *>(D.cand);
        float *lw = reinterpret_cast<float *>(D.cand) + WCAP;
        for (int j = tid; j < n2; j += NT) {
            const uint32_t tj = ~(uint32_t)srt[j];
            int r = 0;
            for (int i = 0; i < n2; i++) r += (~(uint32_t)srt[i]) < tj ? 1 : 0;
            ltok[r] = (int)tj;
            lw[r] = weight(key2f((uint32_t)(srt[j] >> 32)), m, s);
        }
        __syncthreads();
        int2 *L = reinterpret_cast<int2 *>(A.lists + (size_t)row_idx * LCAP * 2);
        for (int j = tid; j < n2; j += NT) L[j] = make_int2(ltok[j], __float_as_int(lw[j]));
        SV_MARK(A, row_idx, 14);
        if (want_bonus) {
            if (warp == 0) {
                const float u = __ldg(A.uni + (size_t)row_idx * 2 + 1);
                float w8[8];
#pragma unroll
                for (int t = 0; t < 8; t++) w8[t] = (lane * 8 + t < n2) ? lw[lane * 8 + t] : 0.f;
                const int j = warp_draw8(w8, n2, u);
                if (lane == 0) S.tok = j >= 0 ? ltok[j] : -1;
            }
            __syncthreads();
            st.bonus = S.tok;
        }
        SV_MARK(A, row_idx, 15);
        return true;
    }

    // larger candidate sets: block-wide bitonic sort and scans
    const int np = pow2_at_least(n);
    for (int j = n + tid; j < np; j += NT) D.cand[j] = 0ull;
    __syncthreads();
    block_sort_desc(D.cand, np);
    const int kk = min(K, n);
    const uint32_t kkey = (uint32_t)(D.cand[kk - 1] >> 32);
    int c1 = 0;
    for (int j = tid; j < n; j += NT) c1 += ((uint32_t)(D.cand[j] >> 32) >= kkey) ? 1 : 0;
    const int n1 = block_sum_i(c1, S.redi);
    for (int j = tid; j < n1; j += NT) D.aux[j] = weight(key2f((uint32_t)(D.cand[j] >> 32)), m, s);
    __syncthreads();
    for (int j = tid; j < n1; j += NT) D.aux2[j] = D.aux[j];
    __syncthreads();
    block_scan_incl(D.aux2, n1, S.redf);
    int n2 = n1;
    if (S.topp_on) {
        const float PZ = __fmul_rn(S.P, D.aux2[n1 - 1]);
        int cut = 0x7fffffff;
        for (int j = tid; j < n1; j += NT) {
            if (j > 0 && (uint32_t)(D.cand[j] >> 32) != (uint32_t)(D.cand[j - 1] >> 32) && D.aux2[j - 1] >= PZ)
                cut = min(cut, j);
        }
        cut = block_min_i(cut, S.redi);
        if (cut != 0x7fffffff) n2 = cut;
    }
    const float Z = D.aux2[n2 - 1];
    const uint32_t taukey = (uint32_t)(D.cand[n2 - 1] >> 32);
    st.Z = Z;
    st.invZ = __frcp_rn(Z);
    st.taukey = taukey;
    st.tau = key2f(taukey);
    st.kind = n2 <= LCAP ? KIND_LIST : KIND_THRESH;
    st.nlist = n2 <= LCAP ? n2 : 0;
    __syncthreads();
    if (n2 <= LCAP || want_bonus) {
        const int np2 = pow2_at_least(n2);
        for (int j = tid; j < np2; j += NT) {
            unsigned long long c = D.cand[j];
            D.cand[j] = j < n2 ? ((c << 32) | (c >> 32)) : 0ull;
        }
        __syncthreads();
        block_sort_desc(D.cand, np2);
        for (int j = tid; j < n2; j += NT) D.aux[j] = weight(key2f((uint32_t)D.cand[j]), m, s);
        __syncthreads();
        if (n2 <= LCAP) {
            int2 *L = reinterpret_cast<int2 *>(A.lists + (size_t)row_idx * LCAP * 2);
            for (int j = tid; j < n2; j += NT)
                L[j] = make_int2((int32_t)(~(uint32_t)(D.cand[j] >> 32)), __float_as_int(D.aux[j]));
        }
        if (want_bonus) {
            const float u = __ldg(A.uni + (size_t)row_idx * 2 + 1);
            int j = draw_small(D.aux, D.aux2, n2, u, S);
            st.bonus = j >= 0 ? (int32_t)(~(uint32_t)(D.cand[j] >> 32)) : -1;
        }
    }
    __syncthreads();
    return true;
}

// Kept set by radix select over the whole row (any top-k / top-p).
template <typename E, bool VEC>
__device__ void kept_by_select(const Args &A, Ctx &S, const Dyn &D, const E *row, RowStat &st, int row_idx,
                               bool want_bonus) {
    const int V = A.V, nseg = A.nseg;
    const float m = S.m, s = S.s;
    uint32_t key_lo = 0;
    if (S.topk_on) key_lo = select_kth_row<E, VEC>(S, row, V, nseg, S.K, D.hcnt);
    if (S.topp_on) key_lo = select_mass_row<E, VEC>(S, row, V, nseg, key_lo, m, s, S.P, D.hmass);
    WKept wk{m, s, key_lo};
    seg_sums<E, VEC, false>(S, row, nullptr, V, nseg, D.segB, wk, nullptr, wk);
    float part = 0.f;
    for (int j = threadIdx.x; j < nseg; j += NT) part += D.segB[j];
    const float Z = block_sum(part, S.redf);
    st.Z = Z;
    st.invZ = __frcp_rn(Z);
    st.taukey = key_lo;
    st.tau = key_lo ? key2f(key_lo) : -INFINITY;
    st.kind = KIND_THRESH;
    st.nlist = 0;
    if (want_bonus) {
        const float u = __ldg(A.uni + (size_t)row_idx * 2 + 1);
        st.bonus = draw_by_segments<E, VEC, false>(S, row, nullptr, V, nseg, D.segB, u, wk);
    }
}

template <typename E, bool VEC>
__device__ void row_phase(const Args &A, Ctx &S, const Dyn &D, const int row_idx) {
    const int tid = threadIdx.x;
    const int V = A.V, nseg = A.nseg;
    const E *row = reinterpret_cast<const E *>(A.logits) + (size_t)row_idx * V;
    RowStat st;
    st.m = 0.f; st.s = 0.f; st.tau = -INFINITY; st.Z = 1.f; st.invZ = 1.f; st.taukey = 0;
    st.argmax = -1; st.bonus = -1; st.kind = KIND_SKIP; st.nlist = 0; st.pad0 = 0; st.pad1 = 0;

    const bool sampled = !S.greedy;
    const int i = S.i;
    const bool want_bonus = sampled && i == S.k;
    float s = 0.f;
    if (sampled) s = __fdiv_rn(LOG2E, S.T);
    if (tid == 0) {
        S.s = s;
        S.topk_on = sampled && S.K > 0 && S.K < V;
        S.topp_on = sampled && S.P < 1.f;
    }
    // The last thread prefetches this row's draft token x and the values z_x, q(x) that the
    // accept test needs; they land while the row streams and are used after it.
    int xtok = -1;
    E zraw = E(0);
    float qx = 0.f;
    if (tid == NT - 1 && i < S.k) {
        xtok = __ldg(A.tokens + S.d0 + i);
        if (xtok >= 0 && xtok < V) {
            zraw = __ldg(row + xtok);
            if (sampled) qx = __ldg(A.q + (size_t)(S.d0 + i) * V + xtok);
        }
    }
    __syncthreads();
    const bool need_sum = sampled && !S.topk_on && !S.topp_on;
    bool streamed = true;
    if (VEC) streamed = pass_stats_ring<E>(S, D.ring, row, V, nseg, D.segA, D.segB, need_sum, s);
    else pass_stats<E, VEC>(S, row, V, nseg, D.segA, D.segB, need_sum, s);
    if (tid == NT - 1) {
        S.xtok = xtok;
        S.zx = elem_z_raw(S, zraw, xtok);
        S.qx = qx;
    }
    __syncthreads();
    SV_MARK(A, row_idx, 2);
    if (!streamed) {
        // a bounded wait expired: fail the row (its request's outputs become -1)
        if (tid == 0) {
            record_error(A, SV_DEV_TIMEOUT, S.b);
            st.kind = KIND_FAIL;
            A.stats[row_idx] = st;
        }
        return;
    }
    float mx = -INFINITY;
    for (int j = tid; j < nseg; j += NT) mx = fmaxf(mx, D.segA[j]);
    const float m = block_max(mx, S.redf);
    if (tid == 0) S.m = m;
    __syncthreads();
    st.m = m;
    st.s = s;

    if (!sampled) {
        // greedy: lowest id of the maximum -- first segment holding it, then first lane slot
        int first = 0x7fffffff;
        for (int j = tid; j < nseg; j += NT)
            if (D.segA[j] == m) first = min(first, j);
        first = block_min_i(first, S.redi);
        if (warp_id() == 0) {
            int best = 0x7fffffff;
            if (first != 0x7fffffff) {
                float v[8];
                seg_values<E, VEC>(S, row, V, first, v);
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    int idx = first * SEG + lane_id() * 8 + j;
                    if (idx < V && v[j] == m) best = min(best, idx);
                }
            }
            best = warp_min_i(best);
            if (lane_id() == 0) S.tok = best == 0x7fffffff ? 0 : best;
        }
        __syncthreads();
        st.argmax = S.tok;
        st.kind = KIND_GREEDY;
    } else if (need_sum) {
        // no filter: Z from the segment sums rescaled to the row max (fixed order)
        float part = 0.f;
        for (int j = tid; j < nseg; j += NT) {
            float w = D.segA[j] > -INFINITY ? __fmul_rn(D.segB[j], weight(D.segA[j], m, s)) : 0.f;
            D.segB[j] = w;
            part += w;
        }
        const float Z = block_sum(part, S.redf);
        st.Z = Z;
        st.invZ = __frcp_rn(Z);
        st.kind = KIND_FULL;
        if (want_bonus) {
            const float u = __ldg(A.uni + (size_t)row_idx * 2 + 1);
            WKept wk{m, s, 0u};
            st.bonus = draw_by_segments<E, VEC, false>(S, row, nullptr, V, nseg, D.segB, u, wk);
        }
    } else {
        bool done = false;
        if (S.topk_on && S.K <= KCAP) done = kept_from_candidates<E, VEC>(A, S, D, row, st, row_idx, want_bonus);
        if (!done) kept_by_select<E, VEC>(A, S, D, row, st, row_idx, want_bonus);
    }

    SV_MARK(A, row_idx, 3);
    // the draft of this row: p(x_i) and q(x_i)
    if (tid == 0 && i < S.k) {
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
        A.pq[(size_t)(S.d0 + i) * 2] = p;
        A.pq[(size_t)(S.d0 + i) * 2 + 1] = q;
        if (A.out_pq) {
            A.out_pq[(size_t)(S.d0 + i) * 2] = p;
            A.out_pq[(size_t)(S.d0 + i) * 2 + 1] = q;
        }
    }
    if (tid == 0) A.stats[row_idx] = st;
}

// ------------------------------------------------------------------------------------------
// the request phase (run by the CTA that completes the request's last row)
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ RowStat load_stat(const RowStat *p) {
    const int4 *q = reinterpret_cast<const int4 *>(p);
    int4 a = __ldcg(q), b = __ldcg(q + 1), c = __ldcg(q + 2);
    RowStat st;
    st.m = __int_as_float(a.x); st.s = __int_as_float(a.y); st.tau = __int_as_float(a.z); st.Z = __int_as_float(a.w);
    st.invZ = __int_as_float(b.x); st.taukey = (uint32_t)b.y; st.argmax = b.z; st.bonus = b.w;
    st.kind = c.x; st.nlist = c.y; st.pad0 = c.z; st.pad1 = c.w;
    return st;
}

// Accept test of one draft ("Speculative Decoding in Custom LLM Servicing...", "The Memory
// Bandwidth Wall and Speculative Math"): accept with probability min(1, p/q), i.e. iff
// u < min(1, p/q); q == 0 < p accepts and p == 0 rejects.
__device__ __forceinline__ bool accept_test(float p, float q, float u) {
    if (!(p > 0.f)) return false;
    if (q == 0.f) return true;
    const float ratio = __fdiv_rn(p, q);
    return u < (ratio < 1.f ? ratio : 1.f);
}

template <typename E, bool VEC, bool QVEC>
__device__ void finalize(const Args &A, Ctx &S, const Dyn &D) {
    const int tid = threadIdx.x, warp = warp_id(), lane = lane_id();
    const int b = S.b, k = S.k, r0 = S.r0, d0 = S.d0, V = A.V;
    if (warp == 0) {
        // one lane per draft: validate, test, and find the first rejection by ballot
        int status = S.status;
        int a = -1, tok = -1, need = 0;
        if (status == 0) {
            const bool greedy = S.greedy;
            bool badtok = false, baduni = false, badrow = false;
            a = k;
            for (int i0 = 0; i0 <= k; i0 += 32) {
                const int i = i0 + lane;
                bool rej = false;
                if (i <= k && __ldcg(&A.stats[r0 + i].kind) == KIND_FAIL) badrow = true;
                if (i < k) {
                    const int x = __ldg(A.tokens + d0 + i);
                    if (x < 0 || x >= V) badtok = true;
                    if (greedy) {
                        rej = x != __ldcg(&A.stats[r0 + i].argmax);
                    } else {
                        const float p = __ldcg(A.pq + (size_t)(d0 + i) * 2);
                        const float q = __ldcg(A.pq + (size_t)(d0 + i) * 2 + 1);
                        rej = !accept_test(p, q, __ldg(A.uni + (size_t)(r0 + i) * 2));
                    }
                }
                if (!greedy && i <= k) {
                    const float u0 = __ldg(A.uni + (size_t)(r0 + i) * 2), u1 = __ldg(A.uni + (size_t)(r0 + i) * 2 + 1);
                    if (!(u0 >= 0.f && u0 < 1.f) || !(u1 >= 0.f && u1 < 1.f)) baduni = true;
                }
                const unsigned msk = __ballot_sync(0xffffffffu, rej);
                if (msk && a == k) a = i0 + __ffs(msk) - 1;
            }
            badtok = __any_sync(0xffffffffu, badtok);
            baduni = __any_sync(0xffffffffu, baduni);
            badrow = __any_sync(0xffffffffu, badrow);
            if (badtok) status = SV_DEV_BAD_TOKEN;
            else if (baduni) status = SV_DEV_BAD_UNIFORM;
            else if (badrow) status = SV_DEV_TIMEOUT;
            if (status == 0) {
                if (greedy) tok = __ldcg(&A.stats[r0 + a].argmax);
                else if (a == k) tok = __ldcg(&A.stats[r0 + k].bonus);
                else need = 1;
            } else {
                a = -1;
            }
        }
        if (lane == 0) {
            if (status) record_error(A, status, b);
            S.a = a;
            S.tok = tok;
            S.need_resid = need;
        }
    }
    __syncthreads();
    if (S.need_resid) {
        // residual max(0, p - q) at the rejected row a ("Speculative Decoding in Custom LLM
        // Servicing...", "The Memory Bandwidth Wall and Speculative Math")
        const int a = S.a;
        const RowStat st = load_stat(A.stats + r0 + a);
        const float *qrow = A.q + (size_t)(d0 + a) * V;
        const float u = __ldg(A.uni + (size_t)(r0 + a) * 2 + 1);
        if (st.kind == KIND_LIST) {
            // p is zero outside the stored kept list, so r is too: gather q on the list only
            if (warp == 0) {
                const int n = st.nlist;
                const int2 *L = reinterpret_cast<const int2 *>(A.lists + (size_t)(r0 + a) * LCAP * 2);
                int tk[8];
                float pw[8], rw[8];
#pragma unroll
                for (int t = 0; t < 8; t++) {
                    const int idx = lane * 8 + t;
                    int2 e = idx < n ? __ldcg(L + idx) : make_int2(-1, 0);
                    tk[t] = e.x;
                    pw[t] = idx < n ? __fmul_rn(__int_as_float(e.y), st.invZ) : 0.f;
                }
#pragma unroll
                for (int t = 0; t < 8; t++) {
                    const float q = tk[t] >= 0 ? __ldg(qrow + tk[t]) : 0.f;
                    rw[t] = tk[t] >= 0 ? fmaxf(__fsub_rn(pw[t], q), 0.f) : 0.f;
                }
                int j = warp_draw8(rw, n, u);
                if (j < 0) j = warp_draw8(pw, n, u);      // empty residual: draw from p
                int sel = -1;
#pragma unroll
                for (int t = 0; t < 8; t++)
                    if (lane * 8 + t == j) sel = tk[t];
                sel = __shfl_sync(0xffffffffu, sel, j >= 0 ? (j >> 3) : 0);
                if (lane == 0) S.tok = j >= 0 ? sel : -1;
            }
            __syncthreads();
        } else {
            if (warp == 0) build_penalties(A, S, a);
            __syncthreads();
            const E *row = reinterpret_cast<const E *>(A.logits) + (size_t)(r0 + a) * V;
            WResid wr{st.m, st.s, st.invZ, st.taukey};
            WProb wp{st.m, st.s, st.invZ, st.taukey};
            seg_sums<E, VEC, QVEC>(S, row, qrow, V, A.nseg, D.segB, wr, D.segC, wp);
            int tok = draw_by_segments<E, VEC, QVEC>(S, row, qrow, V, A.nseg, D.segB, u, wr);
            if (tok < 0) tok = draw_by_segments<E, VEC, QVEC>(S, row, nullptr, V, A.nseg, D.segC, u, wp);
            if (tid == 0) S.tok = tok;
            __syncthreads();
        }
    }
    // outputs: accepted drafts, the final token, -1 padding
    const int a = S.a, kw = A.k_max + 1;
    for (int j = tid; j < kw; j += NT) {
        int v = -1;
        if (a >= 0) v = j < a ? __ldg(A.tokens + d0 + j) : (j == a ? S.tok : -1);
        A.out_tok[(size_t)b * kw + j] = v;
    }
    if (tid == 0) {
        A.acc[b] = a;
        A.counters[b] = 0;
    }
}

// Writes -1 outputs for a request that owns no rows (inconsistent row_offsets).
__device__ __forceinline__ void fail_request(const Args &A, int b) {
    const int kw = A.k_max + 1;
    for (int j = threadIdx.x; j < kw; j += NT) A.out_tok[(size_t)b * kw + j] = -1;
    if (threadIdx.x == 0) {
        A.acc[b] = -1;
        record_error(A, 1, b);
    }
}

template <typename E, bool VEC, bool QVEC>
__global__ void __launch_bounds__(NT, 4) verify_kernel(const Args A) {
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ Ctx S;
    const int tid = threadIdx.x;
    const int r = blockIdx.x;
    const Dyn D = carve(dsm, A.nseg);
    SV_MARK(A, r, 0);
#ifdef SV_TIMING
    if (tid == 0) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        A.timing[(size_t)r * NTIME + 6] = smid;
        A.timing[(size_t)r * NTIME + 7] = 0;
    }
#endif
    // start streaming this CTA's row right away; the request lookup overlaps the first copies
    if (VEC && tid == 0) ring_start(S, D.ring, reinterpret_cast<const E *>(A.logits) + (size_t)r * A.V, A.V, (int)sizeof(E));

    // locate the row: request b, row i within it
    if (tid < 32) {
        int b, r0, nrows;
        bool ok = true;
        if (A.row_off) {
            b = find_request(A.row_off, A.B, r);
            ok = b >= 0 && b < A.B;
            r0 = ok ? __ldg(A.row_off + b) : 0;
            int r1 = ok ? __ldg(A.row_off + b + 1) : 0;
            ok = ok && r0 <= r && r < r1;
            nrows = r1 - r0;
        } else {
            b = r / (A.k_max + 1);
            r0 = b * (A.k_max + 1);
            nrows = A.k_max + 1;
        }
        if (tid == 0) {
            S.r0 = r0;
            S.nrows = nrows;
            S.i = r - r0;
            S.d0 = r0 - b;
            if (ok) {
                load_request(A, S, b);
            } else {
                S.b = -1;
                S.status = 1;
                record_error(A, 1, b < 0 ? 0 : (b >= A.B ? A.B - 1 : b));
            }
            S.active = ok && S.status == 0 && S.i <= S.k;
        }
    }
    __syncthreads();
    SV_MARK(A, r, 1);
    if (VEC && !S.active) {   // nothing to compute: let the speculative copies land first
        if (tid == 0) ring_drain(S);
        __syncthreads();
    }
    if (S.b < 0) return;   // row outside every request: nothing to count

    // requests with no rows (row_offsets[j] == row_offsets[j+1]) are failed by the first row
    // of the nearest non-empty request before them; leading ones by the request of row 0
    if (A.row_off && S.i == 0) {
        if (r == 0) {
            for (int j = S.b - 1; j >= 0; j--) fail_request(A, j);
        }
        for (int j = S.b + 1; j < A.B && __ldg(A.row_off + j) == __ldg(A.row_off + j + 1); j++) fail_request(A, j);
    }

    if (S.active) {
        if (tid < 32) build_penalties(A, S, S.i);
        __syncthreads();
        row_phase<E, VEC>(A, S, D, r);
    }
    SV_MARK(A, r, 4);

    // arrival: the CTA that brings the count to the request's row count finalises it
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        int old = atomicAdd(A.counters + S.b, 1);
        S.last = (old == S.nrows - 1);
    }
    __syncthreads();
    if (S.last) {
        __threadfence();
        finalize<E, VEC, QVEC>(A, S, D);
#ifdef SV_TIMING
        if (tid == 0) A.timing[(size_t)r * NTIME + 7] = 1;
#endif
    }
    SV_MARK(A, r, 5);
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

template <typename E, bool VEC, bool QVEC>
static cudaError_t launch(const Args &A, cudaStream_t stream) {
    static size_t smem_set = 0;   // largest dynamic shared memory size enabled so far
    const size_t smem = dyn_bytes(A.nseg);
    auto kern = verify_kernel<E, VEC, QVEC>;
    if (smem > 48 * 1024 && smem > smem_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
    kern<<<A.R, NT, smem, stream>>>(A);
    return cudaGetLastError();
}

}  // namespace sv

using namespace sv;

extern "C" size_t sv_workspace_bytes(int32_t B, int32_t total_rows, int32_t V) {
    if (B < 1 || total_rows < B || V < 1) return 0;
    return ws_layout(B, total_rows).total;
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

extern "C" sv_status spec_verify(const void *target_logits, sv_dtype logits_dtype, const float *draft_probs,
                                 const int32_t *draft_tokens, const int32_t *num_drafts, const int32_t *row_offsets,
                                 int32_t B, int32_t k_max, int32_t V, int32_t total_rows, sv_params params,
                                 const float *uniforms, int32_t *out_tokens, int32_t *accept_len, float *out_pq,
                                 void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 1 || k_max < 0 || V < 1 || total_rows < B) return SV_ERR_INVALID_ARG;
    if (k_max > MAXK || V > MAXV) return SV_ERR_UNSUPPORTED;
    if (logits_dtype != SV_F32 && logits_dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (!row_offsets && (long long)total_rows != (long long)B * (k_max + 1)) return SV_ERR_INVALID_ARG;
    const int D = total_rows - B;
    if (!target_logits || !num_drafts || !uniforms || !out_tokens || !accept_len || !workspace) return SV_ERR_INVALID_ARG;
    if (D > 0 && (!draft_probs || !draft_tokens)) return SV_ERR_INVALID_ARG;
    if (!params.temperature || !params.top_k || !params.top_p || !params.greedy) return SV_ERR_INVALID_ARG;
    if ((long long)total_rows * V > (1ll << 62)) return SV_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(B, total_rows);
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
    A.uni = uniforms;
    A.out_tok = out_tokens;
    A.acc = accept_len;
    A.out_pq = out_pq;
    A.hdr = reinterpret_cast<int32_t *>(ws);
    A.counters = reinterpret_cast<int32_t *>(ws + L.counters);
    A.stats = reinterpret_cast<RowStat *>(ws + L.stats);
    A.pq = reinterpret_cast<float *>(ws + L.pq);
    A.lists = reinterpret_cast<int32_t *>(ws + L.lists);
    A.timing = reinterpret_cast<unsigned long long *>(ws + L.timing);
    A.B = B;
    A.k_max = k_max;
    A.V = V;
    A.R = total_rows;
    A.nseg = (V + SEG - 1) / SEG;
    const size_t esz = logits_dtype == SV_BF16 ? 2 : 4;
    const bool vec = ((uintptr_t)target_logits % 16 == 0) && ((size_t)V * esz) % 16 == 0;
    const bool qvec = (!draft_probs || (uintptr_t)draft_probs % 16 == 0) && ((size_t)V * 4) % 16 == 0;
    A.q_vec = qvec;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // clear the error word and the per-request arrival counters
    if (cudaMemsetAsync(ws, 0, L.counters + (size_t)B * 4, st) != cudaSuccess) return SV_ERR_CUDA;
    cudaError_t e;
    if (logits_dtype == SV_BF16) {
        if (vec) e = qvec ? launch<uint16_t, true, true>(A, st) : launch<uint16_t, true, false>(A, st);
        else e = qvec ? launch<uint16_t, false, true>(A, st) : launch<uint16_t, false, false>(A, st);
    } else {
        if (vec) e = qvec ? launch<float, true, true>(A, st) : launch<float, true, false>(A, st);
        else e = qvec ? launch<float, false, true>(A, st) : launch<float, false, false>(A, st);
    }
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
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

// sv_row.cuh -- per-row work of the verify kernel: locating the row, building the
// presence/frequency penalties of the drafts before it, streaming the row once for its
// statistics, selecting the kept set (top-k / top-p) and drawing tokens by inverse CDF.
//
// Method ("Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust",
// "The Verification Algorithm"; FreeToken PR #836, "Design"): each of a request's k+1 target
// rows becomes p = softmax(z / T) over the tokens kept by top-k and then top-p, where
// z = logit - presence*[c > 0] - frequency*c counts the drafts before the row.
//
// All sums that feed a decision use a fixed association (deterministic reductions), so
// results are bitwise reproducible run to run.
#pragma once

#include "sv_block.cuh"

namespace sv {

// Static shared state of one row CTA.
struct Ctx {
    unsigned long long full[NS];    // ring stage holds its chunk (transaction-count barrier)
    unsigned long long empty[NS];   // every warp is done with the stage
    int issued, ring_fail;
    int b, i, k, r0, d0, nrows, status, active, greedy;
    int K, topk_on, topp_on;
    float T, P, pres, freq, s, m;
    int npen;
    int pid[MAXK];
    float ppen[MAXK];
    int draft_raw[MAXK];
    float redf[NWARP];
    int redi[NWARP];
    int ncand, nsel, n2;
    float zx, qx, zk;
    int xtok;
    uint32_t cutkey;
    int sel_digit;
    long long sel_below;
    unsigned long long sel_mass;
    double sel_target;
    int last, a, tok, need_resid;
};

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

// Request-level checks shared by every row of the request (thread 0 only).
__device__ __forceinline__ void load_request(const Args &A, Ctx &S, int b) {
    S.b = b;
    int k = __ldg(A.nd + b);
    S.k = k;
    int status = 0;
    if (k < 0 || k > A.k_max || k > S.nrows - 1) status = 1;           // SV_DEV_BAD_LAYOUT
    S.greedy = __ldg(A.greedy + b) != 0;
    S.pres = A.pres ? __ldg(A.pres + b) : 0.f;
    S.freq = A.freq ? __ldg(A.freq + b) : 0.f;
    if (!isfinite(S.pres) || !isfinite(S.freq)) status = status ? status : 6;
    // every field is loaded up front (one round trip); greedy requests ignore T, P and K
    const float T = __ldg(A.T + b);
    const float P = __ldg(A.topp + b);
    const int K = __ldg(A.topk + b);
    S.T = 1.f;
    S.P = 1.f;
    S.K = 0;
    if (!S.greedy) {
        if (!(T > 0.f) || !isfinite(T)) status = status ? status : 3;
        if (!(P > 0.f && P <= 1.f)) status = status ? status : 4;
        S.T = T;
        S.P = P;
        S.K = K;
    }
    S.status = status;
}

// Penalties of row i: the distinct drafts d_0..d_{i-1} with pen = presence + frequency * count
// (FreeToken PR #836, "Design": earlier drafts count as already generated).  Run by warp 0.
__device__ __forceinline__ void build_penalties(const Args &A, Ctx &S, int i) {
    const int lane = lane_id();
    if (lane == 0) S.npen = 0;
    __syncwarp();
    if (i == 0 || (S.pres == 0.f && S.freq == 0.f)) return;
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
            pen = __fadd_rn(S.pres, __fmul_rn(S.freq, (float)c));
            keep = first && v >= 0 && v < A.V && pen != 0.f;
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
__device__ __forceinline__ void patch_seg(const Ctx &S, int seg_lo, float v[8]) {
    const int npen = S.npen;
    if (npen == 0) return;
    const int lane = lane_id();
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

// Penalised value of a single token x of the row.
template <typename E>
__device__ __forceinline__ float elem_z(const Ctx &S, const E *row, int x);

template <>
__device__ __forceinline__ float elem_z<uint16_t>(const Ctx &S, const uint16_t *row, int x) {
    float z = __uint_as_float((uint32_t)__ldg(row + x) << 16);
    for (int h = 0; h < S.npen; h++)
        if (S.pid[h] == x) z = __fsub_rn(z, S.ppen[h]);
    return z;
}
template <>
__device__ __forceinline__ float elem_z<float>(const Ctx &S, const float *row, int x) {
    float z = __ldg(row + x);
    for (int h = 0; h < S.npen; h++)
        if (S.pid[h] == x) z = __fsub_rn(z, S.ppen[h]);
    return z;
}

// Penalised value of token x from its raw stored element.
__device__ __forceinline__ float elem_z_raw(const Ctx &S, uint16_t raw, int x) {
    float z = __uint_as_float((uint32_t)raw << 16);
    for (int h = 0; h < S.npen; h++)
        if (S.pid[h] == x) z = __fsub_rn(z, S.ppen[h]);
    return z;
}
__device__ __forceinline__ float elem_z_raw(const Ctx &S, float raw, int x) {
    float z = raw;
    for (int h = 0; h < S.npen; h++)
        if (S.pid[h] == x) z = __fsub_rn(z, S.ppen[h]);
    return z;
}

// Loads and penalises the 8 values of this lane in segment seg.
template <typename E, bool VEC>
__device__ __forceinline__ void seg_values(const Ctx &S, const E *row, int V, int seg, float v[8]) {
    Raw8<E> raw = load_raw8<VEC>(row, seg * SEG + lane_id() * 8, V);
    unpack8(raw, v);
    patch_seg(S, seg * SEG, v);
}

// ------------------------------------------------------------------------------------------
// pass 1: one streaming read of the row -> per-segment max (and weight sum)
// ------------------------------------------------------------------------------------------

template <typename E, bool VEC>
__device__ __forceinline__ void pass_stats(const Ctx &S, const E *row, int V, int nseg, float *segmax,
                                           float *segsum, bool need_sum, float s) {
    constexpr int U = sizeof(E) == 2 ? 4 : 2;   // segments in flight per warp
    const int warp = warp_id(), lane = lane_id();
    for (int s0 = warp; s0 < nseg; s0 += NWARP * U) {
        Raw8<E> raw[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            int seg = s0 + u * NWARP;
            if (seg < nseg) raw[u] = load_raw8<VEC>(row, seg * SEG + lane * 8, V);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            int seg = s0 + u * NWARP;
            if (seg < nseg) {
                float v[8];
                unpack8(raw[u], v);
                patch_seg(S, seg * SEG, v);
                float mx = warp_max(max8(v));
                float sum = 0.f;
                if (need_sum && mx > -INFINITY) {
                    float ms = __fmul_rn(mx, s);
#pragma unroll
                    for (int j = 0; j < 8; j++) sum += ex2(fmaf(v[j], s, -ms));
                    sum = warp_sum(sum);
                }
                if (lane == 0) {
                    segmax[seg] = mx;
                    segsum[seg] = sum;
                }
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// pass 1 through a shared-memory ring fed by bulk copies (16-byte aligned rows)
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ int ring_chunks(int V, int esize) {
    const uint32_t RB = (uint32_t)V * esize;
    return (int)((RB + SB - 1) / SB);
}

// Thread 0: copy chunk c (SB bytes, the last one shorter) of the row into its ring stage.
__device__ __forceinline__ void ring_issue(Ctx &S, unsigned char *ring, const void *row, uint32_t RB, int c) {
    const int st = c % NS;
    const uint32_t off = (uint32_t)c * SB;
    const uint32_t bytes = min((uint32_t)SB, RB - off);
    mbar_expect_tx(&S.full[st], bytes);
    bulk_g2s(ring + st * SB, reinterpret_cast<const unsigned char *>(row) + off, bytes, &S.full[st]);
    S.issued = c + 1;
}

// Thread 0: set up the ring barriers and start the first NS chunks of the row.
__device__ __forceinline__ void ring_start(Ctx &S, unsigned char *ring, const void *row, int V, int esize) {
    for (int s = 0; s < NS; s++) {
        mbar_init(&S.full[s], 1);
        mbar_init(&S.empty[s], NWARP);
    }
    mbar_fence_init();
    S.issued = 0;
    S.ring_fail = 0;
    const uint32_t RB = (uint32_t)V * esize;
    const int nc = ring_chunks(V, esize);
    for (int c = 0; c < NS && c < nc; c++) ring_issue(S, ring, row, RB, c);
}

// Thread 0: wait (bounded) for the latest chunk of every stage, so that no copy into shared
// memory is still in flight when the CTA moves on or exits.
__device__ __forceinline__ void ring_drain(Ctx &S) {
    for (int c = max(0, S.issued - NS); c < S.issued; c++) mbar_wait(&S.full[c % NS], (uint32_t)(c / NS) & 1u);
}

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

// Pass 1 over the ring: per-segment max (and weight sums), same results as pass_stats.
// Thread 0 refills a stage once all warps released it.  Returns false if a bounded wait
// expired (the caller fails the row).
template <typename E>
__device__ bool pass_stats_ring(Ctx &S, unsigned char *ring, const E *row, int V, int nseg, float *segmax,
                                float *segsum, bool need_sum, float s) {
    const int warp = warp_id(), lane = lane_id();
    const uint32_t RB = (uint32_t)V * sizeof(E);
    const int nc = ring_chunks(V, (int)sizeof(E));
    constexpr int SPC = SB / (SEG * (int)sizeof(E));   // segments per chunk
    int c = 0;
    for (; c < nc; c++) {
        const int st = c % NS;
        const uint32_t par = (uint32_t)(c / NS) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&S.full[st], par))) break;
        const unsigned char *buf = ring + st * SB;
        for (int j = warp; j < SPC; j += NWARP) {
            const int seg = c * SPC + j;
            if (seg >= nseg) break;
            float v[8];
            ring_values<E>(buf, j, v);
            const int base = seg * SEG + lane * 8;
            if (base + 8 > V) {
#pragma unroll
                for (int t = 0; t < 8; t++)
                    if (base + t >= V) v[t] = -INFINITY;
            }
            patch_seg(S, seg * SEG, v);
            const float mx = warp_max(max8(v));
            float sum = 0.f;
            if (need_sum && mx > -INFINITY) {
                const float ms = __fmul_rn(mx, s);
#pragma unroll
                for (int t = 0; t < 8; t++) sum += ex2(fmaf(v[t], s, -ms));
                sum = warp_sum(sum);
            }
            if (lane == 0) {
                segmax[seg] = mx;
                segsum[seg] = sum;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[st]);
        if (threadIdx.x == 0 && c + NS < nc) {
            if (mbar_wait(&S.empty[st], par)) ring_issue(S, ring, row, RB, c + NS);
            else S.ring_fail = 1;
        }
    }
    if (c < nc) atomicOr(&S.ring_fail, 1);
    __syncthreads();
    if (S.ring_fail) {
        if (threadIdx.x == 0) ring_drain(S);
        __syncthreads();
        return false;
    }
    return true;
}

// ------------------------------------------------------------------------------------------
// selection helpers (radix select with 11/11/10-bit digits, MSB first)
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ void digit_round(int round, int &shift, int &width, uint32_t &mask) {
    shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
    width = round == 2 ? 10 : 11;
    mask = round == 0 ? 0u : (round == 1 ? 0xFFE00000u : 0xFFFFFC00u);
}

// Warp 0 scans a count histogram from the highest bin down and finds the bin d holding the
// need-th largest element (cum_above(d) < need <= cum_above(d) + cnt[d]).  Writes S.sel_digit
// and S.sel_below (= cum_above(d)).  need >= 1.
__device__ __forceinline__ void find_count_bin(Ctx &S, const uint32_t *cnt, int nbins, long long need) {
    if (warp_id() != 0) return;
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

// Warp 0 finds, in a 256-bin count histogram scanned from the top, the bin holding the
// need-th largest element; 8 bins per lane.  Writes S.sel_digit and S.sel_below.
__device__ __forceinline__ void find_count_bin256(Ctx &S, const uint32_t *cnt, long long need) {
    if (warp_id() != 0) return;
    const int lane = lane_id();
    const int top = 256 - lane * 8;
    uint32_t c8[8];
    long long tot = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        c8[j] = cnt[top - 1 - j];
        tot += c8[j];
    }
    long long incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    long long excl = incl - tot;
    unsigned msk = __ballot_sync(0xffffffffu, excl < need && need <= incl);
    int owner = msk ? __ffs(msk) - 1 : 31;
    if (lane == owner) {
        long long c = excl;
        int dsel = top - 8;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            if (c + (long long)c8[j] >= need) {
                dsel = top - 1 - j;
                break;
            }
            c += c8[j];
        }
        S.sel_digit = dsel;
        S.sel_below = c;
    }
}

// A lower bound on the need-th largest of n float keys in shared memory: the top 16 bits of
// that key (two 8-bit radix rounds) with the low 16 bits cleared.  At least `need` keys are
// >= the bound, and every key above it shares the bound's 16-bit prefix or exceeds it.
__device__ uint32_t select_bound16(Ctx &S, const float *vals, int n, int need, uint32_t *cnt) {
    uint32_t prefix = 0;
    long long nd = need;
    for (int round = 0; round < 2; round++) {
        const int shift = 24 - 8 * round;
        const uint32_t mask = round == 0 ? 0u : 0xFF000000u;
        for (int d = threadIdx.x; d < 256; d += NT) cnt[d] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < n; j += NT) {
            uint32_t key = fkey(vals[j]);
            if ((key & mask) == prefix) atomicAdd(&cnt[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        find_count_bin256(S, cnt, nd);
        __syncthreads();
        prefix |= (uint32_t)S.sel_digit << shift;
        nd -= S.sel_below;
        __syncthreads();
    }
    return prefix;
}

// The need-th largest (1-based) of n float keys fkey(vals[j]) held in shared memory.
__device__ uint32_t select_kth_smem(Ctx &S, const float *vals, int n, int need, uint32_t *cnt) {
    uint32_t prefix = 0;
    long long nd = need;
    for (int round = 0; round < 3; round++) {
        int shift, width;
        uint32_t mask;
        digit_round(round, shift, width, mask);
        const int nb = 1 << width;
        for (int d = threadIdx.x; d < nb; d += NT) cnt[d] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < n; j += NT) {
            uint32_t key = fkey(vals[j]);
            if ((key & mask) == prefix) atomicAdd(&cnt[(key >> shift) & (nb - 1)], 1u);
        }
        __syncthreads();
        find_count_bin(S, cnt, nb, nd);
        __syncthreads();
        prefix |= (uint32_t)S.sel_digit << shift;
        nd -= S.sel_below;
        __syncthreads();
    }
    return prefix;
}

// The need-th largest key among the row's tokens (full passes over the row, re-read from L2).
template <typename E, bool VEC>
__device__ uint32_t select_kth_row(Ctx &S, const E *row, int V, int nseg, int need, uint32_t *cnt) {
    uint32_t prefix = 0;
    long long nd = need;
    const int warp = warp_id(), lane = lane_id();
    for (int round = 0; round < 3; round++) {
        int shift, width;
        uint32_t mask;
        digit_round(round, shift, width, mask);
        const int nb = 1 << width;
        for (int d = threadIdx.x; d < nb; d += NT) cnt[d] = 0;
        __syncthreads();
        for (int seg = warp; seg < nseg; seg += NWARP) {
            float v[8];
            seg_values<E, VEC>(S, row, V, seg, v);
#pragma unroll
            for (int j = 0; j < 8; j++) {
                int idx = seg * SEG + lane * 8 + j;
                uint32_t key = fkey(v[j]);
                if (idx < V && (key & mask) == prefix) atomicAdd(&cnt[(key >> shift) & (nb - 1)], 1u);
            }
        }
        __syncthreads();
        find_count_bin(S, cnt, nb, nd);
        __syncthreads();
        prefix |= (uint32_t)S.sel_digit << shift;
        nd -= S.sel_below;
        __syncthreads();
    }
    return prefix;
}

// Warp 0 scans a fixed-point mass histogram from the top and finds the first bin d where the
// mass above plus the bin's own mass reaches target (mass_above(d) < target <= ... + mass[d]).
__device__ __forceinline__ void find_mass_bin(Ctx &S, const unsigned long long *mass, int nbins,
                                              unsigned long long above, double target) {
    if (warp_id() != 0) return;
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
// histogram sums exact and order-independent.
template <typename E, bool VEC>
__device__ uint32_t select_mass_row(Ctx &S, const E *row, int V, int nseg, uint32_t key_lo, float m, float s,
                                    float P, unsigned long long *mass) {
    uint32_t prefix = 0;
    unsigned long long above = 0;
    double target = 0.0;
    const int warp = warp_id(), lane = lane_id();
    for (int round = 0; round < 3; round++) {
        int shift, width;
        uint32_t mask;
        digit_round(round, shift, width, mask);
        const int nb = 1 << width;
        for (int d = threadIdx.x; d < nb; d += NT) mass[d] = 0ull;
        __syncthreads();
        for (int seg = warp; seg < nseg; seg += NWARP) {
            float v[8];
            seg_values<E, VEC>(S, row, V, seg, v);
#pragma unroll
            for (int j = 0; j < 8; j++) {
                int idx = seg * SEG + lane * 8 + j;
                uint32_t key = fkey(v[j]);
                if (idx < V && key >= key_lo && (key & mask) == prefix) {
                    unsigned long long f = __float2ull_rz(__fmul_rn(weight(v[j], m, s), (float)FIXED_ONE));
                    if (f) atomicAdd(&mass[(key >> shift) & (nb - 1)], f);
                }
            }
        }
        __syncthreads();
        if (round == 0) {
            // total mass of the top-k set (every bin of round 0), summed by warp 0
            if (warp == 0) {
                unsigned long long t = 0;
                for (int d = lane; d < nb; d += 32) t += mass[d];
#pragma unroll
                for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == 0) S.sel_target = (double)P * (double)t;
            }
            __syncthreads();
            target = S.sel_target;
        }
        find_mass_bin(S, mass, nb, above, target);
        __syncthreads();
        prefix |= (uint32_t)S.sel_digit << shift;
        above = S.sel_mass;
        __syncthreads();
    }
    return prefix;
}

// ------------------------------------------------------------------------------------------
// draws by inverse CDF in token order
// ------------------------------------------------------------------------------------------

// Index j of the draw from weights w[0..n) in shared memory with uniform u: the first j whose
// running sum exceeds u * W (W = total); the last positive-weight j if rounding leaves none;
// -1 when no weight is positive.  `pre` (n floats) receives the prefix sums.
__device__ int draw_small(const float *w, float *pre, int n, float u, Ctx &S) {
    for (int j = threadIdx.x; j < n; j += NT) pre[j] = w[j];
    __syncthreads();
    if (n <= 0) return -1;
    block_scan_incl(pre, n, S.redf);
    float W = pre[n - 1];
    if (!(W > 0.f)) return -1;
    float target = __fmul_rn(u, W);
    int best = 0x7fffffff;
    for (int j = threadIdx.x; j < n; j += NT)
        if (pre[j] > target) best = min(best, j);
    best = block_min_i(best, S.redi);
    if (best == 0x7fffffff) {
        int last = -1;
        for (int j = threadIdx.x; j < n; j += NT)
            if (w[j] > 0.f) last = max(last, j);
        best = block_max_i(last, S.redi);
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

// Draw from a whole row with per-segment weight sums segw[0..nseg) (overwritten by their
// prefix sums).  The crossing segment is re-read by warp 0 and scanned lane by lane.
// Returns the token, or -1 when no weight is positive.
template <typename E, bool VEC, bool QVEC, typename WF>
__device__ int draw_by_segments(Ctx &S, const E *row, const float *qrow, int V, int nseg, float *segw,
                                float u, const WF &wf) {
    block_scan_incl(segw, nseg, S.redf);
    const float W = segw[nseg - 1];
    if (!(W > 0.f)) return -1;
    const float target = __fmul_rn(u, W);
    int best = 0x7fffffff;
    for (int j = threadIdx.x; j < nseg; j += NT)
        if (segw[j] > target) best = min(best, j);
    best = block_min_i(best, S.redi);
    bool fallback = false;
    if (best == 0x7fffffff) {
        int last = -1;
        for (int j = threadIdx.x; j < nseg; j += NT) {
            float prev = j ? segw[j - 1] : 0.f;
            if (segw[j] > prev) last = max(last, j);
        }
        best = block_max_i(last, S.redi);
        fallback = true;
        if (best < 0) return -1;
    }
    if (warp_id() == 0) {
        const int lane = lane_id();
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
        run += seg ? segw[seg - 1] : 0.f;
        int pick = 0x7fffffff, lastpos = -1;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            int idx = seg * SEG + lane * 8 + j;
            run += w[j];
            if (!fallback && run > target && pick == 0x7fffffff) pick = idx;
            if (w[j] > 0.f) lastpos = idx;
        }
        pick = warp_min_i(pick);
        lastpos = warp_max_i(lastpos);
        if (lane == 0) S.tok = pick != 0x7fffffff ? pick : lastpos;
    }
    __syncthreads();
    return S.tok;
}

// Per-segment sums of a weight functor over the whole row (one pass; q row optional).
template <typename E, bool VEC, bool QVEC, typename WF, typename WF2>
__device__ __forceinline__ void seg_sums(Ctx &S, const E *row, const float *qrow, int V, int nseg, float *out1,
                                         const WF &wf1, float *out2, const WF2 &wf2) {
    const int warp = warp_id(), lane = lane_id();
    for (int seg = warp; seg < nseg; seg += NWARP) {
        float v[8], qv[8];
        seg_values<E, VEC>(S, row, V, seg, v);
        if (qrow) {
            load_q8<QVEC>(qrow, seg * SEG + lane * 8, V, qv);
        } else {
#pragma unroll
            for (int j = 0; j < 8; j++) qv[j] = 0.f;
        }
        float a = 0.f, c = 0.f;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            int idx = seg * SEG + lane * 8 + j;
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
    }
    __syncthreads();
}

}  // namespace sv

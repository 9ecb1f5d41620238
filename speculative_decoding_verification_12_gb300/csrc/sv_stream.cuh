// sv_stream.cuh -- the streaming pass of the stream kernel: per-segment statistics of a
// row computed from its chunks in the shared-memory ring, specialised per statistics mode so
// that a clean segment costs a handful of instructions per lane.
//
// A segment is "clean" when it lies wholly inside the row and holds no penalised token; clean
// bf16 segments are reduced on packed bf16 pairs.  The rest (the row's ragged last segment,
// segments holding a penalised token, and every fp32 segment) take the float path.
#pragma once

#include "sv_row.cuh"

namespace sv {

// Warp result of one segment from each lane's top value m1: lane 0 writes the max, the lowest
// lane holding it and, in MODE_TOP2, the largest value held by any other lane (every element
// outside lane `at` is at most that value).
template <int MODE>
__device__ __forceinline__ void seg_emit(int seg, float m1, const SegStats &o) {
    const float mx = redux_max(m1);
    if constexpr (MODE == MODE_ARG || MODE == MODE_TOP2) {
        const int at = __ffs(__ballot_sync(0xffffffffu, m1 == mx)) - 1;
        float sec = 0.f;
        if constexpr (MODE == MODE_TOP2) sec = redux_max(lane_id() == at ? -INFINITY : m1);
        if (lane_id() == 0) {
            o.mx[seg] = mx;
            o.lane[seg] = at;
            if constexpr (MODE == MODE_TOP2) o.b[seg] = sec;
        }
    } else {
        if (lane_id() == 0) o.mx[seg] = mx;
    }
}

// Statistics of a segment from this lane's 8 values (already masked and penalised).
template <int MODE>
__device__ __forceinline__ void seg_from_values(const float v[8], int seg, float s, const SegStats &o) {
    if constexpr (MODE == MODE_SUM) {
        const float mx = redux_max(max8(v));
        float sum = 0.f;
        if (mx > -INFINITY) {
            const float ms = __fmul_rn(mx, s);
#pragma unroll
            for (int t = 0; t < 8; t++) sum += ex2(fmaf(v[t], s, -ms));
            sum = warp_sum(sum);
        }
        if (lane_id() == 0) {
            o.mx[seg] = mx;
            o.b[seg] = sum;
        }
    } else {
        seg_emit<MODE>(seg, max8(v), o);
    }
}

// Greedy rows: each lane keeps the largest value it has seen and where: a strictly larger value
// is the only reason to move, since its segments arrive in token order.  For clean segments the
// lane keeps the segment's raw elements (register selects, no branch) and finds the position
// within them once, at the end of the unit.
template <typename E>
struct ArgRun {
    float best;
    int seg;        // segment of best (clean), or -1
    int idx;        // token of best when it came from a dirty segment
    Raw8<E> raw;    // the lane's elements of segment seg
};

// Offset (0..7) of the first of the lane's 8 values equal to m (IEEE equality: -0 == +0).
template <typename E>
__device__ __forceinline__ int first_equal8(const Raw8<E> &raw, float m) {
    float v[8];
    unpack8(raw, v);
    int t = 7;
#pragma unroll
    for (int j = 6; j >= 0; j--)
        if (v[j] == m) t = j;
    return t;
}

template <typename E>
__device__ __forceinline__ void arg_clean(const Raw8<E> &raw, int seg, ArgRun<E> &a) {
    float m1;
    if constexpr (sizeof(E) == 2) {
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&raw.a);
        const __nv_bfloat162 M = __hmax2(__hmax2(p[0], p[1]), __hmax2(p[2], p[3]));
        m1 = fmaxf(__low2float(M), __high2float(M));
    } else {
        float v[8];
        unpack8(raw, v);
        m1 = max8(v);
    }
    const bool up = m1 > a.best;
    a.best = up ? m1 : a.best;
    a.seg = up ? seg : a.seg;
    a.raw.a = up ? raw.a : a.raw.a;
    if constexpr (sizeof(E) == 4) a.raw.b = up ? raw.b : a.raw.b;
}

// The history part of patch_seg out of line, for the inlined greedy path (keeps its registers
// out of the streaming loop; v goes through memory only for rows that have a history).
static __device__ __noinline__ void patch_hist_ext(const RowCtx &R, int seg_lo, float *v) {
    float w[8];
#pragma unroll
    for (int t = 0; t < 8; t++) w[t] = v[t];
    patch_hist(R, seg_lo, w);
#pragma unroll
    for (int t = 0; t < 8; t++) v[t] = w[t];
}

template <typename E, bool HIST>
__device__ __forceinline__ void arg_dirty(const Raw8<E> &raw, int seg, int V, const RowCtx &R, ArgRun<E> &a) {
    float v[8];
    unpack8(raw, v);
    const int base = seg * SEG + lane_id() * 8;
#pragma unroll
    for (int t = 0; t < 8; t++)
        if (base + t >= V) v[t] = -INFINITY;
    if constexpr (HIST) patch_hist_ext(R, seg * SEG, v);   // history first, as patch_seg orders them
    patch_seg<false>(R, seg * SEG, v);
    const float m1 = max8(v);
    if (m1 > a.best) {
        int t = 7;
#pragma unroll
        for (int j = 6; j >= 0; j--)
            if (v[j] == m1) t = j;
        a.best = m1;
        a.seg = -1;
        a.idx = base + t;
    }
}

// Folds a warp's running argmax into the row's 64-bit key (order key of the max, then the
// complement of the lowest position holding it): one atomicMax per warp and unit.
template <typename E>
__device__ __forceinline__ void arg_flush(const ArgRun<E> &a, unsigned long long *slot) {
    const int idx = a.seg >= 0 ? a.seg * SEG + lane_id() * 8 + first_equal8<E>(a.raw, a.best) : a.idx;
    const uint32_t k = fkey(a.best);
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, k);
    const uint32_t imin = __reduce_min_sync(0xffffffffu, k == kmax ? (uint32_t)idx : 0xffffffffu);
    if (lane_id() == 0) atomicMax(slot, ((unsigned long long)kmax << 32) | (unsigned long long)(~imin));
}

// Clean segment: bf16 pairs reduced packed.
template <typename E, int MODE>
__device__ __forceinline__ void seg_clean(const Raw8<E> &raw, int seg, float s, const SegStats &o) {
    if constexpr (sizeof(E) == 2 && MODE != MODE_SUM) {
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&raw.a);
        const __nv_bfloat162 M = __hmax2(__hmax2(p[0], p[1]), __hmax2(p[2], p[3]));
        seg_emit<MODE>(seg, fmaxf(__low2float(M), __high2float(M)), o);
    } else {
        float v[8];
        unpack8(raw, v);
        seg_from_values<MODE>(v, seg, s, o);
    }
}

// Segment that is ragged (ends past V) or holds a penalised token.
template <typename E, int MODE, bool HIST>
__device__ __noinline__ void seg_dirty(const Raw8<E> raw, int seg, int V, const RowCtx &R, float s,
                                       const SegStats o) {
    float v[8];
    unpack8(raw, v);
    const int base = seg * SEG + lane_id() * 8;
#pragma unroll
    for (int t = 0; t < 8; t++)
        if (base + t >= V) v[t] = -INFINITY;
    patch_seg<HIST>(R, seg * SEG, v);
    seg_from_values<MODE>(v, seg, s, o);
}

// Ring position shared by the producer and the consumers: stage index and phase parity.
struct RingPos {
    int st;
    uint32_t ph;
    __device__ __forceinline__ void next(int pns) {
        if (++st == pns) {
            st = 0;
            ph ^= 1u;
        }
    }
};

// One streamer warp's share of a row: waits for each chunk, copies its segments to registers,
// releases the stage, then reduces them.  Returns false when a wait timed out.  PEN: 0 no
// penalised token, 1 penalised drafts, 2 penalised drafts and a prior history (only the
// last instantiates the history code, which keeps it out of the others' registers).
template <typename E, int MODE, int PEN>
__device__ __forceinline__ bool stream_row(unsigned long long *full, unsigned long long *empty,
                                           const unsigned char *ring, int pns, RingPos &rp, int c0, int c1, int nseg,
                                           int V, int sw, const RowCtx &R, const SegStats &o, const uint32_t *dmask,
                                           unsigned long long *argslot, unsigned long long *tslot) {
    constexpr int SPC = SB / (SEG * (int)sizeof(E));   // segments per chunk
    constexpr int NSW = pstream<E>();
    constexpr int PER = (SPC + NSW - 1) / NSW;
    constexpr bool EVEN = SPC % NSW == 0;
    const int nfull = V / SEG;                          // segments wholly inside the row
    const float s = R.s;
    (void)tslot;
    ArgRun<E> arg;
    arg.best = -INFINITY;
    arg.seg = -1;
    arg.idx = 0x7fffffff;
    for (int c = c0; c < c1; c++) {
#ifdef SV_TIMING
        const unsigned long long tw = global_ns();
#endif
        if (!__all_sync(0xffffffffu, mbar_wait(&full[rp.st], rp.ph))) return false;
#ifdef SV_TIMING
        if (tslot && lane_id() == 0 && sw == 0) {
            if (c == c0) tslot[8] = global_ns();
            else tslot[10] += global_ns() - tw;
        }
#endif
        const unsigned char *buf = ring + rp.st * SB;
        Raw8<E> raw[PER];
#pragma unroll
        for (int u = 0; u < PER; u++) {
            const int jj = sw + u * NSW;
            if (EVEN || jj < SPC) raw[u] = ring_raw<E>(buf, jj);
        }
        __syncwarp();
        if (lane_id() == 0) mbar_arrive(&empty[rp.st]);
        rp.next(pns);
#pragma unroll
        for (int u = 0; u < PER; u++) {
            const int jj = sw + u * NSW;
            const int seg = c * SPC + jj;
            if ((!EVEN && jj >= SPC) || seg >= nseg) continue;
            bool clean = seg < nfull;
            if constexpr (PEN != 0) clean = clean && !((dmask[seg >> 5] >> (seg & 31)) & 1u);
            if constexpr (MODE == MODE_ARG) {
                if (clean) arg_clean<E>(raw[u], seg, arg);
                else arg_dirty<E, PEN == 2>(raw[u], seg, V, R, arg);
            } else {
                if (clean) seg_clean<E, MODE>(raw[u], seg, s, o);
                else seg_dirty<E, MODE, PEN == 2>(raw[u], seg, V, R, s, o);
            }
        }
    }
    if constexpr (MODE == MODE_ARG) arg_flush(arg, argslot);
    return true;
}

// Dispatch on the row's statistics mode and on whether it has penalised tokens.  Only the
// HIST instance of the stream kernel (launched for calls with a prior history) holds the
// history variants: their code slows every row of a kernel that contains it.
template <typename E, bool HIST>
__device__ __forceinline__ bool stream_row_any(unsigned long long *full, unsigned long long *empty,
                                               const unsigned char *ring, int pns, RingPos &rp, int c0, int c1,
                                               int nseg, int V, int sw, const RowCtx &R, const SegStats &o,
                                               const uint32_t *dmask, unsigned long long *argslot,
                                               unsigned long long *tslot) {
    const int mode = R.mode;
#define SV_STREAM_ROW(PEN_)                                                                                        \
    switch (mode) {                                                                                                \
        case MODE_ARG: return stream_row<E, MODE_ARG, PEN_>(full, empty, ring, pns, rp, c0, c1, nseg, V, sw, R, o, \
                                                             dmask, argslot, tslot);                              \
        case MODE_TOP2: return stream_row<E, MODE_TOP2, PEN_>(full, empty, ring, pns, rp, c0, c1, nseg, V, sw, R, \
                                                              o, dmask, argslot, tslot);                          \
        case MODE_SUM: return stream_row<E, MODE_SUM, PEN_>(full, empty, ring, pns, rp, c0, c1, nseg, V, sw, R, o, \
                                                             dmask, argslot, tslot);                              \
        default: return stream_row<E, MODE_MAX, PEN_>(full, empty, ring, pns, rp, c0, c1, nseg, V, sw, R, o,      \
                                                      dmask, argslot, tslot);                                     \
    }
    if constexpr (HIST) {
        if (R.hdir) SV_STREAM_ROW(2)
    }
    if (R.npen > 0) SV_STREAM_ROW(1)
    SV_STREAM_ROW(0)
#undef SV_STREAM_ROW
}

}  // namespace sv

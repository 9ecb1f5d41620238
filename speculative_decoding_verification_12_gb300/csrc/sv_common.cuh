// sv_common.cuh -- constants, per-row statistics, workspace layout and kernel arguments shared
// by the verification kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int SEG = 256;              // elements per segment: one warp step of 32 lanes x 8
#ifndef SV_CAP
#define SV_CAP 512
#endif
constexpr int CAP = SV_CAP;           // candidate buffer (top-k candidates, kept lists) per group
constexpr int KCAP = 256;             // top-k up to this goes through the candidate buffer
constexpr int WCAP = 256;             // candidate sets up to this are cut and drawn by one warp
constexpr int LCAP = 256;             // kept sets up to this are drawn from as lists (KIND_LIST)
constexpr int HB = 256;               // radix histogram bins (8-bit digits, 4 rounds)
constexpr int NRADIX = 4;             // radix rounds over a 32-bit key
#ifndef SV_SB
#define SV_SB 12288
#endif
constexpr int SB = SV_SB;             // bytes per ring stage (one bulk copy)
constexpr unsigned long long WAIT_NS = 2000000000ull;   // give up on an mbarrier after 2 s
constexpr int MAXK = 64;              // largest k_max
constexpr int MAXV = 1 << 21;         // largest vocabulary
constexpr float LOG2E = 1.4426950408889634f;
constexpr double FIXED_ONE = 1099511627776.0;   // 2^40: fixed-point scale of token weights

// Row kernel (one CTA per row; any alignment): 256 threads, 8 warps.
constexpr int RT = 256;

// Stream kernel (16-byte aligned rows), SCTA CTAs per SM: warp 0 issues bulk copies, warp 1
// schedules work units, pstream<E>() warps reduce the streamed chunks (8 for bf16; 6 for fp32,
// whose 12 segments per chunk then split evenly).  Select kernel: SELT threads per row.
#ifndef SV_SCTA
#define SV_SCTA 3
#endif
#ifndef SV_PSTREAM
#define SV_PSTREAM 8
#endif
#ifndef SV_PSTREAM_F32
#define SV_PSTREAM_F32 6
#endif
#ifndef SV_SPLIT_PARTS
#define SV_SPLIT_PARTS 4              // parts the last wave of rows is split into (1: no split)
#endif
constexpr int SCTA = SV_SCTA;
constexpr int SPLIT_PARTS = SV_SPLIT_PARTS;
template <typename E>
__host__ __device__ constexpr int pstream() { return sizeof(E) == 2 ? SV_PSTREAM : SV_PSTREAM_F32; }
template <typename E>
__host__ __device__ constexpr int stream_threads() { return 32 * (2 + pstream<E>()); }
#ifndef SV_SPLIT_WAVES
#define SV_SPLIT_WAVES 2
#endif
constexpr int SPLIT_WAVES = SV_SPLIT_WAVES;   // waves of rows (one row per CTA each) that are split
#ifndef SV_SELT
#define SV_SELT 128
#endif
constexpr int SELT = SV_SELT;         // threads per select CTA (one row each)
// select CTAs resident per SM (the select kernel's launch bound: 56 registers a thread)
constexpr int SEL_PER_SM = SELT >= 128 ? 9 : 1152 / SELT;
#ifndef SV_PNS_MAX
#define SV_PNS_MAX 3
#endif
constexpr int PNS_MAX = SV_PNS_MAX;   // ring stages at most (the launch picks what fits)
#ifndef SV_NRB
#define SV_NRB 3
#endif
constexpr int NRB = SV_NRB;           // unit buffers between the scheduler and the streamers

// What the streaming pass records per 256-token segment of a row (besides its max).
enum : int32_t {
    MODE_MAX = 0,      // max only (rows whose kept set needs a radix select over the row)
    MODE_ARG = 1,      // + the lowest lane holding the max (greedy rows)
    MODE_TOP2 = 2,     // + that lane, the segment's second-largest value and a histogram of the
                       //   top byte of the maxima's order keys (rows with a small top-k)
    MODE_SUM = 3       // + sum of 2^((z - max) s) (rows that keep every token)
};

// How a row's kept set is represented once its statistics are known.
enum : int32_t {
    KIND_SKIP = 0,     // row not used (padding row, or its request has an error)
    KIND_GREEDY = 1,   // greedy request: argmax only
    KIND_FULL = 2,     // sampled, no filter: every token kept
    KIND_LIST = 3,     // sampled, kept set small: stored as a list (token, weight) in token order
    KIND_THRESH = 4    // sampled, kept set = {z >= tau}, too large for a list
};

// Per-row statistics written by the row's selection and read by the request's finaliser.
// Token weights are e_v = 2^((z_v - m) * s), s = log2(e) / T; p_v = [z_v >= tau] e_v / Z.
struct __align__(16) RowStat {
    float m;        // max of z over the row (z = logit - penalty)
    float s;        // log2(e) / temperature
    float tau;      // kept iff z >= tau
    float Z;        // sum of the kept weights
    float invZ;     // 1 / Z
    uint32_t taukey;  // order key of tau (0: every token kept)
    int32_t argmax; // lowest id of the max (greedy rows)
    int32_t bonus;  // token drawn from this row's p with slot-1 uniform (sampled rows), else -1
    int32_t kind;
    int32_t nlist;  // KIND_LIST: number of list entries
    int32_t resid;  // KIND_LIST rows with a draft: the residual draw should this draft be rejected
    int32_t pad1;
};

struct WsLayout {
    size_t counters, jobcnt, partcnt, rowarg, stats, pq, prep, gstats, hdir, hmask, hstat, listb, jobs, jobsum,
        ready, order, timing, total;
};

// Phase timestamps (globaltimer ns) per work unit, recorded only in builds with SV_TIMING.
constexpr int NTIME = 24;
constexpr int PMAX = 8;               // stream kernel: most parts a row is split into

__host__ __device__ inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }
__host__ __device__ inline int nseg_of(int V) { return (V + SEG - 1) / SEG; }
__host__ __device__ inline int nseg_pad(int nseg) { return (nseg + 31) & ~31; }

// Workspace: [header 256 B: error word, first bad request, work claim counter, stream failure
// flag, lazy scheme: queued row count, residual job count, second work claim counter]
// [per-request arrival counters][per-job slice arrival counters][per-row counts of the stream
// kernel's finished shares][per-row argmax keys of greedy rows]
// [RowStat per row][(p, q) per draft][prepared row context, 640 B per row]
// [segment statistics: 3 words per padded segment per row]
// [history index: np+1 words per request][history segment mask: np/32 words per request]
// [history status: 1 word per request]
// [lazy scheme: queued rows, 1 word per row; residual jobs, 2 words per request; the jobs'
// per-segment residual and target sums, 2 words per padded segment per request]
// [per-row ready words (the call's epoch once the row's statistics are complete)]
// [the streaming order: a ready word, then the row at each position (R words)]
// [timing, SV_TIMING builds only].  The header, the counters and the argmax keys are cleared
// by every call; the history regions are written by the history prepass of calls that pass a
// history, the lazy regions only by the lazy scheme.
__host__ __device__ inline WsLayout ws_layout(int B, int R, int V) {
    WsLayout L;
    const size_t np = (size_t)nseg_pad(nseg_of(V));
    size_t o = 256;
    L.counters = o;
    o += size_t(B) * 4;
    L.jobcnt = o;
    o += size_t(B) * 4;
    L.partcnt = o;
    o = (o + size_t(R) * 4 + 7) & ~size_t(7);
    L.rowarg = o;
    o = up256(o + size_t(R) * 8);
    L.stats = o;
    o = up256(o + size_t(R) * sizeof(RowStat));
    L.pq = o;
    o = up256(o + size_t(R > B ? R - B : 0) * 8);
    L.prep = o;
    o = up256(o + size_t(R) * 640);
    L.gstats = o;
    o = up256(o + size_t(R) * np * 12);
    L.hdir = o;
    o = up256(o + size_t(B) * (np + 1) * 4);
    L.hmask = o;
    o = up256(o + size_t(B) * (np / 32) * 4);
    L.hstat = o;
    o = up256(o + size_t(B) * 4);
    L.listb = o;
    o = up256(o + size_t(R) * 4);
    L.jobs = o;
    o = up256(o + size_t(B) * 8);
    L.jobsum = o;
    o = up256(o + size_t(B) * np * 8);
    L.ready = o;
    o = up256(o + size_t(R) * 4);
    L.order = o;
    o = up256(o + 16 + size_t(R) * 4);
    L.timing = o;
#ifdef SV_TIMING
    o = up256(o + size_t(R) * PMAX * NTIME * 8);
#endif
    L.total = o;
    return L;
}

struct Args {
    const void *logits;
    const float *q;
    const int32_t *tokens;
    const int32_t *nd;
    const int32_t *row_off;   // NULL: uniform layout
    const float *T;
    const int32_t *topk;
    const float *topp;
    const float *pres;        // may be NULL
    const float *freq;        // may be NULL
    const uint8_t *greedy;
    const int32_t *hoff;      // prior history [B+1] offsets, or NULL (then htok, hcnt unused)
    const int32_t *htok;      // history token ids, ascending within each request
    const int32_t *hcnt;      // history counts
    const float *uni;
    int32_t *out_tok;
    int32_t *acc;
    float *out_pq;            // may be NULL
    int32_t *hdr;             // [0] error code, [1] INT_MAX - first bad request, [2] work claim counter,
                              // [3] stream failure flag (a stream CTA gave up on a bounded wait),
                              // [4] lazy scheme: rows queued for phase 2, [5] residual jobs queued,
                              // [6] phase 2's work claim counter, [7] one-pass select: row CTAs
                              // done, [8] residual slices claimed by its worker CTAs, [9] rows
                              // whose kept set is not a candidate list (may need a residual job)
    int32_t *counters;
    unsigned long long *rowarg;   // greedy rows' (max key, ~lowest position), from the stream kernel
    float *gstats;            // per-row segment statistics [R][3][npad] (stream -> select kernel)
    int4 *prep;               // per-row prepared context, 640 B each (stream -> select kernel)
    int32_t *hdir;            // per request: [np+1] history index of each 256-token segment's first entry
    uint32_t *hmask;          // per request: [np/32] bitmask of the segments holding history tokens
    int32_t *hstat;           // per request: 0, or SV_DEV_BAD_HISTORY
    RowStat *stats;
    float *pq;
    unsigned long long *timing;   // SV_TIMING builds only
    int B, k_max, V, R, nseg;
    int pns;                  // stream kernel: ring stages
    int nparts;               // stream kernel: parts each split row is cut into (1: none)
    int nsplit;               // stream kernel: the last nsplit rows are split
    int onehot;               // 1: one-hot drafts -- every row is sampled and the drafts are
                              // accepted while they equal the samples (q is not read)
    int withhold;             // testing aid: the stream kernel's CTA 0 withholds its first unit
    // lazy scheme (rows after a request's first rejection are never read):
    int phase;                // 0: every row at once; 1: each request's row 0; 2: the queued rows
    int ctas;                 // stream kernel: CTAs the launch would use for every row
    int32_t *jobcnt;          // per residual job: slices done
    int32_t *listb;           // rows queued for phase 2 (count in hdr[4])
    // one-pass call: rows are streamed (and selected) in an order of requests -- sampled ones
    // first, greedy ones last -- and each row is selected as soon as its statistics are complete
    uint32_t epoch;           // this call's tag for the ready words (distinct per call)
    int32_t *partcnt;         // per row: finished shares (streamer warps per part, and the preparation)
    uint32_t *ready;          // per row: epoch once the row's statistics and context are in place
    unsigned long long *ordflag;  // key << 32 | (2 * epoch + (1: identity order)) once the order is written
    uint32_t key;             // per-process random tag of ordflag (an old or arbitrary word never matches)
    int32_t *rowmap;          // the row at each position of that order
    int perrow;               // one-pass call: select each row once it is streamed (else once all are)
    int nworkers;             // one-pass call: residual worker CTAs after the select grid's row CTAs
    unsigned long long *jobs; // residual jobs, count in hdr[5]: epoch << 32 | request << 7 | row
    float *jobsum;            // per job and segment: sum of max(0, p - q), then sum of p
};

}  // namespace sv

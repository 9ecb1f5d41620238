// sv_common.cuh -- constants, workspace layout and small device helpers shared by the
// verification kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int NT = 256;               // threads per row CTA
constexpr int NWARP = NT / 32;
constexpr int SEG = 256;              // elements per segment: one warp step of 32 lanes x 8
constexpr int CAP = 2048;             // candidate buffer (top-k candidates, kept lists) per CTA
constexpr int KCAP = 512;             // top-k up to this goes through the candidate buffer
constexpr int WCAP = 256;             // candidate sets up to this are cut and drawn by one warp
constexpr int LCAP = 256;             // kept-list entries stored per row for the residual draw
constexpr int HB = 2048;              // radix histogram bins (11-bit digits)
constexpr int NS = 4;                 // stages of the shared-memory row ring (bulk copies in flight)
constexpr int SB = 8192;              // bytes per ring stage
constexpr unsigned long long WAIT_NS = 2000000000ull;   // give up on an mbarrier after 2 s
constexpr int MAXK = 64;              // largest k_max
constexpr int MAXV = 1 << 21;         // largest vocabulary
constexpr float LOG2E = 1.4426950408889634f;
constexpr double FIXED_ONE = 1099511627776.0;   // 2^40: fixed-point scale of token weights

// How a row's kept set is represented once its statistics are known.
enum : int32_t {
    KIND_SKIP = 0,     // row not used (padding row, or its request has an error)
    KIND_GREEDY = 1,   // greedy request: argmax only
    KIND_FULL = 2,     // sampled, no filter: every token kept
    KIND_LIST = 3,     // sampled, kept set small: stored as a list (token, weight) in token order
    KIND_THRESH = 4,   // sampled, kept set = {z >= tau}, too large for a list
    KIND_FAIL = 5      // the row's stream did not complete (bounded wait expired)
};

// Per-row statistics written by the row CTA and read by the request's finalising CTA.
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
    int32_t pad0, pad1;
};

struct WsLayout {
    size_t counters, stats, pq, lists, timing, total;
};

// Phase timestamps (globaltimer ns) per row CTA, recorded only in builds with SV_TIMING:
// [0] start, [1] request located, [2] row streamed, [3] kept set done, [4] row written,
// [5] finalised, [6] SM id, [7] 1 if this CTA finalised its request, [8..15] steps of the
// candidate path (bound, segment list, re-read, sort, cut, list, draw).
constexpr int NTIME = 16;

__host__ __device__ inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: [header 256 B: error word, first bad request][per-request arrival counters]
// [RowStat per row][(p, q) per draft][kept lists: LCAP x (token, weight) per row].
__host__ __device__ inline WsLayout ws_layout(int B, int R) {
    WsLayout L;
    size_t o = 256;
    L.counters = o;
    o = up256(o + size_t(B) * 4);
    L.stats = o;
    o = up256(o + size_t(R) * sizeof(RowStat));
    L.pq = o;
    o = up256(o + size_t(R > B ? R - B : 0) * 8);
    L.lists = o;
    o = up256(o + size_t(R) * LCAP * 8);
    L.timing = o;
#ifdef SV_TIMING
    o = up256(o + size_t(R) * NTIME * 8);
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
    const float *uni;
    int32_t *out_tok;
    int32_t *acc;
    float *out_pq;            // may be NULL
    int32_t *hdr;             // [0] error code, [1] first bad request
    int32_t *counters;
    RowStat *stats;
    float *pq;
    int32_t *lists;
    unsigned long long *timing;   // SV_TIMING builds only
    int B, k_max, V, R, nseg;
    int q_vec;                // draft-prob rows are 16-byte aligned
};

}  // namespace sv

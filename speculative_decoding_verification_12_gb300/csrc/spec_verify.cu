// spec_verify.cu -- batched speculative-decoding verification for GB300 (sm_103a): the
// C-ABI entry points and the two verify kernels.
//
// Persistent kernel (16-byte aligned rows; the fast path).  A grid of two CTAs per SM claims
// target rows from a counter in the workspace.  Inside a CTA the warps specialise:
//   warp 0     issues cp.async.bulk copies of row after row into a 6 x 8 KB shared-memory
//              ring (completion on mbarriers with transaction counts);
//   warp 1     claims the next rows and prepares them: request lookup, sampling
//              parameters, penalties of the earlier drafts, and the row's draft gathers
//              (x_i, z(x_i), q(x_i)), up to NRB rows ahead;
//   warps 2-9  reduce each streamed 256-token segment to its max (and weight sum);
//   warps 10-13 turn a finished row's segment statistics into its kept set, draws and
//              draft probabilities while the next row streams, and finalise a request when
//              its last row is done.
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
    const Scratch X = carve_scratch(dsm + segstats_bytes(np), np);
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
        float qx = 0.f;
        if (g.t == RT - 1 && S.i < S.k) {
            x = __ldg(A.tokens + S.d0 + S.i);
            if (x >= 0 && x < A.V) {
                zraw = __ldg(row + x);
                if (!S.greedy) qx = __ldg(A.q + (size_t)(S.d0 + S.i) * A.V + x);
            }
        }
        pass_stats<E, VEC>(g, S, row, A.V, A.nseg, o);
        if (g.t == RT - 1) {
            S.xtok = x;
            S.zx = elem_z_raw(S, zraw, x);
            S.qx = qx;
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
// persistent kernel: 16-byte aligned rows
// ------------------------------------------------------------------------------------------

struct PShared {
    unsigned long long full[PNS_MAX];   // ring stage holds its chunk (transaction count)
    unsigned long long empty[PNS_MAX];  // every streamer warp released the stage
    unsigned long long rb_desc[NRB];  // row buffer prepared by the scheduler
    unsigned long long rb_stats[NRB]; // row buffer's segment statistics complete
    unsigned long long rb_free[NRB];  // selector done with the row buffer
    int fail;
    RowCtx rc[NRB];
};

// Per row buffer of the persistent kernel: segment max, second value / weight sum, lane of the
// max, and a bitmask of the segments holding a penalised token; rounded to 128 bytes so that
// every buffer after it (and the 8-byte candidate keys of the scratch) stays aligned.
__host__ __device__ inline size_t pstats_bytes(int np) { return ((size_t(3) * np + np / 32) * 4 + 127) & ~size_t(127); }

__device__ __forceinline__ SegStats carve_pstats(unsigned char *p, int np, uint32_t *&dmask) {
    SegStats o;
    o.mx = reinterpret_cast<float *>(p);
    o.b = o.mx + np;
    o.lane = reinterpret_cast<int *>(o.b + np);
    o.hist = nullptr;
    dmask = reinterpret_cast<uint32_t *>(o.lane + np);
    return o;
}

__host__ __device__ inline size_t persistent_smem(int nseg, int pns) {
    const int np = nseg_pad(nseg);
    return size_t(pns) * SB + size_t(NRB) * pstats_bytes(np) + scratch_bytes(np);
}

__device__ __forceinline__ void pfail(const Args &A, PShared &P, int b) {
    P.fail = 1;
    record_error(A, 7, b < 0 ? 0 : b);
}

template <typename E, bool QVEC>
__global__ void __launch_bounds__(PT, PCTA) verify_persistent_kernel(const Args A) {
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ PShared P;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int V = A.V, nseg = A.nseg, np = nseg_pad(nseg), PNS = A.pns;
    const uint32_t RB = (uint32_t)V * sizeof(E);
    const int nc = (int)((RB + SB - 1) / SB);
    constexpr int SPC = SB / (SEG * (int)sizeof(E));   // segments per chunk
    unsigned char *ring = dsm;
    unsigned char *rbstats = dsm + size_t(PNS) * SB;   // after the ring
    const Scratch X = carve_scratch(rbstats + size_t(NRB) * pstats_bytes(np), np);

    if (threadIdx.x == 0) {
        for (int s = 0; s < PNS; s++) {
            mbar_init(&P.full[s], 1);
            mbar_init(&P.empty[s], PSTREAM);
        }
        for (int s = 0; s < NRB; s++) {
            mbar_init(&P.rb_desc[s], 1);
            mbar_init(&P.rb_stats[s], PSTREAM);
            mbar_init(&P.rb_free[s], 1);
        }
        P.fail = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ---- issuer: bulk copies of each prepared row, chunk by chunk, through the ring
        if (lane != 0) return;
        const unsigned long long pol = l2_evict_last();
        int q = 0;
        RingPos rp{0, 0u};
        for (int j = 0;; j++) {
            const int slot = j % NRB;
            if (!mbar_wait(&P.rb_desc[slot], (uint32_t)(j / NRB) & 1u)) {
                pfail(A, P, -1);
                return;
            }
            const RowCtx &R = P.rc[slot];
            if (R.r < 0) return;
            const unsigned char *src = reinterpret_cast<const unsigned char *>(A.logits) + (size_t)R.r * RB;
            for (int c = 0; c < R.nchunks; c++, q++) {
                const int st = rp.st;
#ifdef SV_TIMING
                const unsigned long long tw = global_ns();
#endif
                // the stage's previous fill (one lap earlier) must have been released
                if (q >= PNS && !mbar_wait(&P.empty[st], rp.ph ^ 1u)) {
                    pfail(A, P, R.b);
                    return;
                }
#ifdef SV_TIMING
                A.timing[(size_t)R.r * NTIME + 11] += global_ns() - tw;
#endif
                const uint32_t off = (uint32_t)c * SB;
                const uint32_t bytes = min((uint32_t)SB, RB - off);
                mbar_expect_tx(&P.full[st], bytes);
                bulk_g2s(ring + st * SB, src + off, bytes, &P.full[st], pol);
                rp.next(PNS);
            }
        }
    } else if (warp == 1) {
        // ---- scheduler: claim rows and prepare their descriptors up to NRB rows ahead
        for (int j = 0;; j++) {
            const int slot = j % NRB;
            bool ok = true;
            if (j >= NRB) ok = mbar_wait_idle(&P.rb_free[slot], (uint32_t)(j / NRB - 1) & 1u);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) pfail(A, P, -1);
                return;
            }
            RowCtx &R = P.rc[slot];
            int r = 0;
            if (lane == 0) r = atomicAdd(A.hdr + 2, 1);
            r = __shfl_sync(0xffffffffu, r, 0);
            if (r >= A.R) {
                if (lane == 0) {
                    R.r = -1;
                    mbar_arrive(&P.rb_desc[slot]);
                }
                return;
            }
            SV_MARK(A, r, 0);
#ifdef SV_TIMING
            if (lane == 0) {
                unsigned smid;
                asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
                A.timing[(size_t)r * NTIME + 6] = ((unsigned long long)blockIdx.x << 32) | smid;
                A.timing[(size_t)r * NTIME + 7] = 0;
                A.timing[(size_t)r * NTIME + 10] = 0;
                A.timing[(size_t)r * NTIME + 11] = 0;
            }
#endif
            locate_row(A, R, r);
            if (R.active) build_penalties(A, R, R.i);
            __syncwarp();
            if (R.active && R.npen > 0) {
                // segments holding a penalised token take the streamers' slow path
                uint32_t *dmask;
                carve_pstats(rbstats + size_t(slot) * pstats_bytes(np), np, dmask);
                for (int w = lane; w < np / 32; w += 32) dmask[w] = 0u;
                __syncwarp();
                for (int h = lane; h < R.npen; h += 32) {
                    const int x = R.pid[h];
                    if (x >= 0 && x < V) atomicOr(&dmask[(x / SEG) >> 5], 1u << ((x / SEG) & 31));
                }
            }
            __syncwarp();
            if (lane == 0) {
                prefetch_draft<E>(A, R, reinterpret_cast<const E *>(A.logits) + (size_t)r * V);
                R.nchunks = R.active ? nc : 0;
                SV_MARK(A, r, 1);
                mbar_arrive(&P.rb_desc[slot]);
            }
            __syncwarp();
        }
    } else if (warp < 2 + PSTREAM) {
        // ---- streamers: per-segment statistics of each row from the ring
        const int sw = warp - 2;
        RingPos rp{0, 0u};
        for (int j = 0;; j++) {
            const int slot = j % NRB;
            if (!__all_sync(0xffffffffu, mbar_wait(&P.rb_desc[slot], (uint32_t)(j / NRB) & 1u))) {
                if (lane == 0) pfail(A, P, -1);
                return;
            }
            const RowCtx &R = P.rc[slot];
            if (R.r < 0) return;
            uint32_t *dmask;
            const SegStats o = carve_pstats(rbstats + size_t(slot) * pstats_bytes(np), np, dmask);
            unsigned long long *tslot = nullptr;
#ifdef SV_TIMING
            tslot = A.timing + (size_t)R.r * NTIME;
#endif
            if (!stream_row_any<E>(P.full, P.empty, ring, PNS, rp, R.nchunks, nseg, V, sw, R, o, dmask, tslot)) {
                if (lane == 0) pfail(A, P, R.b);
                return;
            }
            __syncwarp();
            if (lane == 0) {
                if (sw == 0) SV_MARK(A, R.r, 2);
                mbar_arrive(&P.rb_stats[slot]);
            }
        }
    } else {
        // ---- selectors: kept set, draws and gathers of each finished row; finalisation
        const Grp<PSEL * 32, 1> g(threadIdx.x - 32 * (2 + PSTREAM));
        for (int j = 0;; j++) {
            const int slot = j % NRB;
            const uint32_t par = (uint32_t)(j / NRB) & 1u;
            const bool ok = mbar_wait_idle(&P.rb_desc[slot], par);
            RowCtx &R = P.rc[slot];
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) pfail(A, P, -1);
            }
            g.sync();
            if (P.fail || R.r < 0) return;
            const bool ok2 = mbar_wait_idle(&P.rb_stats[slot], par);
            if (!__all_sync(0xffffffffu, ok2)) {
                if (lane == 0) pfail(A, P, R.b);
            }
            g.sync();
            if (P.fail) return;
            SV_MARK(A, R.r, 9);
            if (R.b >= 0) {
                fail_empty_requests(g, A, R);
                uint32_t *dmask;
                const SegStats o = carve_pstats(rbstats + size_t(slot) * pstats_bytes(np), np, dmask);
                if (R.active) select_row<E, true>(g, A, R, X, o);
                SV_MARK(A, R.r, 4);
                arrive_and_finalize<E, true, QVEC>(g, A, R, X);
                SV_MARK(A, R.r, 5);
            }
            g.sync();
            if (g.t == 0) mbar_arrive(&P.rb_free[slot]);
        }
    }
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

template <typename K>
static cudaError_t ensure_smem(K kern, size_t smem, size_t &enabled) {
    if (smem > 48 * 1024 && smem > enabled) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        enabled = smem;
    }
    return cudaSuccess;
}

template <typename E, bool VEC, bool QVEC>
static cudaError_t launch_rows(const Args &A, cudaStream_t stream) {
    static size_t enabled = 0;
    const size_t smem = rows_smem(A.nseg);
    auto kern = verify_rows_kernel<E, VEC, QVEC>;
    cudaError_t e = ensure_smem(kern, smem, enabled);
    if (e != cudaSuccess) return e;
    kern<<<A.R, RT, smem, stream>>>(A);
    return cudaGetLastError();
}

// Launches the persistent kernel with (SMs x resident CTAs) CTAs; returns cudaErrorNotSupported
// (nothing launched) when it cannot be resident for this vocabulary.
template <typename E, bool QVEC>
static cudaError_t launch_persistent(const Args &A, cudaStream_t stream) {
    static size_t enabled = 0;
    static int sms[64] = {0};
    static int occ_for_nseg[64] = {0};
    static int occ_val[64] = {0};
    // the deepest ring (3..PNS_MAX stages) that still lets two CTAs share an SM
    Args B = A;
    B.pns = PNS_MAX;
    while (B.pns > 3 && PCTA * (persistent_smem(A.nseg, B.pns) + sizeof(PShared) + 1024) > 228 * 1024) B.pns--;
    const size_t smem = persistent_smem(A.nseg, B.pns);
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    auto kern = verify_persistent_kernel<E, QVEC>;
    cudaError_t e = ensure_smem(kern, smem, enabled);
    if (e != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
    if (!sms[dev] && (e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if (occ_for_nseg[dev] != A.nseg) {
        int occ = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, PT, smem)) != cudaSuccess) return e;
        occ_val[dev] = occ;
        occ_for_nseg[dev] = A.nseg;
    }
    const int occ = occ_val[dev];
    if (occ < 1) return cudaErrorNotSupported;
    const int grid = (int)((long long)sms[dev] * occ < (long long)A.R ? sms[dev] * occ : A.R);
    kern<<<grid, PT, smem, stream>>>(B);
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
    A.pns = 0;
    const size_t esz = logits_dtype == SV_BF16 ? 2 : 4;
    const bool vec = ((uintptr_t)target_logits % 16 == 0) && ((size_t)V * esz) % 16 == 0;
    const bool qvec = (!draft_probs || (uintptr_t)draft_probs % 16 == 0) && ((size_t)V * 4) % 16 == 0;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // clear the error word, the row claim counter and the per-request arrival counters
    if (cudaMemsetAsync(ws, 0, L.counters + (size_t)B * 4, st) != cudaSuccess) return SV_ERR_CUDA;
    cudaError_t e = cudaErrorNotSupported;
    if (vec) {
        if (logits_dtype == SV_BF16) e = qvec ? launch_persistent<uint16_t, true>(A, st) : launch_persistent<uint16_t, false>(A, st);
        else e = qvec ? launch_persistent<float, true>(A, st) : launch_persistent<float, false>(A, st);
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

// spec_verify.cu -- batched speculative-decoding verification for GB300 (sm_103a): the C-ABI
// entry points, the small kernels every call shares (clearing the workspace, the history
// prepass, rollback) and the library's static workspace.  The verify kernels and their launch
// sequences live in sv_kernels.cuh, instantiated per logits dtype and scheme by verify_*.cu.
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
#include <chrono>

#include "../../include/spec_verify.h"
#include "sv_launch.h"
#include "sv_row.cuh"

namespace sv {
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

// The current device, checked against MAX_DEVICES.
static cudaError_t current_device(int &dev) {
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return (dev < 0 || dev >= MAX_DEVICES) ? cudaErrorNotSupported : cudaSuccess;
}
// Clears n16 16-byte words at p (the workspace header, counters and argmax keys) and the
// residual job records; with `order` (per-row selection) block 0 also zeroes the rows' ready
// words and builds the streaming order (build_order).  Lets its programmatic dependent (the
// stream kernel) be scheduled early; that kernel waits for this grid before it reads or writes
// anything.
__global__ void __launch_bounds__(256) clear_kernel(uint4 *p, size_t n16, const Args A, int order) {
    // Launched as a programmatic dependent of whatever ran before it on the stream, so that its
    // CTAs can be resident before that work ends.  Every CTA of that work has started by then
    // (a dependent launches only once each CTA of its primary has triggered or exited), so the
    // stream kernel's CTAs, once scheduled, can keep none of it from running; they wait for
    // this grid, and so for that work, before their first access.  With per-row selection they
    // are let in at once, to take SMs as the work before frees them; otherwise only once that
    // work is done (measured the faster order for each scheme).
    if (order) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!order) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#ifdef SV_TIMING
    if (threadIdx.x == 0) atomicMin(A.timing + (size_t)5 * A.R * NTIME + 4, global_ns());
#endif
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
    // the residual job records: a worker reads a slot only after this grid is done, and then
    // finds it zero until its job is written (no stale word can pass for one of this call's)
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < A.B; j += gridDim.x * blockDim.x) A.jobs[j] = 0ull;
#ifdef SV_TIMING
    if (order && blockIdx.x == 0 && threadIdx.x == 0) A.timing[(size_t)5 * A.R * NTIME + 0] = global_ns();
#endif
    if (order && blockIdx.x == 0) build_order<256>(A);
#ifdef SV_TIMING
    if (order && blockIdx.x == 0 && threadIdx.x == 0) A.timing[(size_t)5 * A.R * NTIME + 1] = global_ns();
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(A.timing + (size_t)5 * A.R * NTIME + 5, global_ns());
#endif
}

// Per-call epochs (tags of the ready words; never 0) and the per-process key of the order flag.
static std::atomic<uint32_t> g_epoch{0};
static uint32_t process_key() {
    static const uint32_t key = [] {
        uint64_t x = (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count() ^
                     ((uint64_t)(uintptr_t)&g_epoch << 17) ^ 0x9E3779B97F4A7C15ull;
        x ^= x >> 33;
        x *= 0xFF51AFD7ED558CCDull;
        x ^= x >> 33;
        return (uint32_t)x | 1u;
    }();
    return key;
}
// Events recorded around the stream kernel when set (sv_set_phase_events): process-wide, for
// every device and stream (a measurement aid for one caller at a time).  Recording them
// separates the two kernels, so the select kernel no longer overlaps the stream's end.
static std::atomic<cudaEvent_t> g_phase_start{nullptr}, g_phase_end{nullptr};

// Testing aid (sv_set_test_withhold): process-wide; while set, every stream kernel withholds
// one work unit so that its bounded waits run out.
static std::atomic<bool> g_withhold{false};

}  // namespace sv

using namespace sv;

extern "C" size_t sv_workspace_bytes(int32_t B, int32_t total_rows, int32_t V) {
    if (B < 1 || total_rows < B || V < 1) return 0;
    return ws_layout(B, total_rows, V).total;
}

// Cost model of sv_prefer_lazy, fitted to one-pass and lazy calls timed on a GB300 over batches
// whose share of requests rejecting draft 0 was set from 0 to 1: the lazy call saves the bytes
// of the rows it skips at about the copy rate, and its second phase (a second stream launch and
// a second round of row selection) costs a fixed time that grows with the vocabulary.
constexpr double LAZY_SKIP_BYTES_PER_US = 6.8e6;   // 6.8 TB/s
constexpr double LAZY_PHASE2_US = 10.3;
constexpr double LAZY_PHASE2_US_PER_TOKEN = 1.46e-4;

extern "C" int32_t sv_prefer_lazy(int32_t B, int32_t total_rows, int32_t V, sv_dtype logits_dtype,
                                  float row0_reject_share) {
    if (B < 1 || total_rows < B || V < 1 || (logits_dtype != SV_F32 && logits_dtype != SV_BF16) ||
        !(row0_reject_share >= 0.f && row0_reject_share <= 1.f))
        return -1;
    // every request decided at row 0: the lazy call has no second phase
    if (row0_reject_share >= 1.f) return 1;
    const double esz = logits_dtype == SV_BF16 ? 2.0 : 4.0;
    const double skipped = (double)row0_reject_share * (double)(total_rows - B) * (double)V * esz;
    const double saved_us = skipped / LAZY_SKIP_BYTES_PER_US;
    const double phase2_us = LAZY_PHASE2_US + LAZY_PHASE2_US_PER_TOKEN * (double)V;
    return saved_us > phase2_us ? 1 : 0;
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
                             void *workspace, size_t workspace_bytes, void *stream, bool onehot, bool lazy) {
    if (onehot) draft_probs = nullptr;
    if (B < 1 || k_max < 0 || V < 1 || total_rows < B) return SV_ERR_INVALID_ARG;
    if (k_max > MAXK || V > MAXV || B >= (1 << 25)) return SV_ERR_UNSUPPORTED;
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
    A.jobcnt = reinterpret_cast<int32_t *>(ws + L.jobcnt);
    A.listb = reinterpret_cast<int32_t *>(ws + L.listb);
    A.jobs = reinterpret_cast<unsigned long long *>(ws + L.jobs);
    A.jobsum = reinterpret_cast<float *>(ws + L.jobsum);
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
    A.phase = 0;
    A.ctas = 0;
    A.nworkers = 0;
    A.partcnt = reinterpret_cast<int32_t *>(ws + L.partcnt);
    A.ready = reinterpret_cast<uint32_t *>(ws + L.ready);
    A.ordflag = reinterpret_cast<unsigned long long *>(ws + L.order);
    A.rowmap = reinterpret_cast<int32_t *>(ws + L.order + 16);
    uint32_t ep = g_epoch.fetch_add(1) + 1;
    if ((ep & 0x7fffffffu) == 0) ep = g_epoch.fetch_add(1) + 1;   // (2 * epoch + 1 fits 32 bits; never 0)
    A.epoch = ep & 0x7fffffffu;
    A.key = process_key();
    const size_t esz = logits_dtype == SV_BF16 ? 2 : 4;
    const bool vec = ((uintptr_t)target_logits % 16 == 0) && ((size_t)V * esz) % 16 == 0;
    const bool qvec = (!draft_probs || (uintptr_t)draft_probs % 16 == 0) && ((size_t)V * 4) % 16 == 0;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (current_device(dev) != cudaSuccess) return SV_ERR_UNSUPPORTED;
    // multiprocessors per device, read once (0: not read yet)
    static std::atomic<int> sms[MAX_DEVICES];
    int nsm = sms[dev].load(std::memory_order_relaxed);
    if (!nsm) {
        if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SV_ERR_CUDA;
        sms[dev].store(nsm, std::memory_order_relaxed);
    }
    // The one-pass two-kernel path selects each row as soon as it is streamed when the batch has
    // more rows than the select kernel holds at once: its first wave then runs while the stream
    // ends.  With one wave, early select CTAs would only share the SMs with the stream's last
    // units, so every row is selected once the whole stream is done.
    A.perrow = (vec && !lazy && (long long)total_rows > (long long)SEL_PER_SM * nsm) ? 1 : 0;

    // clear the error word, the work claim counter, the per-request arrival counters, the
    // per-row part counters and the greedy rows' argmax keys
    {
        // (the clear ends below the statistics region, which starts at a 256-byte boundary)
        const size_t n16 = (L.rowarg + (size_t)total_rows * 8 + 15) / 16;
        const unsigned blocks = (unsigned)((n16 + 255) / 256 < 304 ? (n16 + 255) / 256 : 304);
        // (with per-row selection, block 0 also builds the streaming order).  A programmatic
        // dependent of the work before it on the stream, which it waits for.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(blocks);
        cfg.blockDim = dim3(256);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, clear_kernel, reinterpret_cast<uint4 *>(ws), n16, A, A.perrow) != cudaSuccess)
            return SV_ERR_CUDA;
    }
    if (A.hoff) {
        history_kernel<<<B, 256, 0, st>>>(A, params.prior_len);
        if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    }
    const LaunchOpts o{nsm, g_phase_start.load(), g_phase_end.load()};
    const bool bf16 = logits_dtype == SV_BF16;
    cudaError_t e = cudaErrorNotSupported;
    if (lazy && vec) e = bf16 ? launch_lazy_bf16(A, st, o, qvec) : launch_lazy_f32(A, st, o, qvec);
    if (e == cudaErrorNotSupported) {
        cudaGetLastError();   // clear a sticky "not supported" from the probe, if any
        e = bf16 ? launch_onepass_bf16(A, st, o, vec, qvec) : launch_onepass_f32(A, st, o, vec, qvec);
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
                       stream, false, false);
}

extern "C" sv_status spec_verify_onehot(const void *target_logits, sv_dtype logits_dtype, const int32_t *draft_tokens,
                                        const int32_t *num_drafts, const int32_t *row_offsets, int32_t B,
                                        int32_t k_max, int32_t V, int32_t total_rows, sv_params params,
                                        const float *uniforms, int32_t *out_tokens, int32_t *accept_len,
                                        float *out_pq, void *workspace, size_t workspace_bytes, void *stream) {
    return verify_call(target_logits, logits_dtype, nullptr, draft_tokens, num_drafts, row_offsets, B, k_max, V,
                       total_rows, params, uniforms, out_tokens, accept_len, out_pq, workspace, workspace_bytes,
                       stream, true, false);
}

extern "C" sv_status spec_verify_lazy(const void *target_logits, sv_dtype logits_dtype, const float *draft_probs,
                                      const int32_t *draft_tokens, const int32_t *num_drafts,
                                      const int32_t *row_offsets, int32_t B, int32_t k_max, int32_t V,
                                      int32_t total_rows, sv_params params, const float *uniforms,
                                      int32_t *out_tokens, int32_t *accept_len, float *out_pq, void *workspace,
                                      size_t workspace_bytes, void *stream) {
    return verify_call(target_logits, logits_dtype, draft_probs, draft_tokens, num_drafts, row_offsets, B, k_max, V,
                       total_rows, params, uniforms, out_tokens, accept_len, out_pq, workspace, workspace_bytes,
                       stream, false, true);
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

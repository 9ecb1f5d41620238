// sv_launch.h -- the launch sequences of the verify kernels, one translation unit per logits
// dtype and scheme (they compile in parallel), called by the C-ABI entry points.
#pragma once

#include <cuda_runtime.h>

#include "sv_common.cuh"

namespace sv {

// Devices a process may drive (a device index at or beyond it is SV_ERR_UNSUPPORTED).
constexpr int MAX_DEVICES = 64;

struct LaunchOpts {
    int nsm;                 // multiprocessors of the current device
    cudaEvent_t ph0, ph1;    // measurement aid: recorded around the stream kernel when set
};

// The one-pass call: the stream and select kernels for 16-byte aligned rows (vec) that they can
// hold, else the row kernel.  Returns the launch status.
cudaError_t launch_onepass_bf16(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool vec, bool qvec);
cudaError_t launch_onepass_f32(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool vec, bool qvec);

// The one-pass call with per-row selection (Args::perrow) for 16-byte aligned rows;
// cudaErrorNotSupported (nothing launched) when the kernels cannot hold the vocabulary.
cudaError_t launch_rows_bf16(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool qvec);
cudaError_t launch_rows_f32(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool qvec);

// The lazy scheme for 16-byte aligned rows; cudaErrorNotSupported (nothing launched) when the
// kernels cannot hold the vocabulary.
cudaError_t launch_lazy_bf16(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool qvec);
cudaError_t launch_lazy_f32(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool qvec);

}  // namespace sv

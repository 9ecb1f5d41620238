// verify_f32.cu -- the one-pass verify call for fp32 logits (stream and select kernels, or the row
// kernel).
#include "sv_kernels.cuh"

namespace sv {

cudaError_t launch_onepass_f32(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool vec, bool qvec) {
    return launch_onepass_dtype<float>(A, stream, o, vec, qvec);
}

}  // namespace sv

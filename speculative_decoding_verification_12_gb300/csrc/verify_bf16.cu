// verify_bf16.cu -- the one-pass verify call for bf16 logits (stream and select kernels, or the row
// kernel).
#include "sv_kernels.cuh"

namespace sv {

cudaError_t launch_onepass_bf16(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool vec, bool qvec) {
    return launch_onepass_dtype<uint16_t>(A, stream, o, vec, qvec);
}

}  // namespace sv

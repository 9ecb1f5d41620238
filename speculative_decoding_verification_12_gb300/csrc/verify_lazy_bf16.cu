// verify_lazy_bf16.cu -- the lazy scheme for bf16 logits (spec_verify_lazy).
#include "sv_kernels.cuh"

namespace sv {

cudaError_t launch_lazy_bf16(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool qvec) {
    return qvec ? launch_lazy_kernels<uint16_t, true>(A, stream, o) : launch_lazy_kernels<uint16_t, false>(A, stream, o);
}

}  // namespace sv

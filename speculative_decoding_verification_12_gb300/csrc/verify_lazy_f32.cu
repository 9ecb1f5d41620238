// verify_lazy_f32.cu -- the lazy scheme for fp32 logits (spec_verify_lazy).
#include "sv_kernels.cuh"

namespace sv {

cudaError_t launch_lazy_f32(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool qvec) {
    return qvec ? launch_lazy_kernels<float, true>(A, stream, o) : launch_lazy_kernels<float, false>(A, stream, o);
}

}  // namespace sv

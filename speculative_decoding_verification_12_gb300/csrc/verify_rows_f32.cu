// verify_rows_f32.cu -- the one-pass verify call for fp32 logits with per-row selection (rows
// streamed in the order the clearing kernel built, each selected once it is streamed).
#include "sv_kernels.cuh"

namespace sv {

cudaError_t launch_rows_f32(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool qvec) {
    return qvec ? launch_two_kernels<float, true, SCH_ROWS>(A, stream, o)
                : launch_two_kernels<float, false, SCH_ROWS>(A, stream, o);
}

}  // namespace sv

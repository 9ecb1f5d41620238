// verify_f32.cu -- the one-pass verify call for fp32 logits (stream and select kernels, or the row
// kernel).
#include "sv_kernels.cuh"

namespace sv {

cudaError_t launch_onepass_f32(const Args &A, cudaStream_t stream, const LaunchOpts &o, bool vec, bool qvec) {
    if (vec && A.perrow) {
        // per-row selection (its instances compile in a unit of their own)
        const cudaError_t e = launch_rows_f32(A, stream, o, qvec);
        if (e != cudaErrorNotSupported) return e;
        cudaGetLastError();   // the vocabulary does not fit the two kernels: the row kernel below
    }
    return launch_onepass_dtype<float>(A, stream, o, vec, qvec);
}

}  // namespace sv

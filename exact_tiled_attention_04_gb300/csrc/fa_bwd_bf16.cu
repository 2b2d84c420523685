// Backward-pass main kernel, bf16 inputs: instantiations and launcher.
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_bf16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& dout, const CUtensorMap& dk, const CUtensorMap& dv,
                           const CUtensorMap& dq, const BwdParams& p, unsigned int grid,
                           cudaStream_t stream) {
    if (d == 64) return launch_bwd<64, false>(q, k, v, dout, dk, dv, dq, p, grid, stream);
    if (d == 128) return launch_bwd<128, false>(q, k, v, dout, dk, dv, dq, p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa

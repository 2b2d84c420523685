// fp16 instantiations of the forward kernel (head dimension 64 and 128):
// fp16 operands on the kind::f16 tensor-core path, P and O rounded to fp16.
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_f16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                               cudaStream_t stream) {
    return launch_fwd<false, 64, true>(q, k, v, o, p, grid, stream);
}

cudaError_t launch_fwd_f16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                cudaStream_t stream) {
    return launch_fwd<false, 128, true>(q, k, v, o, p, grid, stream);
}

}  // namespace fa

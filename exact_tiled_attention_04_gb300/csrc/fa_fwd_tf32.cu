// fp32-in/out instantiation of the forward kernel: both contractions on the
// TF32 tensor-core path, head dimension 64.
#include "fa_fwd_kernel.cuh"

namespace fa {

size_t fwd_smem_bytes_tf32_d64() { return FwdCfg<true, 64>::kSmemBytes; }

cudaError_t launch_fwd_tf32_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                cudaStream_t stream) {
    return launch_fwd<true, 64>(q, k, v, o, p, grid, stream);
}

}  // namespace fa

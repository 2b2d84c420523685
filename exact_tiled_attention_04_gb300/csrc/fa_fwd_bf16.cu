// bf16 instantiations of the forward kernel (head dimension 64 and 128).
#include "fa_fwd_kernel.cuh"

namespace fa {

size_t fwd_smem_bytes_bf16_d64() { return FwdCfg<false, 64>::kSmemBytes; }
size_t fwd_smem_bytes_bf16_d128() { return FwdCfg<false, 128>::kSmemBytes; }

cudaError_t launch_fwd_bf16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                cudaStream_t stream) {
    return launch_fwd<false, 64>(q, k, v, o, p, grid, stream);
}

cudaError_t launch_fwd_bf16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                 cudaStream_t stream) {
    return launch_fwd<false, 128>(q, k, v, o, p, grid, stream);
}

}  // namespace fa

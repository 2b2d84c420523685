// fp16 instantiations of the decode kernel (head dimension 64 and 128,
// causal and unmasked, 16 or 32 rows per CTA).
#include "fa_decode_kernel.cuh"

namespace fa {

cudaError_t launch_decode_f16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                              const FwdParams& p, unsigned int grid, cudaStream_t stream) {
    if (d == 64) return launch_decode<64, true>(q, k, v, p, grid, stream);
    return launch_decode<128, true>(q, k, v, p, grid, stream);
}

}  // namespace fa

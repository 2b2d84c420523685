// bf16 instantiations of the forward kernel (head dimension 64 and 128).
#include "fa.h"
#include "fa_fwd_kernel.cuh"

namespace fa {

// Waits on phase 0 of an mbarrier that nothing arrives on, through the same
// bounded wait as the forward kernel: it gives up after kWaitLimitNs and
// reports a timeout in the device status.  Used to test failure reporting
// without faulting or hanging the GPU.
__global__ void fa_selftest_wait_kernel(const FwdParams p) {
    __shared__ __align__(8) uint64_t never;
    __shared__ uint32_t abort_word;
    volatile uint32_t* abort_flag = &abort_word;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&never), 1);
        *abort_flag = 0u;
        mbar_init_fence();
    }
    __syncthreads();
    wait_phase(smem_u32(&never), 0, abort_flag, p, 99);
    __syncthreads();
}


int fwd_max_merge_parts(int dtype, int d) {
    if (dtype == FA_DTYPE_F32) return d == 64 ? FwdCfg<true, 64>::kMaxMergeParts : 1;
    return d == 64 ? FwdCfg<false, 64>::kMaxMergeParts : d == 128 ? FwdCfg<false, 128>::kMaxMergeParts : 1;
}

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

cudaError_t launch_selftest_wait(const FwdParams& p, cudaStream_t stream) {
    fa_selftest_wait_kernel<<<1, 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fa

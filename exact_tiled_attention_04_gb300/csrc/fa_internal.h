// Declarations shared by the host entry points (fa_api.cu) and the kernel
// translation units.  Not part of the public C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Parameters of one forward launch, passed by value.
struct FwdParams {
    float* lse;              // fp32 [BH, N] or nullptr
    unsigned int* err;       // device error word (bounded-wait timeouts)
    int N;                   // sequence length
    int n_kv_tiles;          // ceil(N / 128)
    int n_q_blocks;          // ceil(N / 256): query blocks per (b, h)
    float scale_log2;        // scale * log2(e)
};

// Device error word bits.
constexpr unsigned int kDevErrTimeout = 1u;

// Shared memory a CTA of a variant needs (bytes, including alignment slack).
size_t fwd_smem_bytes_bf16_d64();
size_t fwd_smem_bytes_bf16_d128();
size_t fwd_smem_bytes_tf32_d64();

// Launchers: one CTA per 256 query rows of one (b, h); 320 threads.
cudaError_t launch_fwd_bf16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                cudaStream_t stream);
cudaError_t launch_fwd_bf16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                 cudaStream_t stream);
cudaError_t launch_fwd_tf32_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                cudaStream_t stream);

}  // namespace fa

// Declarations shared by the host entry points (fa_api.cu) and the kernel
// translation units.  Not part of the public C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Device status shared by every launch on one device.
struct DevStatus {
    unsigned int word;       // sticky error bits, read and cleared by fa_device_status
    unsigned int abort_gen;  // generation of the last launch that aborted
};

// Parameters of one forward launch, passed by value.
struct FwdParams {
    float* lse;              // fp32 [BH, N] or nullptr
    DevStatus* status;       // device status word of the current device
    unsigned int gen;        // this launch's generation (never 0)
    int N;                   // sequence length
    int n_kv_tiles;          // ceil(N / 128)
    int n_q_blocks;          // ceil(N / 256): query blocks per (b, h)
    float scale_log2;        // scale * log2(e)
};

// Device error word bits.
constexpr unsigned int kDevErrTimeout = 1u;

// A one-CTA kernel that waits, with the forward kernel's bounded wait, on a
// barrier phase nothing completes; it must give up and report a timeout.
cudaError_t launch_selftest_wait(const FwdParams& p, cudaStream_t stream);

// Shared memory a CTA of a variant needs (bytes, including alignment slack).
size_t fwd_smem_bytes_bf16_d64();
size_t fwd_smem_bytes_bf16_d128();
size_t fwd_smem_bytes_tf32_d64();

// Launchers: one CTA per 256 query rows of one (b, h); 384 threads.
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

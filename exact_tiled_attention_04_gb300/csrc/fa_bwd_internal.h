// Declarations shared by the backward-pass entry points (fa_bwd_api.cu) and
// its kernel translation units.  Not part of the public C ABI.
//
// The backward pass runs three kernels on the caller's stream:
//   1. prep:  per query row i, D_i = dO_i . O_i and the negated base-2
//             log-sum-exp -lse_i * log2(e) (the row statistics the main
//             kernel reads), and a zeroed fp32 dQ accumulator row;
//   2. main:  one CTA per 128 keys of one (batch, key/value head): dK and dV
//             of those keys accumulated in tensor memory over every query
//             tile of the head's query heads, and the dQ contribution of
//             each (query tile, key block) pair added into the accumulator;
//   3. dq:    dQ = scale * accumulator, converted to the input dtype.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"

namespace fa {

// Row statistics, one 1 KB block per 128-row query tile (tile t of head bh
// is block bh * Nq_pad / 128 + t): 128 floats -lse * log2(e) (-inf for a
// padding row or a row with no visible key), then 128 floats
// D = sum_c dO[c] * O[c] (0 for a padding row).
constexpr int kStatFloatsPerTile = 256;

// Parameters of the prep kernel.
struct BwdPrepParams {
    const void* o;        // [B*H, Nq, d] input dtype
    const void* dout;     // [B*H, Nq, d] input dtype
    const float* lse;     // [B*H, Nq] natural log
    float* stats;         // B*H*Nq_pad/128 blocks of kStatFloatsPerTile
    float* dq_acc;        // [B*H, Nq, d] fp32, zeroed here
    long long rows_pad;   // B*H*Nq_pad
    int Nq;
    int Nq_pad;           // Nq rounded up to a multiple of 128
};

// Parameters of one main-kernel launch, passed by value.
struct BwdParams {
    DevStatus* status;    // device status word of the current device
    unsigned int gen;     // this launch's generation (never 0)
    const float* stats;   // B*H*Nq_pad/128 blocks of kStatFloatsPerTile
    int Nq;               // query rows per head
    int Nkv;              // key / value rows per head
    int Nq_pad;           // Nq rounded up to a multiple of 128
    int n_q_tiles;        // Nq_pad / 128
    int n_kv_blocks;      // ceil(Nkv / 128): CTAs per (batch, key/value head)
    int H;                // query heads
    int H_kv;             // key / value heads
    int group;            // H / H_kv
    int causal;           // 1: query i sees keys j <= i + causal_offset only
    int causal_offset;    // Nkv - Nq
    float scale_log2;     // scale * log2(e)
    float scale;          // applied to dK in the epilogue
};

// Parameters of the dQ conversion.
struct BwdDqParams {
    const float* dq_acc;  // [n] fp32
    void* dq;             // [n] input dtype
    long long n;          // B*H*Nq*d (a multiple of 8)
    float scale;
};

// Host-side argument checks of fa_bwd on the tensors alone (sizes, dtype,
// flags, alignment, and that dq, dk, dv overlap no input and no other
// output); returns an FA_* status.  The workspace is the caller's to check.
int validate_bwd_tensors(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, const void* dq, const void* dk, const void* dv, int64_t B, int64_t H,
                         int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, float scale, int dtype_arg);
// Bytes of q, k, v, o, dout, lse (16-bit inputs) into len[0..5].
void bwd_tensor_bytes(int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_kv, int64_t d, size_t* len);

cudaError_t launch_bwd_prep(const BwdPrepParams& p, int d, int dtype, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdDqParams& p, int dtype, cudaStream_t stream);

// Main kernel: grid = B * H_kv * n_kv_blocks CTAs of 384 threads (512 for
// d = 128 without the causal mask).  Maps:
// q, dO over [B*H, Nq, d]; k, v, dk, dv over [B*H_kv, Nkv, d] (input dtype);
// dq over the fp32 accumulator [B*H, Nq, d].
cudaError_t launch_bwd_bf16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& dk, const CUtensorMap& dv,
                            const CUtensorMap& dq, const BwdParams& p, unsigned int grid,
                            cudaStream_t stream);
cudaError_t launch_bwd_f16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& dout, const CUtensorMap& dk, const CUtensorMap& dv,
                           const CUtensorMap& dq, const BwdParams& p, unsigned int grid,
                           cudaStream_t stream);

}  // namespace fa

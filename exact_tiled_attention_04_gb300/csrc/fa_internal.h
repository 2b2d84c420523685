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
//
// Packed launches (pack = 1; grouped heads with Nq * group <= 128, e.g. a
// decode step): a CTA serves one key/value head, and query tile 0 holds the
// Nq rows of each of its `group` query heads, row r = g * Nq + i for query
// head (key/value head * group + g) and query index i.  The Q and O tensor
// maps then use boxes of Nq rows x group heads.
struct FwdParams {
    float* lse;              // fp32 [B*H, Nq] or nullptr (unsplit launches)
    DevStatus* status;       // device status word of the current device
    unsigned int gen;        // this launch's generation (never 0)
    int Nq;                  // query rows per head
    int Nkv;                 // key / value rows per head
    int n_kv_tiles;          // ceil(Nkv / 128)
    int n_q_blocks;          // ceil(Nq / 256): query blocks per (b, h)
    int H;                   // query heads
    int group;               // query heads per key/value head (H / H_kv)
    int H_kv;                // key / value heads
    int pack;                // 1: grouped heads packed into one tile (see below)
    int causal;              // 1: query i sees keys j <= i + causal_offset only
    int causal_offset;       // Nkv - Nq (the last query sees every key)
    int splits;              // key-range partitions per query block (1 = none)
    int tiles_per_split;     // key tiles per partition
    float scale_log2;        // scale * log2(e)
    // splits > 1: unnormalised partial results, one slab per partition
    float* o_part;           // fp32 [splits, B*H, Nq, d]
    float* ml_part;          // fp32 [splits, B*H, Nq, 4]: m (base 2, scaled), l, lq, unused
    void* out;               // decode kernel, splits == 1: O [B*H, Nq, d] (input dtype)
    int item_offset;         // first query block (work item) of this launch: 0, or the
                             // first block of a tail launch (see launch_ex)
    long long part_row0;     // splits > 1: output row of the first row of a partition's slab
    long long part_rows;     // splits > 1: rows of one partition's slab
    int cluster;             // splits > 1 and 1 here: the partitions of a query block form
                             // one thread-block cluster (of `splits` CTAs) and merge their
                             // partial results through distributed shared memory; no
                             // workspace (o_part, ml_part unused), O and lse written directly
};

// Merge of split partial results: O = sum_s w_s O_s / sum_s w_s lq_s,
// lse = ln 2 * (M + log2 sum_s w_s l_s), w_s = 2^(m_s - M), M = max_s m_s.
struct MergeParams {
    const float* o_part;
    const float* ml_part;
    void* o;                 // [B*H, Nq, d] in the output dtype
    float* lse;              // [B*H, Nq] or nullptr
    long long rows;          // B*H*Nq
    int splits;
};

// Device error word bits.
constexpr unsigned int kDevErrTimeout = 1u;

// A one-CTA kernel that waits, with the forward kernel's bounded wait, on a
// barrier phase nothing completes; it must give up and report a timeout.
cudaError_t launch_selftest_wait(const FwdParams& p, cudaStream_t stream);

// Largest thread-block cluster whose key partitions the forward kernel can
// merge in shared memory, for a dtype (fa_dtype_t) and head dimension; 1 when
// none.
int fwd_max_merge_parts(int dtype, int d);

// Shared memory a CTA of a variant needs (bytes, including alignment slack).
size_t fwd_smem_bytes_bf16_d64();
size_t fwd_smem_bytes_bf16_d128();
size_t fwd_smem_bytes_tf32_d64();

cudaError_t launch_merge(const MergeParams& m, int d, int dtype, cudaStream_t stream);

// Launchers: one CTA per 256 query rows of one (b, h) and key partition;
// 384 threads.
cudaError_t launch_fwd_bf16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                cudaStream_t stream);
cudaError_t launch_fwd_bf16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                 cudaStream_t stream);
cudaError_t launch_fwd_f16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                               cudaStream_t stream);
cudaError_t launch_fwd_f16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                cudaStream_t stream);
cudaError_t launch_fwd_tf32_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, unsigned int grid,
                                cudaStream_t stream);

// Decode kernel (fa_decode_kernel.cuh): rows Nq * group <= 32 per key/value
// head, one CTA per (batch, key/value head) and key partition: grid =
// B * H_kv * p.splits.  q over [B*H, Nq, d] with boxes of Nq rows x group
// heads; k, v over [B*H_kv, Nkv, d].  d is 64 or 128.
cudaError_t launch_decode_bf16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const FwdParams& p, unsigned int grid, cudaStream_t stream);
cudaError_t launch_decode_f16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                              const FwdParams& p, unsigned int grid, cudaStream_t stream);

}  // namespace fa
